"""GPU parity for the verification-attention readout and the windowed
drafter cross-attention (Alignment Drift §5, App. A.2 and D.2): after every
target pass the head-averaged audio attention of the row that produced the
next anchor is read at one layer; its peak frame centres a +-20-frame window
on the drafter's cross-attention.  The centres and the windowed drafter's
logits match the oracle, and the output stays autoregressive greedy."""
import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from gpu_common import logits_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def RB():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding, runtime
    return runtime, binding


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_tiny_readout_centers_and_windowed_drafter(RB):
    """fp32 tiny model, readout layer 2, half-width 20: the window centre after
    the prompt and after every round equals the oracle's, the windowed
    drafter's logits match the oracle's (1e-4), and the transcript is the
    oracle's greedy transcript."""
    R, B = RB
    s = synth.TINY
    tw = synth.target_weights(s, 0)
    dw = synth.drafter_weights(s, 0, tw)
    A = synth.encoder_states(s, 0, 0)
    orc = M.Oracle(s, tw, dw)
    budget, layer, hw = 32, 2, 20
    ref = M.speculative_greedy_windowed(orc, orc.new_request(A), budget, layer, hw)
    ar = M.greedy_cached(orc, orc.new_request(A), budget).tokens
    assert ref.tokens == ar
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=1500)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    dec.set_readout(layer, hw)
    b = dec.new_batch(req, [budget], draft_logits=True)
    b.prefill()
    centers = [int(dec.centers(req)[0])]
    # the first windowed draft against the oracle's, at the oracle's state after the prompt
    r = orc.new_request(A)
    logits = orc.verify(r, list(s.prompt), layer)
    r.center = r.peaks[len(s.prompt) - 1]
    r.L = len(s.prompt)
    anchor = int(np.argmax(logits[-1]))
    assert int(b.block[0, 0].item()) == anchor
    dec.draft(req, b.block, 0.0, 0, 0, b.q_logits)
    logits_close(b.q_logits[0].cpu().numpy(), orc.draft_logits(r, anchor, hw), 1e-4)
    b2 = dec.new_batch(req, [budget], draft_logits=True)
    b2.prefill()
    while b2.poll_done() < 1:
        b2.spec_step(0, graph=False)
        centers.append(int(dec.centers(req)[0]))
    assert b2.transcripts()[0] == ar
    assert centers[:len(ref.margins)] == ref.margins, (centers, ref.margins)
    assert dec.status() == 0


def test_large_v3_windowed_speculation_equals_autoregressive(RB):
    """Large-v3 bf16 batch 1, readout at layer 21 (the pages' choice for a
    32-layer target), +-20 frames: 96 tokens bit-identical to autoregressive
    decoding, every centre inside the 1500 frames."""
    R, B = RB
    s = synth.LARGE_V3
    tw = synth.target_weights(s, 1)
    dw = synth.drafter_weights(s, 1, tw)
    A = synth.encoder_states(s, 1, 0)
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=1500)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    b = dec.new_batch(req, [96])
    R.run_ar(dec, b)
    ar = b.transcripts()[0]
    dec.set_readout(21, 20)
    b2 = dec.new_batch(req, [96])
    R.run_spec(dec, b2)
    assert b2.transcripts()[0] == ar
    c = int(dec.centers(req)[0])
    assert 0 <= c < 1500
    assert dec.status() == 0
