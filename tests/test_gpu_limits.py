"""GPU parity for truncated verification and confidence-threshold stopping
(Whisper-Flash Table A5: verify only the first K' proposals; Alignment Drift
Table 21: stop drafting below a confidence threshold): the proposals each
round sends to verification match the oracle's limit rule, and the output
stays equal to autoregressive greedy decoding."""
import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from gpu_common import dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def RB():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding, runtime
    return runtime, binding


@pytest.fixture(scope="module")
def tiny(RB):
    R, B = RB
    s = synth.TINY
    tw = synth.target_weights(s, 0)
    dw = synth.drafter_weights(s, 0, tw)
    A = synth.encoder_states(s, 0, 0)
    orc = M.Oracle(s, tw, dw)
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=1500)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    return s, tw, dw, A, orc, dec, req


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("k_verify,quantile", [(1, None), (2, None), (4, 0.5), (2, 0.5), (8, None)])
def test_tiny_limited_rounds_match_oracle(RB, tiny, k_verify, quantile):
    """Round by round on the fp32 tiny model: the number of proposals each
    round sends to verification (after truncation and the confidence rule)
    equals the oracle's, and the transcript equals the oracle's greedy one.
    The threshold is a quantile of the oracle's own drafted-token
    confidences (random-weight drafters are far from confident), so the
    rule cuts some rounds and not others; a round whose oracle confidence
    sits within 1e-3 (relative) of the threshold ends the comparison."""
    R, B = RB
    s, tw, dw, A, orc, dec, req = tiny
    budget = 40
    threshold = 0.0
    if quantile is not None:
        log0 = []
        M.speculative_greedy_limited(orc, orc.new_request(A), budget, k_verify, 0.0, log0)
        # in the widest gap between the oracle's distinct confidences around the
        # quantile, so that no round's confidence sits on the threshold
        vals = np.unique(np.asarray(log0)[:, :k_verify])
        lo = int(max(0.0, quantile - 0.25) * len(vals))
        hi = max(int(min(1.0, quantile + 0.25) * len(vals)), lo + 2)
        i = lo + 1 + int(np.argmax(vals[lo + 1:hi] / vals[lo:hi - 1]))
        threshold = float(np.sqrt(vals[i - 1] * vals[i]))
    log = []
    ref = M.speculative_greedy_limited(orc, orc.new_request(A), budget, k_verify, threshold, log)
    b = dec.new_batch(req, [budget], draft_logits=True)
    b.prefill()
    K, H = s.K, k_verify + 1
    got = []
    while b.poll_done() < 1:
        dec.draft(req, b.block, 0.0, 0, 0, b.q_logits)
        B.ws_draft_limit(dec.ctx, 1, req.data_ptr(), b.block.data_ptr(), K + 1, b.q_logits.data_ptr(), k_verify,
                         threshold, 0.0, b.vblock.data_ptr(), H, b.blen.data_ptr(), _stream())
        got.append(int(b.blen[0].item()) - 1)
        B.ws_verify(dec.ctx, 1, req.data_ptr(), H, b.vblock.data_ptr(), b.blen.data_ptr(), b.target.data_ptr(), 0,
                    _stream())
        a = b._args(B.WS_ACCEPT_GREEDY, H, b.vblock, b.blen, b.target, b.block, b.blen)
        B.ws_accept(dec.ctx, 1, req.data_ptr(), a, _stream())
    compared = 0
    for i, (g, e) in enumerate(zip(got, ref.proposed)):
        if threshold > 0 and any(abs(c - threshold) < 1e-3 * threshold for c in log[i][:k_verify]):
            break
        assert g == e, (i, got, ref.proposed)
        compared += 1
    assert compared >= len(ref.proposed) // 2
    if compared == len(ref.proposed):
        assert got == ref.proposed
        assert b.transcripts()[0] == ref.tokens
    assert dec.status() == 0


def test_large_v3_truncated_and_thresholded_equal_autoregressive(RB):
    """Large-v3 bf16 batch 1, 96 tokens: verifying only 2 or 4 of the 8
    proposals, and with a confidence threshold, all give the autoregressive
    transcript bit for bit (one captured graph per verify length)."""
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
    traj = np.zeros((1, s.max_pos), dtype=np.int32)
    t = list(s.prompt) + ar
    traj[0, :len(t)] = t
    plan = synth.corruption_plan(1, s.max_pos, s.K, synth.corruption_p_const(s.K, 0.2), s.vocab, 5)
    syn = (torch.as_tensor(traj, device="cuda"), torch.as_tensor(plan.mask, device="cuda"),
           torch.as_tensor(plan.tok, device="cuda"))
    rounds = {}
    for kv, thr in ((2, 0.0), (4, 0.0), (8, 1e-4)):
        b2 = dec.new_batch(req, [96], draft_logits=True)
        rounds[kv] = R.run_spec(dec, b2, synthetic=syn, k_verify=kv, threshold=thr)
        assert b2.transcripts()[0] == ar, kv
    assert rounds[2] > rounds[4]                  # fewer proposals per round, more rounds
    assert dec.status() == 0
