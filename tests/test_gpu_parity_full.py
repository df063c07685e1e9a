"""Full-size GPU parity where the method's own checks are weakest:

  * a whole 9-row block verification at large-v3 batch 96 (864 rows through
    the batched tcgen05 GEMMs and the streaming attention), three requests'
    rows compared with the oracle element by element;
  * the bf16 drafter (fusion projection, history K/V with RoPE, block
    projections, joint attention, own acoustic K/V, shared LM head) against
    the oracle's bf16-emulating drafter, after the prompt and after one
    verified round (Whisper-Flash §3.2, Eq. 2; App. A.2);
  * speculative sampling through the bf16 drafter: the first token of a
    round follows the target's distribution (Whisper-Flash §3.1, the
    rejection rule preserves p; App. A.4), checked by chi-square against the
    oracle's p at the same prefix.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from gpu_common import dev_i32, logits_close, small_shape

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def RB():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding, runtime
    return runtime, binding


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_large_v3_batch96_block_verify_vs_oracle(RB):
    """96 requests with their own encoder states: prompt prefill, then one
    verify of [anchor, 8 random tokens] per request.  Requests 0, 47 and 95
    are compared with the oracle's cached verify of the same blocks."""
    R, B = RB
    s = synth.LARGE_V3
    tw = synth.target_weights(s, 1)
    n, K = 96, s.K
    As = [synth.encoder_states(s, 1, 500 + i) for i in range(n)]
    dec = R.Decoder(s, tw, None, max_batch=n, max_frames=1500)
    req = dec.slots(list(range(n)))
    dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in As]), [1500] * n)
    b = dec.new_batch(req, [100] * n)
    b.prefill()                                            # L = 4 for every request
    orc = M.Oracle(s, tw, None)
    anchors = b.block[:, 0].cpu().numpy().copy()
    refs = {}
    for i in (0, 47, 95):                                  # the compared requests take the oracle's anchor
        r = orc.new_request(As[i])
        pre = orc.verify(r, list(s.prompt))
        r.L = len(s.prompt)
        anchors[i] = int(np.argmax(pre[-1]))
        refs[i] = r
    rng = np.random.default_rng(96)
    cand = rng.integers(0, s.vocab, size=(n, K))
    block = np.concatenate([anchors[:, None], cand], axis=1).astype(np.int32)
    tgt = torch.zeros(n, K + 1, dtype=torch.int32, device="cuda")
    lg = torch.empty(n, K + 1, s.vocab, device="cuda")
    dec.verify(req, dev_i32(block), dev_i32([K + 1] * n), tgt, lg)
    torch.cuda.synchronize()
    for i, r in refs.items():
        ora = orc.verify(r, block[i].tolist())
        logits_close(lg[i].cpu().numpy(), ora, 2e-2)
        assert tgt[i].tolist() == lg[i].argmax(dim=1).tolist()
    assert dec.status() == 0


def _drafter_vs_oracle(R, B, s, tw, dw, A, F):
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=F)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [F])
    orc = M.Oracle(s, tw, dw)
    b = dec.new_batch(req, [64], sampling=True)
    b.prefill()
    r = orc.new_request(A)
    acc, logits = M.prefill(orc, r, 64)
    anchor = acc.next_anchor                               # the oracle's first token is the anchor
    b.block[0, 0] = anchor
    dec.draft(req, b.block, 1.0, 3, 1, b.q_logits)
    q1 = b.q_logits[0].cpu().numpy()
    logits_close(q1, orc.draft_logits(r, anchor), 2e-2)
    # one round with the oracle's own continuation as the first 3 candidates
    ref = M.greedy_cached(orc, orc.new_request(A), 5).tokens
    cand = ref[1:4] + [7] * (s.K - 3)
    b.block[0, 0] = anchor
    b.block[0, 1:] = dev_i32(cand)
    b.blen[0] = s.K + 1
    dec.verify(req, b.block, b.blen, b.target)
    a = b._args(B.WS_ACCEPT_FORCED, s.K + 1, b.block, b.blen, b.target, b.block, b.blen)
    B.ws_accept(dec.ctx, 1, req.data_ptr(), a, _stream())   # teacher-forced: L advances by 9
    lg = orc.verify(r, [anchor] + cand)
    r.L += s.K + 1
    anchor2 = int(np.argmax(lg[-1]))
    b.block[0, 0] = anchor2
    dec.draft(req, b.block, 1.0, 3, 2, b.q_logits)
    logits_close(b.q_logits[0].cpu().numpy(), orc.draft_logits(r, anchor2), 2e-2)
    assert dec.status() == 0


def test_bf16_drafter_small_vs_oracle(RB):
    R, B = RB
    s = small_shape("bf16")
    tw = synth.target_weights(s, 61)
    dw = synth.drafter_weights(s, 61, tw)
    A = synth.encoder_states(s, 61, 0, frames=200)
    _drafter_vs_oracle(R, B, s, tw, dw, A, 200)


def test_bf16_drafter_large_v3_vs_oracle(RB):
    """The 60.7M-parameter large-v3 drafter (fusion 5d -> d over layers
    {1, 8, 15, 22, 29}) with 1500 frames."""
    R, B = RB
    s = synth.LARGE_V3
    tw = synth.target_weights(s, 1)
    dw = synth.drafter_weights(s, 1, tw)
    A = synth.encoder_states(s, 1, 0)
    _drafter_vs_oracle(R, B, s, tw, dw, A, 1500)


def test_bf16_speculative_sampling_first_token_distribution(RB):
    """Small bf16 model, T = 0.7: from the prompt, the drafter samples K
    proposals and the rejection rule accepts or resamples; over 4096 seeds
    the first emitted token of the round must follow softmax(z/T) of the
    target at the anchor (z from the oracle, bf16 storage points), tested
    by chi-square over 40 equal-mass bins (alpha = 1e-3)."""
    from scipy.stats import chi2
    R, B = RB
    s = small_shape("bf16", vocab=500, eos_id=499, prompt=(490, 491, 492, 493))
    tw = synth.target_weights(s, 62)
    dw = synth.drafter_weights(s, 62, tw)
    A = synth.encoder_states(s, 62, 0, frames=128)
    n, T = 64, 0.7
    dec = R.Decoder(s, tw, dw, max_batch=n, max_frames=128)
    req = dec.slots(list(range(n)))
    dec.cross_kv(req, torch.cat([dec.enc_tensor(A)] * n), [128] * n)
    orc = M.Oracle(s, tw, None)
    r = orc.new_request(A)
    acc, _ = M.prefill(orc, r, 1000)
    anchor = acc.next_anchor                               # the oracle's greedy first token
    counts = np.zeros(s.vocab)
    for rep in range(64):
        b = dec.new_batch(req, [1000] * n, tcap=4, sampling=True)
        b.prefill()                                       # cache: the prompt (L = 4)
        b.block[:, 0] = anchor
        dec.draft(req, b.block, T, 1000 + rep, 1, b.q_logits)
        dec.verify(req, b.block, b.blen, b.target, b.p_logits)
        a = b._args(B.WS_ACCEPT_SAMPLE, s.K + 1, b.block, b.blen, b.target, b.block, b.blen, b.p_logits,
                    b.q_logits, T, 1000 + rep, 1)
        B.ws_accept(dec.ctx, n, req.data_ptr(), a, _stream())
        tr = b.transcript.cpu().numpy()
        counts += np.bincount(tr[:, 1], minlength=s.vocab)   # transcript[0] = prefill token
    N = counts.sum()
    assert N == 64 * n
    z = orc.verify(r, [anchor])[0]
    p = M.probs_fp32(z, T).astype(np.float64)
    order = np.argsort(-p)
    bins = np.minimum((np.cumsum(p[order]) * 40).astype(int), 39)
    obs = np.bincount(bins, weights=counts[order], minlength=40)
    exp = np.bincount(bins, weights=p[order], minlength=40) * N
    keep = exp > 0
    stat = float(((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum())
    assert stat < chi2.ppf(1 - 1e-3, int(keep.sum()) - 1), stat
    assert dec.status() == 0
