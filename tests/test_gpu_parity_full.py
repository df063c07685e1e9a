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
    oracle's p at the same prefix;
  * bf16 sampled transcripts, autoregressive and speculative, token by token
    against the oracle's, with the near-boundary rule widened to the
    precision the bf16 logits measurably have.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from gpu_common import (ar_sampling_from, dev_i32, logits_close, small_shape, teacher_forced_logits, tokens_match,
                        tokens_match_resuming)

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


def test_bf16_sampling_transcripts_vs_oracle(RB):
    """Small bf16 shape, T = 0.7, 40 tokens.  First the bf16 logit precision
    of this model is measured: the largest |GPU - oracle| logit difference,
    target over the oracle's own sampled transcript (teacher forced) and
    drafter after the prompt, delta.  A logit error of delta moves a
    probability of softmax(z / T) by a factor within exp(+-2 delta / T), so
    a sampled decision counts as a near boundary where the oracle's
    acceptance test u q < p sat within exp(4 delta / T) - 1 of equality (p
    and q both move) or its inverse-CDF draw within exp(2 delta / T) - 1 of a
    boundary (delta doubled for margin).  The autoregressive transcript is
    compared over all 40 tokens, restarting from the oracle's token at a near
    boundary; speculative ones (four seeds) up to their first difference,
    which must be a near boundary, at least 40 tokens in all."""
    R, B = RB
    s = small_shape("bf16", vocab=500, eos_id=499, prompt=(490, 491, 492, 493))
    tw = synth.target_weights(s, 63)
    dw = synth.drafter_weights(s, 63, tw)
    A = synth.encoder_states(s, 63, 0, frames=160)
    orc = M.Oracle(s, tw, dw)
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=160)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [160])
    T, seed, budget = 0.7, 4242, 40
    ref = M.sampling_plain(orc, orc.new_request(A), budget, T, seed, 0)
    toks = ref.tokens[:-1]
    gpu = teacher_forced_logits(dec, req, s, toks)
    ora, _ = orc.forward_full(orc.new_request(A), list(s.prompt) + toks)
    delta = float(np.abs(gpu - ora).max())
    b = dec.new_batch(req, [64], sampling=True)
    b.prefill()
    r = orc.new_request(A)
    acc, _ = M.prefill(orc, r, 64)
    b.block[0, 0] = acc.next_anchor
    dec.draft(req, b.block, 1.0, 3, 1, b.q_logits)
    delta = max(delta, float(np.abs(b.q_logits[0].cpu().numpy() - orc.draft_logits(r, acc.next_anchor)).max()))
    assert delta < 2e-2 * 4                                # the stated bf16 tolerance, |logits| < 4 here
    d2 = 2.0 * delta
    ca_thr, cc_thr = math.exp(4 * d2 / T) - 1.0, math.exp(2 * d2 / T) - 1.0

    def near(m):
        ca, cc = m
        return ca < ca_thr or cc < cc_thr

    b = dec.new_batch(req, [budget], sampling=True)
    R.run_ar_sampling(dec, b, T, seed)
    n1, _ = tokens_match_resuming(ar_sampling_from(R, dec, req, s, budget, T, seed), ref.tokens, ref.margins, near,
                                  first=b.transcripts()[0])
    assert n1 == budget
    compared = []
    for sd in (seed, seed + 1, seed + 2, seed + 3):        # speculative: four seeds, each up to its first difference
        b2 = dec.new_batch(req, [budget], sampling=True)
        rounds = R.run_spec(dec, b2, temperature=T, seed=sd)
        ref2 = M.speculative_sampling(orc, orc.new_request(A), budget, T, sd, 0)
        n2 = tokens_match(b2.transcripts()[0], ref2.tokens, ref2.margins, near)
        if n2 == len(ref2.tokens):
            assert rounds == ref2.rounds
        compared.append(n2)
    assert sum(compared) >= budget, compared
    print(f"bf16 sampling: delta {delta:.4f}, thresholds {ca_thr:.4f} / {cc_thr:.4f}, spec compared {compared}")
    assert dec.status() == 0
