"""GPU parity for the sampling path and the batched / varlen workloads.

  * rejection-rule acceptance and the drafter's sampler element by element
    against the oracle on shared logits (decisions compared exactly except
    where the uniform lies within 1e-5 (acceptance test, relative) or 1e-7
    (inverse-CDF draw, fraction of the mass) of a decision boundary);
  * temperature sampling end to end on the tiny fp32 model: GPU transcripts
    equal the oracle's (autoregressive and speculative, same Philox streams);
  * the large-v3 batch-96 sampling study: 10^5 first tokens after a fixed
    prefix at T = 0.7 with drafter logits = target logits + N(0, 1), checked
    against the oracle's target distribution with a chi-square test
    (200 equal-mass bins, 199 dof, alpha = 1e-3);
  * large-v3-turbo, batch 16, transcript lengths U[40, 224], drafter run +
    continuation drafts with corruption 0.1 -> 0.5;
  * varlen batch of 64 turbo requests (frames U[250, 1500]): packed and
    padded runs give the same transcripts as autoregressive decoding.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from oracle import philox
from gpu_common import (ar_from, ar_sampling_from, dev_i32, greedy_near_tie_bf16, logits_close,
                        sampled_near_boundary, small_shape, tokens_match, tokens_match_resuming)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def RB():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding, runtime
    return runtime, binding


def _stream():
    return torch.cuda.current_stream().cuda_stream


# ---------------------------------------------------------------- element-wise sampling parity

def _near_boundary(det, eps=1e-5):
    for d in det:
        if d[0] == "accept":
            _, j, u, q, p, acc = d
            if abs(u * q - p) <= eps * max(p, 1e-30):
                return True
    return False


def _cdf_margin(w, u):
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    t = u * c[-1]
    return np.min(np.abs(c - t)) / c[-1]


def test_accept_and_sampler_match_oracle(RB):
    R, B = RB
    s = small_shape("f32", n_layers=1, vocab=2000)
    tw = synth.target_weights(s, 51)
    dec = R.Decoder(s, tw, None, max_batch=64, max_frames=32)
    n, K, V, T, seed = 64, s.K, s.vocab, 0.7, 12345
    g = np.random.default_rng(5)
    zp = (g.standard_normal((n, K + 1, V)) * 2).astype(np.float32)
    zq = (zp[:, :K] + g.standard_normal((n, K, V))).astype(np.float32)
    req = dec.slots(list(range(n)))
    # drafter sampler
    draft = torch.zeros(n, K, dtype=torch.int32, device="cuda")
    dec.sample(req, torch.as_tensor(zq, device="cuda"), T, seed, 3, draft)
    draft = draft.cpu().numpy()
    checked = 0
    for i in range(n):
        for j in range(K):
            qv = M.probs_fp32(zq[i, j], T)
            u = float(philox.uniform(seed, i, 3, j + 1, philox.PURPOSE_DRAFT))
            if _cdf_margin(qv, u) < 1e-7:
                continue
            assert draft[i, j] == M.sample_draft(zq[i, j], T, seed, i, 3, j + 1)
            checked += 1
    assert checked > 0.95 * n * K
    # acceptance with the rejection rule; half the candidates copied from the
    # target argmax so that both branches (accept / residual) occur
    block = np.zeros((n, K + 1), dtype=np.int32)
    block[:, 1:] = draft
    block[::2, 1:4] = zp[::2, 0:3].argmax(-1)
    blen = g.integers(1, K + 2, size=n).astype(np.int32)
    budget = np.full(n, 1000, dtype=np.int32)
    b = dec.new_batch(req, budget, sampling=True)
    b.p_logits.copy_(torch.as_tensor(zp, device="cuda"))
    b.q_logits.copy_(torch.as_tensor(zq, device="cuda"))
    bt = torch.as_tensor(block, device="cuda")
    bl = torch.as_tensor(blen, device="cuda")
    dec.reset(req)
    a = b._args(B.WS_ACCEPT_SAMPLE, K + 1, bt, bl, None, b.block, b.blen, b.p_logits, b.q_logits, T, seed, 9)
    B.ws_accept(dec.ctx, n, req.data_ptr(), a, _stream())
    got_a, got_ne = b.n_acc.cpu().numpy(), b.n_emit.cpu().numpy()
    got_tr = b.transcripts()
    compared, accepted_any, rejected_any = 0, 0, 0
    for i in range(n):
        acc, det = M.accept_sampling(block[i], blen[i] - 1, zp[i], zq[i], T, seed, i, 9, 1000, s.eos_id)
        if _near_boundary(det):
            continue
        if any(d[0] in ("residual", "bonus") and _cdf_margin(
                np.maximum(M.probs_fp32(zp[i, d[1] - 1], T) - (M.probs_fp32(zq[i, d[1] - 1], T) if d[0] == "residual"
                                                                else 0), 0), d[2]) < 1e-7 for d in det):
            continue
        assert got_a[i] == acc.a and got_tr[i] == acc.emitted, (i, got_a[i], acc.a, got_tr[i], acc.emitted)
        compared += 1
        accepted_any += acc.a > 0
        rejected_any += any(d[0] == "residual" for d in det)
    assert compared > 0.9 * n and accepted_any > 0 and rejected_any > 0
    lens = dec.lengths(req)
    assert list(lens) == list(1 + got_a)


def test_tiny_sampling_transcripts_match_oracle(RB):
    R, B = RB
    s = synth.TINY
    tw = synth.target_weights(s, 0)
    dw = synth.drafter_weights(s, 0, tw)
    A = synth.encoder_states(s, 0, 0)
    orc = M.Oracle(s, tw, dw)
    dec = R.Decoder(s, tw, dw, max_batch=2, max_frames=1500)
    req = dec.slots([1])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    T, seed, budget = 0.7, 777, 40
    b = dec.new_batch(req, [budget], sampling=True)
    R.run_ar_sampling(dec, b, T, seed)
    ref = M.sampling_plain(orc, orc.new_request(A), budget, T, seed, 1)
    assert len(ref.margins) == len(ref.tokens)
    n1, _ = tokens_match_resuming(ar_sampling_from(R, dec, req, s, budget, T, seed), ref.tokens, ref.margins,
                                  sampled_near_boundary, first=b.transcripts()[0])
    assert n1 == budget
    b2 = dec.new_batch(req, [budget], sampling=True)
    rounds = R.run_spec(dec, b2, temperature=T, seed=seed)
    ref2 = M.speculative_sampling(orc, orc.new_request(A), budget, T, seed, 1)
    n2 = tokens_match(b2.transcripts()[0], ref2.tokens, ref2.margins, sampled_near_boundary)
    if n2 == len(ref2.tokens):
        assert rounds == ref2.rounds
    assert n2 >= 10        # a boundary case this early would be suspicious
    assert dec.status() == 0


def test_large_v3_batch96_first_token_chi_square(RB):
    """Config: large-v3 bf16, 96 request slots, T = 0.7, drafter logits =
    target logits + N(0,1).  The first emitted token of a speculative round
    (accepted candidate or residual draw) must follow the target's softmax."""
    R, B = RB
    from scipy.stats import chi2
    s = synth.LARGE_V3
    tw = synth.target_weights(s, 1)
    A = synth.encoder_states(s, 1, 0)
    n, T, seed, V, K = 96, 0.7, 2024, s.vocab, s.K
    dec = R.Decoder(s, tw, None, max_batch=n, max_frames=1500)
    req = dec.slots(list(range(n)))
    enc = dec.enc_tensor(A)
    dec.cross_kv(req, enc.repeat(n, 1), [1500] * n)
    dec.reset(req)
    H = len(s.prompt)
    tgt = torch.zeros(n, H, dtype=torch.int32, device="cuda")
    lg = torch.empty(n, H, V, device="cuda")
    dec.verify(req, dev_i32([s.prompt] * n), dev_i32([H] * n), tgt, lg)
    z = lg[:, H - 1].contiguous()                                    # target logits after the prefix
    assert torch.equal(z[0], z[n - 1])
    eps = torch.as_tensor(synth.gaussian_noise((V,), 99), device="cuda")
    b = dec.new_batch(req, [10 ** 6] * n, tcap=2, sampling=True)
    b.p_logits[:, 0].copy_(z)
    b.p_logits[:, 1].copy_(z)
    b.q_logits[:, 0].copy_(z + eps)
    qrow = b.q_logits[:, :1].contiguous()
    blk = torch.zeros(n, K + 1, dtype=torch.int32, device="cuda")
    bl = torch.full((n,), 2, dtype=torch.int32, device="cuda")
    cand = torch.zeros(n, 1, dtype=torch.int32, device="cuda")
    trials = math.ceil(100000 / n)
    counts = torch.zeros(V, dtype=torch.int64, device="cuda")
    for r in range(1, trials + 1):
        dec.sample(req, qrow, T, seed, r, cand)
        blk[:, 1] = cand[:, 0]
        b.done.zero_(); b.out_len.zero_()
        a = b._args(B.WS_ACCEPT_SAMPLE, K + 1, blk, bl, None, b.block, b.blen, b.p_logits, b.q_logits, T, seed, r)
        B.ws_accept(dec.ctx, n, req.data_ptr(), a, _stream())
        counts += torch.bincount(b.transcript[:, 0].long(), minlength=V)
    counts = counts.cpu().numpy().astype(np.float64)
    N = counts.sum()
    assert N == trials * n
    # the oracle's target distribution at the same prefix (bf16 storage points)
    orc = M.Oracle(s, tw, None)
    zo = orc.verify(orc.new_request(A), list(s.prompt))[H - 1]
    p = M.probs_fp32(zo, T).astype(np.float64)
    order = np.argsort(-p)
    cp = np.cumsum(p[order])
    bins = np.minimum((cp * 200).astype(int), 199)
    obs = np.bincount(bins, weights=counts[order], minlength=200)
    exp = np.bincount(bins, weights=p[order], minlength=200) * N
    keep = exp > 0
    stat = float(((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum())
    dof = int(keep.sum()) - 1
    assert stat < chi2.ppf(1 - 1e-3, dof), (stat, dof)


# ---------------------------------------------------------------- turbo batch 16

def test_turbo_batch16_continuation_drafts(RB):
    R, B = RB
    s = synth.TURBO
    tw = synth.target_weights(s, 1)
    dw = synth.drafter_weights(s, 1, tw)
    n = 16
    budgets = synth.budgets_uniform(n, 40, 224, 3)
    As = [synth.encoder_states(s, 1, i) for i in range(n)]
    dec = R.Decoder(s, tw, dw, max_batch=n, max_frames=1500)
    req = dec.slots(list(range(n)))
    dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in As]), [1500] * n)
    b = dec.new_batch(req, budgets)
    R.run_ar(dec, b)
    ar = b.transcripts()
    assert [len(t) for t in ar] == list(budgets)
    traj = np.zeros((n, s.max_pos), dtype=np.int32)
    for i in range(n):
        t = list(s.prompt) + ar[i]
        traj[i, :len(t)] = t
    pj = synth.corruption_p_linear(s.K, 0.1, 0.5)
    plan = synth.corruption_plan(n, s.max_pos, s.K, pj, s.vocab, 17)
    syn = tuple(torch.as_tensor(x, device="cuda") for x in (traj, plan.mask, plan.tok))
    b2 = dec.new_batch(req, budgets)
    rounds = R.run_spec(dec, b2, synthetic=syn)
    assert b2.transcripts() == ar
    expect_tau = 1 + sum(np.prod(1 - pj[:k]) for k in range(1, s.K + 1))    # 4.31
    tau = sum(budgets) / float(rounds * n)
    assert rounds < max(budgets) / 2.5
    orc = M.Oracle(s, tw, None)
    for i in (0, n - 1):
        ref = M.greedy_cached(orc, orc.new_request(As[i]), 32)
        cnt, _ = tokens_match_resuming(ar_from(R, dec, dec.slots([i]), s, 32), ref.tokens, ref.margins,
                                       greedy_near_tie_bf16, first=ar[i])
        assert cnt == 32
    assert dec.status() == 0


# ---------------------------------------------------------------- varlen batch 64

def test_varlen_batch64_packed_and_padded(RB):
    R, B = RB
    s = synth.TURBO
    tw = synth.target_weights(s, 1)
    dw = synth.drafter_weights(s, 1, tw)
    n = 64
    F, budgets = synth.varlen_frames_and_budgets(n, 5)
    As = [synth.encoder_states(s, 1, i, frames=int(F[i])) for i in range(n)]
    dec = R.Decoder(s, tw, dw, max_batch=n, max_frames=1500)
    req = dec.slots(list(range(n)))
    # packed acoustic K/V: only the valid frames of each request
    dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in As]), F)
    b = dec.new_batch(req, budgets)
    R.run_ar(dec, b)
    ar = b.transcripts()
    traj = np.zeros((n, s.max_pos), dtype=np.int32)
    for i in range(n):
        t = list(s.prompt) + ar[i]
        traj[i, :len(t)] = t
    plan = synth.corruption_plan(n, s.max_pos, s.K, synth.corruption_p_linear(s.K), s.vocab, 23)
    syn = tuple(torch.as_tensor(x, device="cuda") for x in (traj, plan.mask, plan.tok))
    packed, rounds_p, rows_p = R.run_spec_packed(dec, req, budgets, synthetic=syn)
    assert packed == ar
    # padded: every request carries 1500 frames (masked beyond F) and stays in the batch
    pad = [np.concatenate([a, np.zeros((1500 - a.shape[0], s.d_model), dtype=np.float32)]) for a in As]
    dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in pad]), [1500] * n, valid=F)
    b3 = dec.new_batch(req, budgets)
    rounds_pad = R.run_spec(dec, b3, synthetic=syn)
    assert b3.transcripts() == ar
    assert rows_p < rounds_pad * n * (s.K + 1)
    orc = M.Oracle(s, tw, None)
    i = int(np.argmin(F))
    nb = min(32, int(budgets[i]))
    ref = M.greedy_cached(orc, orc.new_request(As[i]), nb)
    dec.cross_kv(dec.slots([i]), dec.enc_tensor(As[i]), [int(F[i])])     # packed again for the restarts
    cnt, _ = tokens_match_resuming(ar_from(R, dec, dec.slots([i]), s, nb), ref.tokens, ref.margins,
                                   greedy_near_tie_bf16, first=ar[i])
    assert cnt == nb
    assert dec.status() == 0
