"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import synth
from oracle import model as M

MARGIN = 1e-3     # near-tie rule: a token may differ where the oracle's top-2 margin is below this
# bf16 configs: logits are only fixed to within 2e-2 of the oracle's, so two
# logits closer than 2e-2 are not resolved by the stated precision: there a
# near tie is a top-2 margin below 2e-2 (the teacher-forced large-v3 test
# asserts that the margin itself moves by less than that at every position).
MARGIN_BF16 = 2e-2


def logits_close(gpu: np.ndarray, ora: np.ndarray, tol: float):
    """Per row: max |g - o| <= tol * max(max |o|, 1).  Returns the worst ratio."""
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1, ora.shape[-1])
    ora = np.asarray(ora, dtype=np.float64).reshape(-1, ora.shape[-1])
    worst = 0.0
    for g, o in zip(gpu, ora):
        err = np.abs(g - o).max()
        scale = max(np.abs(o).max(), 1.0)
        worst = max(worst, err / scale)
    assert worst <= tol, f"logits differ: {worst:.3e} > {tol:.1e}"
    return worst


def greedy_near_tie(m) -> bool:
    return m < MARGIN


def greedy_near_tie_bf16(m) -> bool:
    return m < MARGIN_BF16


def near_tie_for(dtype: str):
    return greedy_near_tie_bf16 if dtype == "bf16" else greedy_near_tie


def sampled_near_boundary(m) -> bool:
    """A sampled token may differ only where the oracle's decision sat within
    the fp32 error of its boundary: the acceptance test u*q < p within 1e-5
    (relative; GPU and oracle probabilities differ by ~1e-6 at fp32 model
    precision) or the inverse-CDF draw within 1e-7 of a boundary (both sides
    sum FP32 probabilities in FP64; their CDFs differ by ~1e-8)."""
    ca, cc = m
    return ca < 1e-5 or cc < 1e-7


def tokens_match(gpu: list, ora: list, margins: list, near=greedy_near_tie):
    """Exact token equality up to the first difference, which must sit where
    the oracle's decision was a near tie (`near(margin)`).  Returns the number
    of positions compared.  Used where the decoding cannot be restarted from
    the oracle's token with the same random stream (speculative sampling,
    whose Philox counters follow the round boundaries)."""
    for i, (g, o) in enumerate(zip(gpu, ora)):
        if g != o:
            assert near(margins[i]), f"token {i}: gpu {g} != oracle {o} with margin {margins[i]}"
            return i
    assert len(gpu) == len(ora), (len(gpu), len(ora))
    return len(gpu)


def tokens_match_resuming(run_from, ora: list, margins: list, near=greedy_near_tie, max_resumes: int = 12,
                          first=None):
    """Emitted tokens compared exactly over the whole transcript; at a
    difference where the oracle's decision was a near tie the GPU decode is
    restarted from the oracle's tokens up to and including that position and
    the comparison goes on from there.  `run_from(prefix)` returns the GPU
    transcript of a decode that starts from `prefix` (prefix included);
    `first`, when given, is the GPU transcript of the unrestarted decode
    (e.g. one request of a batched run), compared over len(ora) tokens.
    Returns (positions compared, restarts)."""
    prefix: list = []
    gpu = list(first[:len(ora)]) if first is not None else run_from(prefix)
    resumes = 0
    while True:
        n = min(len(gpu), len(ora))
        diff = next((k for k in range(len(prefix), n) if gpu[k] != ora[k]), None)
        if diff is None:
            assert len(gpu) == len(ora), (len(gpu), len(ora))
            return len(ora), resumes
        assert near(margins[diff]), f"token {diff}: gpu {gpu[diff]} != oracle {ora[diff]} with margin {margins[diff]}"
        resumes += 1
        assert resumes <= max_resumes, f"more than {max_resumes} near ties"
        prefix = list(ora[:diff + 1])
        gpu = run_from(prefix)
        assert gpu[:len(prefix)] == prefix


def force_prefix(dec, req, s, prefix: list):
    """Enter the prompt and prefix[:-1] into request `req`'s cache by forced
    verification (one block for the prompt, then one row per token): the
    cache state greedy decoding leaves after emitting those tokens.  The
    caller makes prefix[-1] the next anchor."""
    import speculative_whisper_asr_gb300.binding as B
    stream = torch.cuda.current_stream().cuda_stream
    dec.reset(req)
    scratch = dec.new_batch(req, [10 ** 6])
    for block in [list(s.prompt)] + [[t] for t in prefix[:-1]]:
        H = len(block)
        blk, bl = dev_i32([block]), dev_i32([H])
        t = torch.zeros(1, H, dtype=torch.int32, device="cuda")
        dec.verify(req, blk, bl, t)
        a = scratch._args(B.WS_ACCEPT_FORCED, H, blk, bl, t, scratch.block1, scratch.blen)
        B.ws_accept(dec.ctx, 1, req.data_ptr(), a, stream)


def ar_from(R, dec, req, s, budget: int):
    """`run_from` for tokens_match_resuming: one request's autoregressive
    greedy decode of `budget` tokens on the GPU, restartable from a prefix."""
    def run(prefix):
        if not prefix:
            b = dec.new_batch(req, [budget])
            R.run_ar(dec, b)
            return b.transcripts()[0]
        left = budget - len(prefix)
        if left <= 0 or prefix[-1] == s.eos_id:
            return list(prefix)
        force_prefix(dec, req, s, prefix)
        b = dec.new_batch(req, [left])
        b.block1[0, 0] = int(prefix[-1])
        b.blen[0] = 1
        while b.poll_done() < 1:
            b.ar_step(graph=False)
        return list(prefix) + b.transcripts()[0]
    return run


def ar_sampling_from(R, dec, req, s, budget: int, T: float, seed: int):
    """`run_from` for autoregressive sampling: token r of the transcript is
    drawn in round r (Philox counter (slot, r, 1, 2)), so a restart from the
    oracle's first r tokens continues with round r on both sides."""
    def run(prefix):
        if not prefix:
            b = dec.new_batch(req, [budget], sampling=True)
            R.run_ar_sampling(dec, b, T, seed)
            return b.transcripts()[0]
        left = budget - len(prefix)
        if left <= 0 or prefix[-1] == s.eos_id:
            return list(prefix)
        force_prefix(dec, req, s, prefix)
        b = dec.new_batch(req, [left], sampling=True)
        b.block1[0, 0] = int(prefix[-1])
        b.blen[0] = 1
        rnd = len(prefix)
        while b.poll_done() < 1:
            b.ar_sample_step(rnd, T, seed)
            rnd += 1
        return list(prefix) + b.transcripts()[0]
    return run


def small_shape(dtype="f32", **kw):
    """Multi-tile shape with ragged tails: vocab 1000 is not a multiple of the
    64-feature GEMM tile, 4 heads, FFN 512."""
    args = dict(name="small", n_layers=3, d_model=256, n_heads=4, d_ff=512, vocab=1000, max_pos=96,
                hist_layers=(0, 2), dtype=dtype, eos_id=999, prompt=(990, 991, 992, 993))
    args.update(kw)
    return synth.ModelShape(**args)


def dev_i32(a, dev="cuda"):
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device=dev)


def teacher_forced_logits(dec, req, s, tokens):
    """Logits of the one-request AR path fed the given tokens: the prompt
    block, then one verify per token, each followed by a forced accept (the
    cache advances exactly as in greedy decoding).  Returns [4 + len(tokens), V]
    rows aligned with the oracle's forward_full over prompt + tokens."""
    import speculative_whisper_asr_gb300.binding as B
    stream = torch.cuda.current_stream().cuda_stream
    dec.reset(req)
    b = dec.new_batch(req, [10 ** 6])
    out = []

    def step(block):
        H = len(block)
        blk = dev_i32([block])
        bl = dev_i32([H])
        t = torch.zeros(1, H, dtype=torch.int32, device="cuda")
        lg = torch.empty(1, H, s.vocab, device="cuda")
        dec.verify(req, blk, bl, t, lg)
        a = b._args(B.WS_ACCEPT_FORCED, H, blk, bl, t, b.block1, b.blen)
        B.ws_accept(dec.ctx, 1, req.data_ptr(), a, stream)
        out.append(lg[0].cpu().numpy())

    step(list(s.prompt))
    for tok in tokens:
        step([tok])
    return np.concatenate(out)
