"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import synth
from oracle import model as M

MARGIN = 1e-3     # near-tie rule: a token may differ where the oracle's top-2 margin is below this
# bf16 configs: logits may differ from the oracle by up to 2e-2 relative, and
# the measured top-2 margin differences at large-v3 (32 layers, |logits| < 3.4)
# reach 9e-3 whatever the fp32 summation order, so there a near tie is a
# margin below 1e-2 (test_large_v3_teacher_forced_margin_error pins the bound).
MARGIN_BF16 = 1e-2


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
    """Exact token equality, except at a first difference where the oracle's
    decision was a near tie (`near(margin)`); there the comparison stops."""
    for i, (g, o) in enumerate(zip(gpu, ora)):
        if g != o:
            assert near(margins[i]), f"token {i}: gpu {g} != oracle {o} with margin {margins[i]}"
            return i
    assert len(gpu) == len(ora), (len(gpu), len(ora))
    return len(gpu)


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
