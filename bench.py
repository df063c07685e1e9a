"""Benchmark: accepted decoder tokens/s of speculative Whisper decoding.

One step = the whole decoding path over one batch of synthetic requests:
per-request acoustic K/V (ws_cross_kv), prompt prefill, then propose /
verify / accept rounds (ws_draft with the two-layer parallel drafter,
synthetic proposals from the target's own greedy trajectory, ws_verify,
ws_accept) until every transcript is finished.

Default workload: Whisper-large-v3-shaped decoder, bf16, batch 1, 224-token
transcripts, K = 8, proposals corrupted independently with p = 0.2.
Weights are random N(0, 0.02), encoder states N(0, 1) (seeded).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  --impl reference  times the CPU oracle (the reference arm) on a bounded
                    sample of the same workload.
The default line also carries, under "workloads", the batch-96 sampling
workload (large-v3, T = 0.7, rejection rule) and the batch-16 turbo workload
of the same metric, and the large-v3 audio encoder (the step before the
path) at 1 and 16 windows with its share of request time (--no-sub leaves
them out).  Timed steps of the headline
cycle through four corruption plans, so tau is an average over plans.
Under torchrun (N > 1) every rank decodes its own batch (weak scaling); the
time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "accepted decoder tokens/s at batch 1/16/96; verify-step HBM GB/s vs peak"
SEED = 1
BUDGET = 224
P_CORRUPT = 0.2
N_PLANS = 4          # corruption plans; step k uses plan k mod 4, so tau averages over plans


class Workload:
    """One measured configuration: model shape, batch, transcript lengths,
    acoustic frames per request and how proposals are made."""

    def __init__(self, name, shape, n, budgets, frames, pj=None, temperature=0.0, text=""):
        self.name, self.shape, self.n = name, shape, n
        self.budgets = np.asarray(budgets, dtype=np.int32)
        self.frames = np.asarray(frames, dtype=np.int32)
        self.pj = None if pj is None else np.asarray(pj, dtype=np.float64)
        self.temperature = temperature
        self.text = text

    def config(self):
        return {"workload": self.text, "global_batch": self.n, "seq_len": int(self.budgets.max()),
                "K": self.shape.K, "frames": int(self.frames.max()),
                "l2": "no flush: every step streams the decoder weights (>= 0.3 GB) and the acoustic K/V "
                      "(>= 0.25 GB per large-v3 request), larger than the 129 MB L2"}


def make_workload(name: str, batch: int = 1) -> Workload:
    if name == "large-v3-b1":
        return Workload(name, synth.LARGE_V3, batch, [BUDGET] * batch, [1500] * batch,
                        synth.corruption_p_const(synth.LARGE_V3.K, P_CORRUPT),
                        text=f"whisper-large-v3-shaped decoder, bf16, batch {batch}, {BUDGET}-token transcripts, "
                             f"K=8, 2-layer parallel drafter run + synthetic proposals (p={P_CORRUPT}), "
                             f"1500-frame encoder states")
    if name == "turbo-b16":
        s = synth.TURBO
        return Workload(name, s, 16, synth.budgets_uniform(16, 40, 224, 3), [1500] * 16,
                        synth.corruption_p_linear(s.K),
                        text="whisper-large-v3-turbo-shaped decoder (4 layers), bf16, batch 16, transcripts "
                             "U[40,224] tokens, K=8, 2-layer drafter run + continuation proposals "
                             "(p_j 0.1..0.5), 1500-frame encoder states")
    if name == "large-v3-b96-t0.7":
        return Workload(name, synth.LARGE_V3, 96, [BUDGET] * 96, [1500] * 96, None, temperature=0.7,
                        text="whisper-large-v3-shaped decoder, bf16, batch 96, 224-token transcripts, K=8, "
                             "2-layer drafter sampling q at T=0.7, rejection-rule acceptance, 1500-frame "
                             "encoder states")
    if name == "turbo-b64-varlen":
        F, bud = synth.varlen_frames_and_budgets(64, 5)
        return Workload(name, synth.TURBO, 64, bud, F, synth.corruption_p_linear(synth.TURBO.K),
                        text="whisper-large-v3-turbo-shaped decoder, bf16, batch 64 varlen: frames U{250..1500}, "
                             "transcripts F/1500*200 +-20%, K=8, drafter run + continuation proposals, "
                             "packed (frames and finished requests dropped)")
    raise ValueError(name)


WORKLOADS = ("large-v3-b1", "turbo-b16", "large-v3-b96-t0.7", "turbo-b64-varlen")


def workload(batch: int):
    return make_workload("large-v3-b1", batch).config()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------- algorithmic bytes
def verify_bytes(s: synth.ModelShape, n_req: int, H: int, L_mean: float, frames: int = 1500) -> float:
    """Bytes one ws_verify must move at least: every weight once (layers +
    tied LM head), each request's acoustic K/V for every layer, its self K/V
    up to the block, plus the logits-free outputs (negligible)."""
    d, f, nl = s.d_model, s.d_ff, s.n_layers
    es = 2
    w_layer = (3 * d * d + d * d + d * d + d * d + d * f + f * d) * es   # w_kvc is only read by ws_cross_kv
    weights = nl * w_layer + s.vocab * d * es
    xkv = n_req * nl * 2 * frames * d * es
    skv = n_req * nl * 2 * (L_mean + H) * d * es
    return float(weights + xkv + skv)


def tau_closed_form(pj) -> float | None:
    """Expected tokens per verify of a full round with independent
    corruption probabilities p_j: 1 + sum_k prod_{j<=k} (1 - p_j) (chance
    matches of a random token, ~1/V, ignored)."""
    if pj is None:
        return None
    return float(1.0 + sum(np.prod(1.0 - np.asarray(pj)[:k]) for k in range(1, len(pj) + 1)))


# ---------------------------------------------------------------- clocks
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.idx = dev_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- multi-rank
def rank_requests(rank: int, n: int) -> list:
    """Each rank decodes its own batch of n requests (weak scaling): request
    ids rank*n .. rank*n+n-1 seed its encoder states."""
    return [rank * n + i for i in range(n)]


def reduce_over_ranks(ms: float, ms_e2e: float, tokens: int, world: int, device):
    """Whole-job numbers: the slowest rank's times, the sum of tokens."""
    if world <= 1:
        return ms, ms_e2e, float(tokens)
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, ms_e2e], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    tt = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(tt)
    return float(t[0]), float(t[1]), float(tt[0])


# ---------------------------------------------------------------- GPU arm
_WEIGHTS: dict = {}


def _weights(s: synth.ModelShape, with_drafter: bool):
    """Seeded target (and drafter) weights of a shape, drawn once per process."""
    if s.name not in _WEIGHTS:
        _WEIGHTS.clear()
        tw = synth.target_weights(s, SEED)
        _WEIGHTS[s.name] = (tw, synth.drafter_weights(s, SEED, tw))
    tw, dw = _WEIGHTS[s.name]
    return tw, (dw if with_drafter else None)


def _setup(wl: Workload, rank: int, with_drafter: bool = True, max_frames: int | None = None):
    """Context, request slots and pinned host encoder states of one workload."""
    import torch
    from speculative_whisper_asr_gb300 import runtime as R
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    dev = torch.device("cuda", torch.cuda.current_device())
    s, n = wl.shape, wl.n
    tw, dw = _weights(s, with_drafter)
    dec = R.Decoder(s, tw, dw, max_batch=n, max_frames=max_frames or int(wl.frames.max()))
    req = dec.slots(list(range(n)))
    ids = rank_requests(rank, n)
    As = [synth.encoder_states(s, SEED, ids[i], frames=int(wl.frames[i])) for i in range(n)]
    host_enc = torch.from_numpy(np.concatenate([synth.bf16_bits(a) for a in As])).view(torch.int16).pin_memory()
    return dec, req, host_enc, stream, dev


def _trajectory_plan(dec, req, wl: Workload, rank: int, dev):
    """The target's own greedy transcripts (untimed) and, from them, the
    corrupted-proposal tensors (reference trajectory, mask, random tokens)."""
    import torch
    from speculative_whisper_asr_gb300 import runtime as R
    s, n = wl.shape, wl.n
    b_ar = dec.new_batch(req, wl.budgets)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    R.run_ar(dec, b_ar)
    torch.cuda.synchronize()
    ar_time = time.perf_counter() - t0
    ar = b_ar.transcripts()
    traj = np.zeros((n, s.max_pos), dtype=np.int32)
    for i in range(n):
        t = list(s.prompt) + ar[i]
        traj[i, :len(t)] = t
    plans = [synth.corruption_plan(n, s.max_pos, s.K, wl.pj, s.vocab, SEED + 100 + 10 * rank + k)
             for k in range(N_PLANS)]
    syn = (torch.as_tensor(traj, device=dev), torch.as_tensor(plans[0].mask, device=dev),
           torch.as_tensor(plans[0].tok, device=dev))
    stacked = (torch.as_tensor(np.stack([p.mask for p in plans]), device=dev),
               torch.as_tensor(np.stack([p.tok for p in plans]), device=dev))
    return ar, syn, ar_time, stacked


def _timed(step, steps, world, stream):
    """Barrier, then `steps` calls of step() between CUDA events on the
    launching stream, with the clocks sampled meanwhile."""
    import torch
    from speculative_whisper_asr_gb300 import binding as B
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    l0 = B.ws_launch_count()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = []
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.nvtx.range_push("ws_timed")        # lets a profiler restrict itself to the timed steps
        t0.record(stream)
        for _ in range(steps):
            out.append(step())
        t1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    return t0.elapsed_time(t1), B.ws_launch_count() - l0, clk.summary(), out


def run_gpu(args, rank: int, world: int, wl: Workload):
    """Greedy decoding with synthetic proposals (the headline workload and
    turbo batch 16): every timed step repeats the whole path and its
    transcripts equal the autoregressive ones."""
    import torch
    from speculative_whisper_asr_gb300 import binding as B

    dec, req, host_enc, stream, dev = _setup(wl, rank)
    s, n = wl.shape, wl.n
    enc = host_enc.to(dev).view(torch.bfloat16)
    maxF, totF = int(wl.frames.max()), int(wl.frames.sum())
    cu, _ = dec.cross_kv(req, enc, wl.frames)
    ar, syn, ar_time, plans = _trajectory_plan(dec, req, wl, rank, dev)
    n_step = [0]

    batch = dec.new_batch(req, wl.budgets)
    budgets = torch.as_tensor(wl.budgets, device=dev)
    ev_v = []
    live = torch.zeros(n, dtype=torch.int64, device=dev)
    acc = torch.zeros(n, dtype=torch.int64, device=dev)
    prop = torch.zeros(n, dtype=torch.int64, device=dev)

    def draft_calls():
        dec.draft(req, batch.block, 0.0, 0, 0, None)
        B.ws_draft_synthetic(dec.ctx, n, req.data_ptr(), batch.block.data_ptr(), syn[0].data_ptr(),
                             syn[0].shape[1], syn[1].data_ptr(), syn[2].data_ptr(), stream.cuda_stream)

    def accept_calls():
        a = batch._args(B.WS_ACCEPT_GREEDY, s.K + 1, batch.block, batch.blen, batch.target, batch.block,
                        batch.blen)
        B.ws_accept(dec.ctx, n, req.data_ptr(), a, stream.cuda_stream)

    def step(record=False, e2e=False, stats=False):
        """One pass of the whole path; returns the number of rounds."""
        if e2e:
            enc.view(torch.int16).copy_(host_enc, non_blocking=True)
        k = n_step[0] % N_PLANS            # this step's corruption plan (device-to-device, ~0.2 MB)
        n_step[0] += 1
        syn[1].copy_(plans[0][k], non_blocking=True)
        syn[2].copy_(plans[1][k], non_blocking=True)
        B.ws_cross_kv(dec.ctx, n, req.data_ptr(), enc.data_ptr(), cu.data_ptr(), None, maxF, totF,
                      stream.cuda_stream)
        batch.budget.copy_(budgets)
        batch.done.zero_(); batch.out_len.zero_(); batch.n_done.zero_()
        batch.prefill()
        rnd = 0
        while batch.poll_done() < n:
            rnd += 1
            if stats:                       # untimed bookkeeping for tau and alpha
                live.add_((batch.done == 0).long())
                prop.add_((batch.blen - 1).clamp(min=0))
            # each phase of the round replays its own captured graph (greedy
            # rounds do not depend on the round number)
            batch.replay("draft", draft_calls)
            if record:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            batch.replay("verify", lambda: dec.verify(req, batch.block, batch.blen, batch.target))
            if record:
                e1.record(stream)
                ev_v.append((e0, e1))
            batch.replay("accept", accept_calls)
            if stats:
                acc.add_(batch.n_acc)
        if e2e:
            out = batch.transcript.to("cpu", non_blocking=True)
            torch.cuda.current_stream().synchronize()
            _ = out.numpy().sum()
        return rnd

    for w in range(args.warmup):
        step(stats=True)
    spec = batch.transcripts()
    assert spec == ar, "speculative transcript differs from autoregressive"
    n_step[0] = 0

    # ---- device-resident timed region
    ms, launches, clocks, rounds = _timed(lambda: step(record=True), args.steps, world, stream)
    tokens = int(batch.out_len.sum().item()) * args.steps
    # ---- end to end: host encoder states in, host transcript out
    ms_e2e, _, _, _ = _timed(lambda: step(e2e=True), args.steps, world, stream)

    vt = [a.elapsed_time(b) for a, b in ev_v]
    L_mean = len(s.prompt) + float(wl.budgets.mean()) / 2.0
    vbytes = verify_bytes(s, n, s.K + 1, L_mean, float(wl.frames.mean()))
    hbm, bf16_tf, src = peaks()
    v_ms = float(np.mean(vt))
    achieved = vbytes / (v_ms * 1e-3) / 1e9

    ms, ms_e2e, tokens_all = reduce_over_ranks(ms, ms_e2e, tokens, world, dev)
    value = tokens_all / (ms * 1e-3)
    e2e_val = tokens_all / (ms_e2e * 1e-3)
    audio_s = float(wl.frames.sum()) * 0.02 * args.steps * world
    n_live = float(live.sum().item())
    return {
        "value": value, "ms_per_step": ms / args.steps, "e2e": e2e_val,
        "h2d": int(host_enc.numel() * 2), "d2h": int(batch.transcript.numel() * 4),
        "launches": int(launches),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": None, "kernel": "ws_verify (one block verification, all its kernels)",
                     "algorithmic_bytes_per_launch": vbytes, "avg_ms": v_ms, "launches_timed": len(vt),
                     "peak_source": src},
        "clocks": clocks,
        "extra": {"rounds_per_step": float(np.mean(rounds)),
                  "tau": float(wl.budgets.sum()) * args.warmup / n_live,
                  "tau_closed_form": tau_closed_form(wl.pj),
                  "tau_note": f"measured over the warm-up steps, corruption plans 0..{min(args.warmup, N_PLANS) - 1}; "
                              f"closed form 1 + sum_k prod_(j<=k) (1 - p_j) for rounds not cut by the budget",
                  "alpha": float(acc.sum().item()) / max(1.0, float(prop.sum().item())),
                  "audio_seconds_per_s": audio_s / (ms * 1e-3),
                  "ar_tokens_per_s_untimed_host_loop": float(wl.budgets.sum()) / ar_time,
                  "gemm_engine": dec.engine, "verify_ms": v_ms},
    }


def run_sampling(args, rank: int, world: int, wl: Workload):
    """Sampling at temperature T with the rejection rule: the drafter samples
    its proposals from q = softmax(z_q / T) and ws_accept accepts or
    resamples against p = softmax(z_p / T); both logits tensors are fp32."""
    import torch
    from speculative_whisper_asr_gb300 import binding as B

    dec, req, host_enc, stream, dev = _setup(wl, rank)
    s, n, T, seed = wl.shape, wl.n, wl.temperature, 7
    enc = host_enc.to(dev).view(torch.bfloat16)
    maxF, totF = int(wl.frames.max()), int(wl.frames.sum())
    cu, _ = dec.cross_kv(req, enc, wl.frames)
    batch = dec.new_batch(req, wl.budgets, sampling=True)
    budgets = torch.as_tensor(wl.budgets, device=dev)
    ev_v = []
    live = torch.zeros(n, dtype=torch.int64, device=dev)
    acc = torch.zeros(n, dtype=torch.int64, device=dev)
    prop = torch.zeros(n, dtype=torch.int64, device=dev)

    def step(record=False, stats=False):
        B.ws_cross_kv(dec.ctx, n, req.data_ptr(), enc.data_ptr(), cu.data_ptr(), None, maxF, totF,
                      stream.cuda_stream)
        batch.budget.copy_(budgets)
        batch.done.zero_(); batch.out_len.zero_(); batch.n_done.zero_()
        batch.prefill(temperature=T, seed=seed)
        rnd = 0
        while batch.poll_done() < n:
            rnd += 1
            if stats:
                live.add_((batch.done == 0).long())
                prop.add_((batch.blen - 1).clamp(min=0))
            dec.draft(req, batch.block, T, seed, rnd, batch.q_logits)
            if record:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            dec.verify(req, batch.block, batch.blen, batch.target, batch.p_logits)
            if record:
                e1.record(stream)
                ev_v.append((e0, e1))
            a = batch._args(B.WS_ACCEPT_SAMPLE, s.K + 1, batch.block, batch.blen, batch.target, batch.block,
                            batch.blen, batch.p_logits, batch.q_logits, T, seed, rnd)
            B.ws_accept(dec.ctx, n, req.data_ptr(), a, stream.cuda_stream)
            if stats:
                acc.add_(batch.n_acc)
        return rnd

    for w in range(args.warmup):
        step(stats=(w == 0))
    ms, launches, clocks, rounds = _timed(lambda: step(record=True), args.steps, world, stream)
    tokens = int(batch.out_len.sum().item()) * args.steps
    vt = [a.elapsed_time(b) for a, b in ev_v]
    v_ms = float(np.mean(vt))
    L_mean = len(s.prompt) + float(wl.budgets.mean()) / 2.0
    vbytes = verify_bytes(s, n, s.K + 1, L_mean, float(wl.frames.mean()))
    hbm, bf16_tf, src = peaks()
    d, f, nl = s.d_model, s.d_ff, s.n_layers
    rows = n * (s.K + 1)
    vflops = 2.0 * rows * (nl * (6 * d * d + 2 * d * f) + s.vocab * d)
    ms, _, tokens_all = reduce_over_ranks(ms, ms, tokens, world, dev)
    return {
        "value": tokens_all / (ms * 1e-3), "ms_per_step": ms / args.steps, "launches": int(launches),
        "roofline": {"bound": "hbm", "achieved": vbytes / (v_ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": vbytes / (v_ms * 1e-3) / 1e9 / hbm, "traffic": None,
                     "kernel": "ws_verify (one block verification, all its kernels, fp32 logits written)",
                     "algorithmic_bytes_per_launch": vbytes, "avg_ms": v_ms, "launches_timed": len(vt),
                     "peak_source": src,
                     "tensor": {"flops_per_launch": vflops, "achieved_tflops": vflops / (v_ms * 1e-3) / 1e12,
                                "peak_tflops": bf16_tf,
                                "frac": vflops / (v_ms * 1e-3) / 1e12 / bf16_tf}},
        "clocks": clocks,
        "extra": {"rounds_per_step": float(np.mean(rounds)),
                  "tau": float(wl.budgets.sum()) / float(live.sum().item()),
                  "alpha": float(acc.sum().item()) / max(1.0, float(prop.sum().item())),
                  "temperature": T, "gemm_engine": dec.engine, "verify_ms": v_ms},
    }


def varlen_flops(s: synth.ModelShape, frames, live_rounds, H: int):
    """FLOPs of a varlen run, counted per decoder row (projections and LM head)
    and per (row, acoustic key) (cross-attention scores and mixing), plus the
    acoustic K/V projection per frame."""
    d, f, nl = s.d_model, s.d_ff, s.n_layers
    per_row = 2.0 * (nl * (6 * d * d + 2 * d * f) + s.vocab * d)
    per_row_key = 4.0 * d * nl
    per_frame = 2.0 * nl * 2 * d * d
    rows = sum(r * H for r in live_rounds)
    rowkeys = sum(r * H * F for r, F in zip(live_rounds, frames))
    return {"rows": rows * per_row, "cross_attention": rowkeys * per_row_key,
            "acoustic_kv": float(sum(frames)) * per_frame}


def run_varlen(args, rank: int, world: int, wl: Workload):
    """Varlen batch: packed (frames of each request only, finished requests
    dropped between rounds) against padded (every request carries the
    longest input, 1500 frames masked beyond its own, and stays in the batch
    until the last one ends).  Both decode the same transcripts."""
    import torch
    from speculative_whisper_asr_gb300 import runtime as R

    Fpad = 1500
    dec, req, host_enc, stream, dev = _setup(wl, rank, max_frames=Fpad)
    s, n = wl.shape, wl.n
    enc = host_enc.to(dev).view(torch.bfloat16)
    F = [int(x) for x in wl.frames]
    dec.cross_kv(req, enc, F)
    ar, syn, _, _ = _trajectory_plan(dec, req, wl, rank, dev)
    # padded encoder states: zeros beyond each request's frames
    pad = torch.zeros(n * Fpad, s.d_model, dtype=torch.bfloat16, device=dev)
    off = 0
    for i in range(n):
        pad[i * Fpad:i * Fpad + F[i]].copy_(enc[off:off + F[i]])
        off += F[i]
    live_p = []

    def packed_step():
        dec.cross_kv(req, enc, F)
        out, rounds, rows = R.run_spec_packed(dec, req, wl.budgets, synthetic=syn, live_rounds=live_p)
        return out, rounds

    def padded_step():
        dec.cross_kv(req, pad, [Fpad] * n, valid=F)
        b = dec.new_batch(req, wl.budgets)
        rounds = R.run_spec(dec, b, synthetic=syn)
        return b, rounds

    for _ in range(args.warmup):
        out_p, rounds_p = packed_step()
        b_pad, rounds_pad = padded_step()
    assert out_p == ar and b_pad.transcripts() == ar, "varlen transcripts differ from autoregressive"
    ms_p, l_p, clocks, _ = _timed(packed_step, args.steps, world, stream)
    ms_pad, l_pad, clocks_pad, _ = _timed(padded_step, args.steps, world, stream)
    tokens = int(wl.budgets.sum()) * args.steps
    H = s.K + 1
    fp = varlen_flops(s, F, live_p, H)
    fd = varlen_flops(s, [Fpad] * n, [rounds_pad] * n, H)
    frac = {k: (fd[k] - fp[k]) / fd[k] for k in fp}
    frac["total"] = (sum(fd.values()) - sum(fp.values())) / sum(fd.values())
    ms_p, ms_pad, tokens_all = reduce_over_ranks(ms_p, ms_pad, tokens, world, dev)
    return {
        "value": tokens_all / (ms_p * 1e-3), "ms_per_step": ms_p / args.steps, "launches": int(l_p),
        "roofline": None, "clocks": clocks,
        "extra": {"padded_tokens_per_s": tokens_all / (ms_pad * 1e-3), "padded_ms_per_step": ms_pad / args.steps,
                  "padded_launches": int(l_pad), "padded_clocks": clocks_pad,
                  "padded_flop_fraction": frac, "rounds_packed": rounds_p, "rounds_padded": rounds_pad,
                  "tau": float(wl.budgets.sum()) / float(sum(live_p)), "gemm_engine": dec.engine},
    }


# ---------------------------------------------------------------- profiling case
def run_profile(args):
    """Short case for kernel profilers: the workload's model and batch, its
    acoustic K/V, prefill and two warm-up rounds, then `--profile` rounds
    (or, with --profile-part cross_kv, that many acoustic K/V projections)
    inside the NVTX range "ws_timed"; --profile-part encoder runs that many
    encodes of --batch windows instead.  Rounds use random proposals (greedy
    workloads) or the drafter's samples (sampling workloads).
    --profile-layers L keeps the widths but builds L decoder layers, so a
    full-metric capture holds a few GB."""
    import dataclasses
    import torch
    from speculative_whisper_asr_gb300 import runtime as R
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    if args.profile_part == "encoder":
        # the large-v3 audio encoder over --batch windows (--profile-layers L: its first L blocks)
        e = synth.ENC_LARGE_V3
        if args.profile_layers:
            e = dataclasses.replace(e, n_layers=args.profile_layers)
        enc = R.Encoder(e, synth.encoder_weights(e, SEED), max_batch=args.batch)
        mel = enc.mel_tensor([synth.mel_input(e, SEED, i) for i in range(args.batch)])
        out = enc.encode(mel)
        enc.encode(mel, out)                  # warm-up
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("ws_timed")
        for _ in range(args.profile):
            enc.encode(mel, out)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        print(json.dumps({"profile_rounds": args.profile, "part": "encoder", "windows": args.batch,
                          "layers": e.n_layers, "status": enc.status()}))
        return
    wl = make_workload(args.workload, args.batch)
    s, n = wl.shape, wl.n
    if args.profile_layers:
        L = args.profile_layers
        s = dataclasses.replace(s, n_layers=L, hist_layers=tuple(h for h in s.hist_layers if h < L) or (0,))
    tw = synth.target_weights(s, SEED)
    dw = synth.drafter_weights(s, SEED, tw)
    F = [int(f) for f in wl.frames]
    dec = R.Decoder(s, tw, dw, max_batch=n, max_frames=max(F))
    del tw, dw
    req = dec.slots(list(range(n)))
    enc = torch.cat([dec.enc_tensor(synth.encoder_states(s, SEED, i, frames=F[i])) for i in range(n)])
    dec.cross_kv(req, enc, F)
    T, seed = wl.temperature, 7
    b = dec.new_batch(req, [BUDGET] * n, sampling=T > 0)
    syn = None
    if T <= 0:
        plan = synth.corruption_plan(n, s.max_pos, s.K, synth.corruption_p_const(s.K, 1.0), s.vocab, SEED)
        syn = (torch.zeros(n, s.max_pos, dtype=torch.int32, device="cuda"), torch.as_tensor(plan.mask, device="cuda"),
               torch.as_tensor(plan.tok, device="cuda"))
    b.prefill(temperature=T, seed=seed)
    for r in range(2):                       # warm-up rounds (graph capture)
        b.spec_step(r + 1, syn, T, seed)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("ws_timed")
    for r in range(args.profile):
        if args.profile_part == "cross_kv":
            dec.cross_kv(req, enc, F)
        else:
            b.spec_step(r + 3, syn, T, seed)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    print(json.dumps({"profile_rounds": args.profile, "part": args.profile_part, "workload": args.workload,
                      "layers": s.n_layers, "status": dec.status(), "engine": dec.engine}))


# ---------------------------------------------------------------- oracle (CPU) arm
def run_oracle_sample(budget_tokens: int = 48):
    """The oracle, as it stands, on a bounded sample of the same workload: one
    request, its own greedy trajectory (untimed, as on the GPU), then the
    timed speculative decode — acoustic K/V of all 34 layers, prompt prefill,
    rounds with proposals corrupted from that trajectory (p = 0.2) — until
    `budget_tokens` are emitted."""
    from oracle import model as M
    s = synth.LARGE_V3
    tw = synth.target_weights(s, SEED)
    dw = synth.drafter_weights(s, SEED, tw)
    orc = M.Oracle(s, tw, dw)
    del tw, dw
    A = synth.encoder_states(s, SEED, 0)
    ar = M.greedy_cached(orc, orc.new_request(A), budget_tokens)
    traj = list(s.prompt) + ar.tokens
    plan = synth.corruption_plan(1, s.max_pos, s.K, synth.corruption_p_const(s.K, P_CORRUPT), s.vocab, SEED + 100)
    t0 = time.perf_counter()
    req = orc.new_request(A)
    res = M.speculative_greedy(orc, req, budget_tokens, M.corrupted_proposer(traj, plan.mask[0], plan.tok[0]))
    dt = time.perf_counter() - t0
    assert res.tokens == ar.tokens
    cores = int(os.environ.get("OMP_NUM_THREADS", os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1)))
    return len(res.tokens), dt, cores


def encoder_flops(e: synth.EncoderShape) -> float:
    """Algorithmic FLOPs of one window: both convolutions (3 taps), and per
    block the q/k/v, output and FFN projections plus S = QK^T and PV."""
    F, d, f = e.n_frames, e.d_model, e.d_ff
    stem = 2.0 * (2 * F) * (3 * e.n_mels) * d + 2.0 * F * (3 * d) * d
    block = 2.0 * F * (3 * d * d + d * d + 2 * d * f) + 4.0 * F * F * d
    return stem + e.n_layers * block


def run_encoder(args, n: int) -> dict:
    """The large-v3 audio encoder over n 30 s windows (the step before the
    decoding path): windows/s, and the whole encoder's tensor throughput
    against the sustained bf16 peak."""
    import torch
    from speculative_whisper_asr_gb300 import runtime as R
    e = synth.ENC_LARGE_V3
    enc = R.Encoder(e, synth.encoder_weights(e, SEED), max_batch=n)
    mel = enc.mel_tensor([synth.mel_input(e, SEED, i) for i in range(n)])
    out = torch.empty(n, e.n_frames, e.d_model, dtype=torch.bfloat16, device=enc.dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        enc.encode(mel, out)
    steps = max(1, args.steps)
    ms, launches, clocks, _ = _timed(lambda: enc.encode(mel, out), steps, 1, stream)
    assert enc.status() == 0
    ms_step = ms / steps
    _, _, src = peaks()
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
        sus = float(json.load(fh).get("bf16_tflops_sustained", 1700.0)) if src == "measured" else 1700.0
    tf = encoder_flops(e) * n / (ms_step * 1e-3) / 1e12
    del enc
    torch.cuda.empty_cache()
    return {"config": {"workload": f"large-v3-encoder-b{n}", "windows": n, "frames": e.n_frames,
                       "mel_frames": 2 * e.n_frames, "layers": e.n_layers, "d_model": e.d_model,
                       "weights_larger_than_l2": True},
            "value": n * steps / (ms * 1e-3), "unit": "windows/s", "audio_s_per_s": 30.0 * n * steps / (ms * 1e-3),
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms_step, "ms_per_window": ms_step / n,
            "gpu_launches": launches // steps,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": sus, "unit": "TFLOP/s", "frac": tf / sus,
                         "peak_kind": f"{src} sustained bf16 (whole encoder, all kernels)", "traffic": None},
            "clocks": clocks}


def run_workload(args, rank: int, world: int, wl: Workload):
    import torch
    if wl.temperature > 0.0:
        r = run_sampling(args, rank, world, wl)
    elif wl.name == "turbo-b64-varlen":
        r = run_varlen(args, rank, world, wl)
    else:
        r = run_gpu(args, rank, world, wl)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()            # the next workload's context gets the memory back
    return r


def sub_summary(wl: Workload, args, r: dict) -> dict:
    """One workload of the metric, as a sub-object of the headline line."""
    out = {"config": wl.config(), "value": r["value"], "unit": "tokens/s", "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "gpu_launches": r["launches"],
           "roofline": r["roofline"], "clocks": r["clocks"], "extra": r["extra"]}
    if "e2e" in r:
        out["e2e"] = {"value": r["e2e"], "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                      "d2h_bytes_per_step": r["d2h"]}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="headline workload only (no batch 16 / 96 sub-objects)")
    ap.add_argument("--profile", type=int, default=0, help="run N rounds of the profiling case and exit")
    ap.add_argument("--profile-part", default="round", choices=["round", "cross_kv", "encoder"])
    ap.add_argument("--profile-layers", type=int, default=0, help="profiling case with fewer decoder layers")
    ap.add_argument("--workload", default="large-v3-b1", choices=WORKLOADS,
                    help="large-v3-b1 is the headline; the others measure the batch 16 / 96 and varlen cases")
    args = ap.parse_args()
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))

    if args.profile > 0:
        run_profile(args)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        vals = []
        run_oracle_sample(2)   # one short warm-up (imports, BLAS threads)
        total_tok, total_t, cores = 0, 0.0, 1
        for _ in range(args.steps):
            tok, dt, cores = run_oracle_sample()
            total_tok += tok
            total_t += dt
            vals.append(tok / dt)
        v = total_tok / total_t
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 0,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload(1),
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": "1 request of the same workload: acoustic K/V of 34 layers + prefill + "
                                           f"speculative rounds until {total_tok // max(1, args.steps)} tokens "
                                           "(numpy float64 oracle)"},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    wl = make_workload(args.workload, args.batch)
    r = run_workload(args, rank, world, wl)
    subs = {}
    if args.workload == "large-v3-b1" and args.batch == 1 and not args.no_sub:
        # the batch-96 and batch-16 workloads of the same metric, fewer timed steps
        sub = argparse.Namespace(**vars(args))
        sub.steps, sub.warmup = min(args.steps, 4), 3
        for name in ("large-v3-b96-t0.7", "turbo-b16"):
            w2 = make_workload(name)
            r2 = run_workload(sub, rank, world, w2)
            subs[name] = sub_summary(w2, sub, r2)
        if rank == 0:
            # the audio encoder before the path, at batch 1 and 16, and its share of request time
            e1 = run_encoder(sub, 1)
            e16 = run_encoder(sub, 16)
            e1["encoder_share_b1"] = e1["ms_per_window"] / (e1["ms_per_window"] + r["ms_per_step"] / wl.n)
            if "turbo-b16" in subs:
                e16["encoder_share_turbo_b16"] = e16["ms_per_step"] / (e16["ms_per_step"] +
                                                                       subs["turbo-b16"]["ms_per_step"])
            subs["large-v3-encoder-b1"] = e1
            subs["large-v3-encoder-b16"] = e16
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "large-v3-b1":
        tok, dt, cores = run_oracle_sample()
        cpu = {"value": tok / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"1 request of the same workload: acoustic K/V (34 layers) + prefill + speculative "
                         f"rounds until {tok} tokens, numpy float64 oracle, {dt:.1f} s"}
    if rank == 0:
        e2e = None
        if "e2e" in r:
            e2e = {"value": r["e2e"], "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                   "d2h_bytes_per_step": r["d2h"]}
        line = {"metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": dict(wl.config(), parallelism=f"replicas x{world}"),
                "e2e": e2e, "gpu_launches": r["launches"], "roofline": r["roofline"], "cpu_baseline": cpu,
                "clocks": r["clocks"], "extra": r["extra"]}
        if subs:
            line["workloads"] = subs
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
