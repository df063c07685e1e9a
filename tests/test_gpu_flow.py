"""GPU tests of the dataflow block verification (one-request bf16 contexts:
the whole target pass in one cooperative kernel whose tasks wait on
per-step counters).  Its rows must agree with the oracle within the bf16
tolerance and with the kernel-per-operation path on the same cache state,
speculative decoding through it must equal autoregressive decoding bit for
bit, and it must replay identically from a captured CUDA graph."""
import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from gpu_common import (ar_from, dev_i32, greedy_near_tie_bf16, logits_close, small_shape,
                        tokens_match_resuming)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def RB():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding, runtime
    return runtime, binding


def _verify(dec, req, block, H):
    n = req.numel()
    tgt = torch.zeros(n, H, dtype=torch.int32, device="cuda")
    lg = torch.empty(n, H, dec.V, device="cuda")
    dec.verify(req, dev_i32(block), dev_i32([H] * n), tgt, lg)
    torch.cuda.synchronize()
    return lg, tgt


@pytest.mark.parametrize("wide", [False, True])
def test_flow_block_vs_oracle_and_per_op(RB, wide):
    """After 12 greedy tokens, one block of 9 (and of 16) random tokens:
    the dataflow kernel's logits equal the oracle's plain forward over
    prompt + transcript + block within 2e-2, the per-op path's within the
    same bound, and its argmax ids are the argmax of its own logits.  d 256
    (one k-block per warp quarter, FC2 in 2 slices, 300 frames = 2 chunk
    groups) and d 1280 (five k-blocks, FC2 in 4 slices, 1500 frames)."""
    R, B = RB
    kw = dict(n_layers=2, d_model=1280, n_heads=20, d_ff=5120) if wide else {}
    s = small_shape("bf16", **kw)
    F = 1500 if wide else 300
    tw = synth.target_weights(s, 41)
    A = synth.encoder_states(s, 41, 0, frames=F)
    dec = R.Decoder(s, tw, None, max_batch=1, max_frames=F, max_block=16)
    assert dec.engine == "tcgen05"
    assert B.ws_fused_verify(dec.ctx, 1) == 1            # eligible
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [F])
    b = dec.new_batch(req, [12])
    R.run_ar(dec, b)                                      # cache holds prompt + 12 tokens
    tr = b.transcripts()[0]
    orc = M.Oracle(s, tw, None)
    rng = np.random.default_rng(5)
    for H in (9, 16):
        block = rng.integers(0, s.vocab, size=(1, H)).tolist()
        lf, tf = _verify(dec, req, block, H)
        seq = list(s.prompt) + tr[:-1] + block[0]
        ora, _ = orc.forward_full(orc.new_request(A), seq)
        logits_close(lf[0].cpu().numpy(), ora[-H:], 2e-2)
        assert tf[0].tolist() == lf[0].argmax(dim=1).tolist()
        assert B.ws_fused_verify(dec.ctx, 0) == 0
        lp, tp = _verify(dec, req, block, H)
        assert B.ws_fused_verify(dec.ctx, 1) == 1
        logits_close(lf[0].cpu().numpy(), lp[0].cpu().numpy().astype(np.float64), 2e-2)
    assert dec.status() == 0


def test_flow_speculative_equals_autoregressive_and_oracle(RB):
    """Drafter-driven speculative decoding through the dataflow verify gives
    the autoregressive transcript bit for bit (the reduction order of every
    row is the same for 1-row and 9-row blocks), and that transcript equals
    the oracle's greedy one (restarting at bf16 near ties)."""
    R, B = RB
    s = small_shape("bf16")
    tw = synth.target_weights(s, 44)
    dw = synth.drafter_weights(s, 44, tw)
    A = synth.encoder_states(s, 44, 0, frames=257)
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=257)
    assert B.ws_fused_verify(dec.ctx, 1) == 1
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [257])
    b = dec.new_batch(req, [40])
    R.run_ar(dec, b)
    ar = b.transcripts()[0]
    b2 = dec.new_batch(req, [40])
    R.run_spec(dec, b2)
    assert b2.transcripts()[0] == ar
    orc = M.Oracle(s, tw, None)
    ref = M.greedy_cached(orc, orc.new_request(A), 40)
    n, _ = tokens_match_resuming(ar_from(R, dec, req, s, 40), ref.tokens, ref.margins, greedy_near_tie_bf16,
                                 first=ar)
    assert n == 40
    assert dec.status() == 0


def test_flow_graph_capture_replays_identically(RB):
    R, B = RB
    s = small_shape("bf16", n_layers=2)
    tw = synth.target_weights(s, 43)
    A = synth.encoder_states(s, 43, 0, frames=200)
    dec = R.Decoder(s, tw, None, max_batch=1, max_frames=200)
    assert B.ws_fused_verify(dec.ctx, 1) == 1
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [200])
    dec.reset(req)
    H = len(s.prompt)
    blk, bl = dev_i32([s.prompt]), dev_i32([H])
    t1 = torch.zeros(1, H, dtype=torch.int32, device="cuda")
    l1 = torch.empty(1, H, s.vocab, device="cuda")
    dec.verify(req, blk, bl, t1, l1)
    t2 = torch.zeros_like(t1)
    l2 = torch.full_like(l1, float("nan"))
    stream = torch.cuda.current_stream().cuda_stream
    B.ws_capture_begin(dec.ctx, stream)
    dec.verify(req, blk, bl, t2, l2)
    g = B.ws_capture_end(dec.ctx, stream)
    for _ in range(3):
        B.ws_graph_launch(g, stream)
    torch.cuda.synchronize()
    B.ws_graph_free(g)
    assert torch.equal(l1, l2)
    assert torch.equal(t1, t2)
    assert dec.status() == 0


@pytest.mark.parametrize("wide", [False, True])
def test_layernorm_in_gemm_bit_identical(RB, wide):
    """Layer norm computed inside the projection GEMMs gives the same logits,
    bit for bit, as the layer-norm kernel path: d 256 (two 128-feature groups
    per lane row) and d 1280 (ten, the widest Whisper decoder), with 16 rows
    (four rows per warp) and with 5 rows (ragged: warps with one and two rows)."""
    R, B = RB
    kw = dict(n_layers=2, d_model=1280, n_heads=20, d_ff=5120) if wide else {}
    s = small_shape("bf16", **kw)
    tw = synth.target_weights(s, 47)
    A = synth.encoder_states(s, 47, 0, frames=200)
    dec = R.Decoder(s, tw, None, max_batch=1, max_frames=200, max_block=16)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [200])
    dec.reset(req)
    B.ws_fused_verify(dec.ctx, 0)                         # the kernel-per-operation path
    assert B.ws_fused_layernorm(dec.ctx, -1) == 1
    rng = np.random.default_rng(11)
    for H in (16, 5):
        block = [list(s.prompt) + rng.integers(0, s.vocab, size=H - len(s.prompt)).tolist()]
        lf, tf = _verify(dec, req, block, H)
        assert B.ws_fused_layernorm(dec.ctx, 0) == 0
        lp, tp = _verify(dec, req, block, H)
        assert B.ws_fused_layernorm(dec.ctx, 1) == 1
        assert torch.equal(lf, lp)
        assert torch.equal(tf, tp)
        orc = M.Oracle(s, tw, None)
        ora, _ = orc.forward_full(orc.new_request(A), block[0])
        logits_close(lf[0].cpu().numpy(), ora, 2e-2)
    assert dec.status() == 0
