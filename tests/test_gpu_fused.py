"""GPU tests of the persistent block-verification kernel (bf16, tcgen05,
at most 16 rows per call): it must give the same rows, bit for bit, as the
kernel-per-operation path on the same context state, agree with the oracle
within the bf16 tolerance, and survive CUDA-graph capture."""
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


def _verify(dec, req, block, H):
    n = req.numel()
    tgt = torch.zeros(n, H, dtype=torch.int32, device="cuda")
    lg = torch.empty(n, H, dec.V, device="cuda")
    dec.verify(req, dev_i32(block), dev_i32([H] * n), tgt, lg)
    torch.cuda.synchronize()
    return lg, tgt


def _both_paths(B, dec, req, block, H):
    """The same verify (same cache state: it rewrites the block's own K/V
    rows) through the persistent kernel and through the per-op path."""
    assert B.ws_fused_verify(dec.ctx, 1) == 1
    lf, tf = _verify(dec, req, block, H)
    assert B.ws_fused_verify(dec.ctx, 0) == 0
    lp, tp = _verify(dec, req, block, H)
    assert B.ws_fused_verify(dec.ctx, 1) == 1
    return (lf, tf), (lp, tp)


@pytest.mark.parametrize("max_batch", [1, 2])
def test_fused_bit_identical_to_per_op_with_split_k(RB, max_batch):
    """Small bf16 model (3 layers, d 256, ragged vocab 1000): contexts of at
    most 64 rows split K, so this covers the split-K fold of the persistent
    kernel; then one request with a 9-row block and two requests with 8 rows
    each (16 rows, the largest persistent call)."""
    R, B = RB
    s = small_shape("bf16")
    tw = synth.target_weights(s, 41)
    dw = synth.drafter_weights(s, 41, tw)
    frames = [300, 171][:max_batch]
    As = [synth.encoder_states(s, 41, i, frames=f) for i, f in enumerate(frames)]
    dec = R.Decoder(s, tw, dw, max_batch=max_batch, max_frames=300)
    assert dec.engine == "tcgen05"
    req = dec.slots(list(range(max_batch)))
    dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in As]), frames)
    b = dec.new_batch(req, [12] * max_batch)
    R.run_ar(dec, b)                                  # cache holds prompt + 12 tokens
    rng = np.random.default_rng(5)
    H = 9 if max_batch == 1 else 8
    block = rng.integers(0, s.vocab, size=(max_batch, H)).tolist()
    (lf, tf), (lp, tp) = _both_paths(B, dec, req, block, H)
    assert torch.equal(lf, lp)
    assert torch.equal(tf, tp)
    # and against the plain definition: the cache holds the prompt and every
    # emitted token but the last (the next anchor), the block follows it
    orc = M.Oracle(s, tw, None)
    tr = b.transcripts()
    for i in range(max_batch):
        seq = list(s.prompt) + tr[i][:-1] + block[i]
        ora, _ = orc.forward_full(orc.new_request(As[i]), seq)
        logits_close(lf[i].cpu().numpy(), ora[-H:], 2e-2)
    assert dec.status() == 0


def test_fused_graph_capture_replays_identically(RB):
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
