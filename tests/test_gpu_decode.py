"""GPU parity: the CUDA decoding path against the CPU oracle (tiny fp32
model and small multi-request shapes in fp32 and bf16), plus the exactness
property of the method: speculative greedy output is bit-identical to
autoregressive greedy output through the same kernels (Whisper-Flash §3.1,
Appendix A.5)."""
import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from gpu_common import (MARGIN, ar_from, dev_i32, logits_close, near_tie_for, small_shape,
                        tokens_match_resuming)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import runtime
    return runtime


# ---------------------------------------------------------------- tiny fp32 model (64 tokens)

@pytest.fixture(scope="module")
def tiny(R):
    s = synth.TINY
    tw = synth.target_weights(s, 0)
    dw = synth.drafter_weights(s, 0, tw)
    A = synth.encoder_states(s, 0, 0)
    orc = M.Oracle(s, tw, dw)
    dec = R.Decoder(s, tw, dw, max_batch=2, max_frames=1500)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    ref = M.greedy_cached(orc, orc.new_request(A), 64)
    return s, A, orc, dec, req, ref


def test_tiny_prefill_logits(tiny):
    s, A, orc, dec, req, _ = tiny
    dec.reset(req)
    blk = dev_i32([s.prompt])
    tgt = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    lg = torch.empty(1, 4, s.vocab, device="cuda")
    dec.verify(req, blk, dev_i32([4]), tgt, lg)
    ora = orc.verify(orc.new_request(A), list(s.prompt))
    logits_close(lg[0].cpu().numpy(), ora, 1e-4)
    assert tgt[0].tolist() == [int(np.argmax(z)) for z in ora]
    assert dec.status() == 0


def test_tiny_autoregressive_matches_oracle(R, tiny):
    s, A, orc, dec, req, ref = tiny
    b = dec.new_batch(req, [64])
    R.run_ar(dec, b)
    got = b.transcripts()[0]
    assert len(got) == 64
    n, _ = tokens_match_resuming(ar_from(R, dec, req, s, 64), ref.tokens, ref.margins, first=got)
    assert n == 64


def test_tiny_speculative_equals_autoregressive(R, tiny):
    s, A, orc, dec, req, ref = tiny
    b = dec.new_batch(req, [64])
    R.run_ar(dec, b)
    ar = b.transcripts()[0]
    b2 = dec.new_batch(req, [64])
    rounds = R.run_spec(dec, b2)
    sp = b2.transcripts()[0]
    assert sp == ar                    # bit-identical through the same kernels
    assert rounds <= 63
    assert dec.status() == 0


def test_tiny_teacher_forced_verify_all_positions(tiny):
    """Blocks of K+1 oracle tokens verified on the GPU: every row's logits
    match the oracle's cached verify of the same block."""
    s, A, orc, dec, req, ref = tiny
    import speculative_whisper_asr_gb300.binding as B
    seq = list(s.prompt) + ref.tokens
    dec.reset(req)
    r = orc.new_request(A)
    pos, H = 0, s.K + 1
    b = dec.new_batch(req, [10 ** 6])
    while pos < len(seq):
        blk = seq[pos:pos + H]
        h = len(blk)
        bt = dev_i32([blk + [0] * (H - h)])
        tgt = torch.zeros(1, H, dtype=torch.int32, device="cuda")
        lg = torch.empty(1, H, s.vocab, device="cuda")
        bl = dev_i32([h])
        dec.verify(req, bt, bl, tgt, lg)
        a = b._args(B.WS_ACCEPT_FORCED, H, bt, bl, tgt, b.block, b.blen)
        B.ws_accept(dec.ctx, 1, req.data_ptr(), a, torch.cuda.current_stream().cuda_stream)
        ora = orc.verify(r, blk)
        r.L += h
        logits_close(lg[0, :h].cpu().numpy(), ora, 1e-4)
        pos += h
    assert list(dec.lengths(req)) == [len(seq)]


def test_tiny_drafter_logits_and_history(R, tiny):
    """Drafter logits after the prompt, and again after one verified round
    whose accepted rows were folded into the history."""
    s, A, orc, dec, req, ref = tiny
    import speculative_whisper_asr_gb300.binding as B
    b = dec.new_batch(req, [64], sampling=True)
    b.prefill()
    r = orc.new_request(A)
    M.prefill(orc, r, 64)
    anchor = ref.tokens[0]
    assert b.block[0, 0].item() == anchor
    dec.draft(req, b.block, 1.0, 3, 1, b.q_logits)
    logits_close(b.q_logits[0].cpu().numpy(), orc.draft_logits(r, anchor), 1e-4)
    # one round: candidates = the next 3 reference tokens then junk, greedy accept
    cand = ref.tokens[1:4] + [7] * (s.K - 3)
    b.block[0, 1:] = dev_i32(cand)
    b.blen[0] = s.K + 1
    dec.verify(req, b.block, b.blen, b.target)
    a = b._args(B.WS_ACCEPT_GREEDY, s.K + 1, b.block, b.blen, b.target, b.block, b.blen)
    B.ws_accept(dec.ctx, 1, req.data_ptr(), a, torch.cuda.current_stream().cuda_stream)
    assert b.n_acc[0].item() == 3
    lg = orc.verify(r, [anchor] + cand)
    r.L += 4
    anchor2 = int(np.argmax(lg[3]))
    assert b.block[0, 0].item() == anchor2
    dec.draft(req, b.block, 1.0, 3, 2, b.q_logits)
    logits_close(b.q_logits[0].cpu().numpy(), orc.draft_logits(r, anchor2), 1e-4)
    # greedy proposals are the argmax of the same logits
    q = b.q_logits[0].cpu().numpy()
    dec.draft(req, b.block, 0.0, 0, 3, None)
    assert b.block[0, 1:].tolist() == [int(np.argmax(z)) for z in q]


# ---------------------------------------------------------------- ragged multi-request batches

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_batch_varlen(R, dtype):
    s = small_shape(dtype)
    tw = synth.target_weights(s, 21)
    dw = synth.drafter_weights(s, 21, tw)
    frames, budgets = [200, 77, 129], [20, 7, 33]
    As = [synth.encoder_states(s, 21, i, frames=f) for i, f in enumerate(frames)]
    orc = M.Oracle(s, tw, dw)
    dec = R.Decoder(s, tw, dw, max_batch=5, max_frames=256)
    req = dec.slots([3, 0, 4])                        # non-contiguous slots
    dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in As]), frames)
    b = dec.new_batch(req, budgets)
    R.run_ar(dec, b)
    ar = b.transcripts()
    b2 = dec.new_batch(req, budgets)
    R.run_spec(dec, b2)
    assert b2.transcripts() == ar
    for i in range(3):
        ref = M.greedy_cached(orc, orc.new_request(As[i]), budgets[i])
        one = dec.slots([[3, 0, 4][i]])
        n, _ = tokens_match_resuming(ar_from(R, dec, one, s, budgets[i]), ref.tokens, ref.margins,
                                     near_tie_for(dtype), first=ar[i])
        assert n == budgets[i]
    # prefill logits of every request
    dec.reset(req)
    blk = dev_i32([s.prompt] * 3)
    tgt = torch.zeros(3, 4, dtype=torch.int32, device="cuda")
    lg = torch.empty(3, 4, s.vocab, device="cuda")
    dec.verify(req, blk, dev_i32([4, 4, 4]), tgt, lg)
    tol = 1e-4 if dtype == "f32" else 2e-2
    for i in range(3):
        logits_close(lg[i].cpu().numpy(), orc.verify(orc.new_request(As[i]), list(s.prompt)), tol)
    assert dec.status() == 0


def test_small_frames_beyond_valid_are_masked(R):
    s = small_shape("f32")
    tw = synth.target_weights(s, 22)
    A = synth.encoder_states(s, 22, 0, frames=160)
    A2 = A.copy()
    A2[100:] = 50.0
    dec = R.Decoder(s, tw, None, max_batch=2, max_frames=160)
    req = dec.slots([0, 1])
    dec.cross_kv(req, torch.cat([dec.enc_tensor(A), dec.enc_tensor(A2)]), [160, 160], valid=[100, 100])
    dec.reset(req)
    tgt = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    lg = torch.empty(2, 4, s.vocab, device="cuda")
    dec.verify(req, dev_i32([s.prompt] * 2), dev_i32([4, 4]), tgt, lg)
    assert torch.equal(lg[0], lg[1])
    orc = M.Oracle(s, tw, None)
    logits_close(lg[0].cpu().numpy(), orc.verify(orc.new_request(A, frames=100), list(s.prompt)), 1e-4)
