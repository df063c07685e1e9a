"""GPU tests of the tcgen05 GEMM engine (bf16) and of the full-size
Whisper-large-v3-shaped workload at batch 1 (32 layers, d 1280, 20 heads,
FFN 5120, V 51866, 1500 frames, 224 tokens, K = 8, synthetic drafts p = 0.2)."""
import numpy as np
import pytest
import torch

import synth
from oracle import model as M
from gpu_common import (MARGIN_BF16, ar_from, dev_i32, greedy_near_tie_bf16, logits_close, small_shape,
                        teacher_forced_logits, tokens_match_resuming)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding, runtime
    return runtime


def _prefill_logits(dec, req, s, n):
    dec.reset(req)
    tgt = torch.zeros(n, len(s.prompt), dtype=torch.int32, device="cuda")
    lg = torch.empty(n, len(s.prompt), s.vocab, device="cuda")
    dec.verify(req, dev_i32([s.prompt] * n), dev_i32([len(s.prompt)] * n), tgt, lg)
    return lg, tgt


def test_tc_engine_matches_simt_and_oracle(R):
    import speculative_whisper_asr_gb300.binding as B
    s = small_shape("bf16")
    tw = synth.target_weights(s, 31)
    dw = synth.drafter_weights(s, 31, tw)
    frames = [300, 129]
    As = [synth.encoder_states(s, 31, i, frames=f) for i, f in enumerate(frames)]
    orc = M.Oracle(s, tw, dw)
    outs, decs = {}, {}
    for eng in (B.WS_GEMM_TC, B.WS_GEMM_SIMT):
        dec = decs[eng] = R.Decoder(s, tw, dw, max_batch=2, max_frames=300, gemm=eng)
        assert dec.engine == ("tcgen05" if eng == B.WS_GEMM_TC else "simt")
        req = dec.slots([0, 1])
        dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in As]), frames)
        lg, _ = _prefill_logits(dec, req, s, 2)
        for i in range(2):
            logits_close(lg[i].cpu().numpy(), orc.verify(orc.new_request(As[i]), list(s.prompt)), 2e-2)
        b = dec.new_batch(req, [30, 25])
        R.run_ar(dec, b)
        b2 = dec.new_batch(req, [30, 25])
        R.run_spec(dec, b2)
        assert b2.transcripts() == b.transcripts()
        outs[eng] = (lg.cpu().numpy(), b.transcripts())
        assert dec.status() == 0
    a, b_ = outs[B.WS_GEMM_TC][0], outs[B.WS_GEMM_SIMT][0]
    assert np.abs(a - b_).max() < 2e-2 * max(1.0, np.abs(b_).max())
    for i in range(2):
        budget = [30, 25][i]
        ref = M.greedy_cached(orc, orc.new_request(As[i]), budget)
        run = ar_from(R, decs[B.WS_GEMM_TC], decs[B.WS_GEMM_TC].slots([i]), s, budget)
        n, _ = tokens_match_resuming(run, ref.tokens, ref.margins, greedy_near_tie_bf16,
                                     first=outs[B.WS_GEMM_TC][1][i])
        assert n == budget


def test_tc_rows_do_not_depend_on_token_tile(R):
    """A row's logits are bit-identical whether its GEMMs ran with 16-token or
    256-token MMA tiles (the property block verification relies on)."""
    s = small_shape("bf16", n_layers=2)
    tw = synth.target_weights(s, 32)
    A = synth.encoder_states(s, 32, 0, frames=64)
    dec = R.Decoder(s, tw, None, max_batch=48, max_frames=64)
    req1 = dec.slots([0])
    dec.cross_kv(req1, dec.enc_tensor(A), [64])
    lg1, _ = _prefill_logits(dec, req1, s, 1)
    reqn = dec.slots(list(range(48)))
    dec.cross_kv(reqn, torch.cat([dec.enc_tensor(A)] * 48), [64] * 48)
    lgn, _ = _prefill_logits(dec, reqn, s, 48)            # 192 rows -> 256-token tiles
    assert torch.equal(lg1[0], lgn[0])
    assert torch.equal(lgn[0], lgn[47])


@pytest.fixture(scope="module")
def large(R):
    s = synth.LARGE_V3
    tw = synth.target_weights(s, 1)
    dw = synth.drafter_weights(s, 1, tw)
    A = synth.encoder_states(s, 1, 0)
    dec = R.Decoder(s, tw, dw, max_batch=1, max_frames=1500)
    req = dec.slots([0])
    dec.cross_kv(req, dec.enc_tensor(A), [1500])
    return s, tw, dw, A, dec, req


@pytest.fixture(scope="module")
def large_ref(large):
    """The oracle's greedy transcript of the benchmark request (224 tokens,
    bf16 storage points) with its top-2 margins, and its logits at every
    position of prompt + transcript."""
    s, tw, dw, A, dec, req = large
    orc = M.Oracle(s, tw, None)
    ref = M.greedy_cached(orc, orc.new_request(A), 224)
    ora, _ = orc.forward_full(orc.new_request(A), list(s.prompt) + ref.tokens[:-1])
    return ref, ora


def test_large_v3_batch1_prefill_and_first_tokens_vs_oracle(R, large, large_ref):
    """Prompt logits, then the whole 224-token greedy transcript against the
    oracle's, restarting from the oracle's token at bf16 near ties."""
    s, tw, dw, A, dec, req = large
    ref, ora = large_ref
    assert dec.engine == "tcgen05"
    lg, tgt = _prefill_logits(dec, req, s, 1)
    logits_close(lg[0].cpu().numpy(), ora[:len(s.prompt)], 2e-2)
    n, resumes = tokens_match_resuming(ar_from(R, dec, req, s, 224), ref.tokens, ref.margins,
                                       greedy_near_tie_bf16)
    assert n == 224 and len(ref.tokens) == 224
    assert dec.status() == 0


def test_large_v3_teacher_forced_margin_error(R, large, large_ref):
    """Fed the oracle's own greedy tokens, the logits of all 227 rows (the
    prompt and 223 forced tokens; 224 of them predict a transcript token)
    stay within 2e-2 of the oracle's, the
    difference between the oracle's top-2 logits moves by less than 2e-2 (the stated bf16 logit precision) at
    every position (the bound behind the bf16 near-tie rule), and the GPU's
    argmax equals the oracle's wherever the oracle's margin is at least 2e-2."""
    s, tw, dw, A, dec, req = large
    ref, ora = large_ref
    toks = ref.tokens[:-1]
    gpu = teacher_forced_logits(dec, req, s, toks)
    assert gpu.shape == ora.shape == (len(s.prompt) + 223, s.vocab)
    logits_close(gpu, ora, 2e-2)
    checked = 0
    for r in range(len(s.prompt) - 1, ora.shape[0]):
        top = np.argsort(-ora[r])[:2]
        d_ora = ora[r][top[0]] - ora[r][top[1]]
        d_gpu = gpu[r][top[0]] - gpu[r][top[1]]
        assert abs(d_gpu - d_ora) < MARGIN_BF16, (r, d_ora, d_gpu)
        if d_ora >= MARGIN_BF16:
            assert int(np.argmax(gpu[r])) == int(top[0]), r
            checked += 1
    assert checked > 0.9 * 224
    assert dec.status() == 0


def test_large_v3_batch1_speculative_bit_identical_224(R, large):
    """The benchmark workload: 224 tokens, synthetic drafts (p = 0.2) with the
    drafter also run; speculative output equals autoregressive output."""
    s, tw, dw, A, dec, req = large
    import speculative_whisper_asr_gb300.binding as B
    b = dec.new_batch(req, [224])
    R.run_ar(dec, b)
    ar = b.transcripts()[0]
    assert len(ar) == 224
    traj = np.zeros((1, s.max_pos), dtype=np.int32)
    t = list(s.prompt) + ar
    traj[0, :len(t)] = t
    plan = synth.corruption_plan(1, s.max_pos, s.K, synth.corruption_p_const(s.K, 0.2), s.vocab, 101)
    syn = (torch.as_tensor(traj, device="cuda"), torch.as_tensor(plan.mask, device="cuda"),
           torch.as_tensor(plan.tok, device="cuda"))
    b2 = dec.new_batch(req, [224])
    rounds = R.run_spec(dec, b2, synthetic=syn)
    assert b2.transcripts()[0] == ar
    # E[a] = sum_k 0.8^k = 3.33 for full rounds: about 224 / 4.33 = 52 rounds
    assert 35 <= rounds <= 75, rounds
    assert dec.status() == 0
