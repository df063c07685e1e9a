"""Pins for the CPU oracle, independent of the oracle itself.

Each test checks the oracle against something the pages or mathematics fix:
published known-answer vectors, printed numbers, library routines that the
definition reduces to (torch's TransformerDecoderLayer / layer_norm / gelu /
scaled_dot_product_attention / bf16 cast, all in float64), closed forms and
exact invariants of the method (speculative greedy == autoregressive greedy).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import model as M
from oracle import philox

GOLD = os.path.join(os.path.dirname(__file__), "golden")

# A small shape that keeps the oracle fast while exercising every code path.
SMALL = synth.ModelShape("small", 3, 128, 2, 512, vocab=1000, max_pos=96,
                         hist_layers=(0, 2), dtype="f32")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def small():
    tw = synth.target_weights(SMALL, 11)
    dw = synth.drafter_weights(SMALL, 11, tw)
    orc = M.Oracle(SMALL, tw, dw)
    A = synth.encoder_states(SMALL, 11, 0, frames=60)
    return orc, tw, dw, A


# ---------------------------------------------------------------- Philox

def test_philox_known_answers():
    for v in _load("philox4x32_10_kat.json")["vectors"]:
        ctr = [int(x, 16) for x in v["ctr"]]
        key = [int(x, 16) for x in v["key"]]
        out = philox.philox4x32_10(ctr, key)
        assert ["%08x" % w for w in out] == v["out"]


def test_philox_uniform_range_and_mean():
    u = np.array([philox.uniform(7, s, r, j, 1) for s in range(4) for r in range(50) for j in range(10)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 4 * math.sqrt(1 / 12 / u.size)


# ---------------------------------------------------------------- numerics

def test_round_bf16_matches_torch_cast():
    x = np.random.default_rng(0).standard_normal(10000) * 3
    x = np.concatenate([x, [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 1e-30]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(M.round_bf16(x), ref)


def test_layer_norm_and_gelu_match_torch():
    g = np.random.default_rng(1)
    x = g.standard_normal((7, 96))
    w, b = g.standard_normal(96), g.standard_normal(96)
    ref = F.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), torch.from_numpy(b), eps=1e-5)
    np.testing.assert_allclose(M.layer_norm(x, w, b), ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(M.gelu(x), F.gelu(torch.from_numpy(x)).numpy(), rtol=0, atol=1e-14)


def test_mha_matches_sdpa_and_softmax_sums_to_one():
    g = np.random.default_rng(2)
    q, k, v = g.standard_normal((5, 128)), g.standard_normal((9, 128)), g.standard_normal((9, 128))
    mask = np.tril(np.ones((5, 9), dtype=bool), k=4)
    o = M.mha(q, k, v, 2, mask)
    th = lambda a: torch.from_numpy(a).reshape(a.shape[0], 2, 64).transpose(0, 1)
    ref = F.scaled_dot_product_attention(th(q), th(k), th(v), attn_mask=torch.from_numpy(mask))
    np.testing.assert_allclose(o, ref.transpose(0, 1).reshape(5, 128).numpy(), atol=1e-12)
    p = M.softmax(g.standard_normal((4, 1000)) * 10)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)


def test_rope_closed_form_and_relative_position():
    dh, H = 64, 2
    th = M.rope_theta(dh)
    # theta_i = 10000^(-2i/64): theta_0 = 1, theta_16 = 10000^-0.5 = 0.01
    assert th[0] == np.float32(1.0) and abs(th[16] - 0.01) < 1e-9
    for p in (0, 1, 7, 300):
        for i in (0, 5, 31):
            e = np.zeros((1, H * dh))
            e[0, 2 * i] = 1.0
            r = M.rope(e, np.array([p]), H)
            ang = float(np.float32(np.float32(p) * th[i]))
            expect = np.zeros(H * dh)
            expect[2 * i], expect[2 * i + 1] = math.cos(ang), math.sin(ang)
            np.testing.assert_allclose(r[0], expect, atol=1e-15)
    g = np.random.default_rng(3)
    q, k = g.standard_normal((1, H * dh)), g.standard_normal((1, H * dh))
    d1 = (M.rope(q, [40], H) * M.rope(k, [13], H)).sum()
    d2 = (M.rope(q, [140], H) * M.rope(k, [113], H)).sum()
    assert abs(d1 - d2) < 1e-4 * (abs(d1) + 1)
    np.testing.assert_allclose(np.linalg.norm(M.rope(q, [77], H)), np.linalg.norm(q), rtol=1e-12)


# ---------------------------------------------------------------- target decoder

def _torch_decoder(shape, tw, l):
    d, f = shape.d_model, shape.d_ff
    lay = torch.nn.TransformerDecoderLayer(d, shape.n_heads, f, dropout=0.0, activation="gelu",
                                           batch_first=True, norm_first=True, dtype=torch.float64)
    T = lambda n: torch.from_numpy(np.asarray(tw[f"layers.{l}.{n}"], dtype=np.float64))
    z = torch.zeros(d, dtype=torch.float64)
    with torch.no_grad():
        lay.self_attn.in_proj_weight.copy_(T("w_qkv"))
        lay.self_attn.in_proj_bias.copy_(torch.cat([T("b_q"), z, T("b_v")]))
        lay.self_attn.out_proj.weight.copy_(T("w_o"))
        lay.self_attn.out_proj.bias.copy_(T("b_o"))
        lay.multihead_attn.in_proj_weight.copy_(torch.cat([T("w_qc"), T("w_kvc")]))
        lay.multihead_attn.in_proj_bias.copy_(torch.cat([T("b_qc"), z, T("b_vc")]))
        lay.multihead_attn.out_proj.weight.copy_(T("w_oc"))
        lay.multihead_attn.out_proj.bias.copy_(T("b_oc"))
        lay.linear1.weight.copy_(T("w_fc1")); lay.linear1.bias.copy_(T("b_fc1"))
        lay.linear2.weight.copy_(T("w_fc2")); lay.linear2.bias.copy_(T("b_fc2"))
        for i in (1, 2, 3):
            getattr(lay, f"norm{i}").weight.copy_(T(f"ln{i}_g"))
            getattr(lay, f"norm{i}").bias.copy_(T(f"ln{i}_b"))
    return lay.eval()


def test_full_forward_matches_torch_decoder_stack(small):
    """The whole target forward (embeddings, every layer, final LN, tied head)
    reduces to torch's pre-LN TransformerDecoderLayer stack."""
    orc, tw, _, A = small
    req = orc.new_request(A)
    toks = [5, 17, 999, 0, 42, 42, 7]
    logits, hist = orc.forward_full(req, toks)
    E = torch.from_numpy(tw["tok_emb"].astype(np.float64))
    x = (E[toks] + torch.from_numpy(tw["pos_emb"].astype(np.float64))[: len(toks)])[None]
    mem = torch.from_numpy(A.astype(np.float64))[None]
    causal = torch.nn.Transformer.generate_square_subsequent_mask(len(toks), dtype=torch.float64)
    hs = []
    with torch.no_grad():
        for l in range(SMALL.n_layers):
            x = _torch_decoder(SMALL, tw, l)(x, mem, tgt_mask=causal)
            if l in SMALL.hist_layers:
                hs.append(x[0].numpy())
        hf = F.layer_norm(x[0], (SMALL.d_model,), torch.from_numpy(tw["lnf_g"].astype(np.float64)),
                          torch.from_numpy(tw["lnf_b"].astype(np.float64)))
        ref = (hf @ E.T).numpy()
    np.testing.assert_allclose(logits, ref, rtol=0, atol=1e-9)
    np.testing.assert_allclose(hist, np.stack(hs, 1), atol=1e-10)


def test_cached_verify_equals_full_forward(small):
    orc, _, _, A = small
    toks = [3, 1, 4, 1, 5, 9, 2, 6, 5, 3, 5, 8]
    full, fh = orc.forward_full(orc.new_request(A), toks)
    req = orc.new_request(A)
    got = []
    for blk in ([0, 4], [4, 5], [5, 9], [9, 12]):
        got.append(orc.verify(req, toks[blk[0]:blk[1]]))
        req.L = blk[1]
    np.testing.assert_allclose(np.concatenate(got), full, atol=1e-10)
    np.testing.assert_allclose(req.hist[:12], fh, atol=1e-10)


def test_causal_and_frame_mask_invariants(small):
    orc, _, _, A = small
    r1, r2 = orc.new_request(A, frames=40), orc.new_request(A, frames=40)
    b1, b2 = [1, 2, 3, 4, 5, 6], [1, 2, 3, 77, 88, 99]
    l1, l2 = orc.verify(r1, b1), orc.verify(r2, b2)
    np.testing.assert_array_equal(l1[:3], l2[:3])         # later block tokens do not leak back
    assert np.abs(l1[3:] - l2[3:]).max() > 1e-3
    A2 = A.copy(); A2[40:] = 1e3                            # frames beyond F are never read
    r3 = orc.new_request(A2, frames=40)
    np.testing.assert_array_equal(orc.verify(r3, b1), l1)


def test_bf16_mode_tracks_fp32(small):
    orc, tw, dw, A = small
    ob = M.Oracle(SMALL, tw, dw, bf16=True)
    toks = [1, 2, 3, 4, 5]
    a, _ = orc.forward_full(orc.new_request(A), toks)
    b, _ = ob.forward_full(ob.new_request(A), toks)
    rel = np.abs(a - b).max() / np.abs(a).max()
    assert 1e-5 < rel < 3e-2


# ---------------------------------------------------------------- drafter

def test_drafter_layer_reduces_to_torch_decoder_layer(small):
    """At RoPE position 0 (identity rotation) the drafter layer is a pre-LN
    decoder layer whose self-attention keys/values are [history ; LN1(block)]
    through the same projections, with no mask — torch's MHA with
    key = value = concat(h_hist, LN1(x))."""
    orc, tw, dw, A = small
    req = orc.new_request(A)
    g = np.random.default_rng(4)
    x = g.standard_normal((9, SMALL.d_model))
    h_hist = g.standard_normal((5, SMALL.d_model))
    got = orc.drafter_layer(x, 1, np.zeros(9, int), h_hist, np.zeros(5, int), req.dck[1], req.dcv[1])
    lay = _torch_decoder(SMALL, dw, 1)
    X, Hh = torch.from_numpy(x)[None], torch.from_numpy(h_hist)[None]
    with torch.no_grad():
        h = lay.norm1(X)
        kv = torch.cat([Hh, h], dim=1)
        y = X + lay.self_attn(h, kv, kv, need_weights=False)[0]
        y = y + lay.multihead_attn(lay.norm2(y), torch.from_numpy(A.astype(np.float64))[None],
                                   torch.from_numpy(A.astype(np.float64))[None], need_weights=False)[0]
        y = y + lay.linear2(F.gelu(lay.linear1(lay.norm3(y))))
    np.testing.assert_allclose(got, y[0].numpy(), atol=1e-10)


def test_history_fusion_special_case(small):
    """With W_f = [I, 0] the fused history is LN_h of the first history
    layer's residual stream."""
    orc, tw, dw, A = small
    d = SMALL.d_model
    dw2 = dict(dw)
    dw2["fuse_w"] = np.concatenate([np.eye(d), np.zeros((d, d))], axis=1).astype(np.float32)
    o2 = M.Oracle(SMALL, tw, dw2)
    resid = np.random.default_rng(5).standard_normal((4, 2, d))
    ref = F.layer_norm(torch.from_numpy(resid[:, 0]), (d,), torch.from_numpy(dw["lnh_g"].astype(np.float64)),
                       torch.from_numpy(dw["lnh_b"].astype(np.float64))).numpy()
    np.testing.assert_allclose(o2.history_features(resid), ref, atol=1e-12)


def test_drafter_history_mask_and_block_symmetry(small):
    orc, _, _, A = small
    req = orc.new_request(A)
    orc.verify(req, [1, 2, 3, 4, 5, 6])
    req.L = 4
    z1 = orc.draft_logits(req, 9)
    req.hist[4:] = 123.0                                   # at/after the anchor: never read
    z2 = orc.draft_logits(req, 9)
    np.testing.assert_array_equal(z1, z2)
    assert z1.shape == (SMALL.K, SMALL.vocab)
    # the mask rows only differ by their RoPE positions: they must not all agree
    assert np.abs(z1[0] - z1[-1]).max() > 1e-6


def _torch_rope(x, pos, n_heads):
    """RoPE written as complex multiplication: each pair (2i, 2i+1) of a head
    is the complex number x_2i + j x_2i+1, turned by e^{j phi}, phi the fp32
    product of the position and theta_i = 10000^(-2i/d_head) (RoFormer;
    Whisper-Flash App. A.2: base 10,000, FP32 phases)."""
    R, d = x.shape
    dh = d // n_heads
    theta = torch.pow(torch.tensor(10000.0, dtype=torch.float64),
                      -torch.arange(0, dh, 2, dtype=torch.float64) / dh).float()
    phi = (torch.as_tensor(pos, dtype=torch.float32)[:, None] * theta[None, :]).double()
    rot = torch.polar(torch.ones_like(phi), phi)[:, None, :]
    xc = torch.view_as_complex(x.reshape(R, n_heads, dh // 2, 2).contiguous())
    return torch.view_as_real(xc * rot).reshape(R, d)


def _torch_heads_attend(q, k, v, n_heads):
    R, d = q.shape
    sp = lambda t: t.reshape(t.shape[0], n_heads, d // n_heads).transpose(0, 1)
    return F.scaled_dot_product_attention(sp(q), sp(k), sp(v)).transpose(0, 1).reshape(R, d)


def _torch_drafter_logits(shape, tw, dw, resid, A, anchor, t, shift=0):
    """The drafter of Whisper-Flash §3.2 (Eq. 2) / App. A.2 assembled from
    torch primitives in float64: input rows [Emb(anchor), m, ..., m] with no
    absolute position; history memory = LN_h(W_f concat(residual streams))
    of the accepted positions 0..t-1; per layer one unmasked softmax of the
    block queries over [history ; block] keys (RoPE at the text positions,
    history at 0..t-1, block at t..t+K, all moved by `shift`), cross-attention
    to the drafter's own acoustic K/V, GELU FFN; then the drafter's final LN
    and the tied head on the K mask rows."""
    d, nh, K = shape.d_model, shape.n_heads, shape.K
    T = lambda src, n: torch.from_numpy(np.asarray(src[n], dtype=np.float64))
    E = T(tw, "tok_emb")
    hh = F.layer_norm(torch.from_numpy(resid.reshape(t, -1)) @ T(dw, "fuse_w").T, (d,),
                      T(dw, "lnh_g"), T(dw, "lnh_b"))
    x = torch.cat([E[anchor][None], T(dw, "mask_emb")[None].repeat(K, 1)])
    pb = [shift + t + j for j in range(K + 1)]
    ph = [shift + j for j in range(t)]
    mem = torch.from_numpy(np.asarray(A, dtype=np.float64))
    for l in range(shape.drafter_layers):
        W = lambda n: T(dw, f"layers.{l}.{n}")
        wq, wk, wv = W("w_qkv")[:d], W("w_qkv")[d:2 * d], W("w_qkv")[2 * d:]
        h = F.layer_norm(x, (d,), W("ln1_g"), W("ln1_b"))
        q = _torch_rope(h @ wq.T + W("b_q"), pb, nh)
        k = torch.cat([_torch_rope(hh @ wk.T, ph, nh), _torch_rope(h @ wk.T, pb, nh)])
        v = torch.cat([hh @ wv.T + W("b_v"), h @ wv.T + W("b_v")])
        x = x + F.linear(_torch_heads_attend(q, k, v, nh), W("w_o"), W("b_o"))
        qc = F.linear(F.layer_norm(x, (d,), W("ln2_g"), W("ln2_b")), W("w_qc"), W("b_qc"))
        kc, vc = mem @ W("w_kvc")[:d].T, mem @ W("w_kvc")[d:].T + W("b_vc")
        x = x + F.linear(_torch_heads_attend(qc, kc, vc, nh), W("w_oc"), W("b_oc"))
        f = F.gelu(F.linear(F.layer_norm(x, (d,), W("ln3_g"), W("ln3_b")), W("w_fc1"), W("b_fc1")))
        x = x + F.linear(f, W("w_fc2"), W("b_fc2"))
    hf = F.layer_norm(x[1:], (d,), T(dw, "lnf_g"), T(dw, "lnf_b"))
    return (hf @ E.T).numpy()


def test_draft_logits_match_torch_drafter_block(small):
    """Pins the drafter's block assembly end to end (anchor row first, K mask
    rows after it, RoPE at t..t+K against history at 0..t-1, proposals from
    rows 1..K): the oracle equals the torch drafter above, and moving every
    position by the same amount leaves the logits unchanged (RoPE only sees
    relative positions), so no absolute offset hides in either."""
    orc, tw, dw, A = small
    req = orc.new_request(A)
    t = 6
    rng = np.random.default_rng(12)
    req.hist[:t] = rng.standard_normal((t, SMALL.n_hist, SMALL.d_model))
    req.L = t
    got = orc.draft_logits(req, 321)
    ref = _torch_drafter_logits(SMALL, tw, dw, req.hist[:t], A, 321, t)
    assert got.shape == (SMALL.K, SMALL.vocab)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-9)
    moved = _torch_drafter_logits(SMALL, tw, dw, req.hist[:t], A, 321, t, shift=37)
    np.testing.assert_allclose(got, moved, rtol=0, atol=1e-4 * np.abs(ref).max())
    # the anchor token and the history both reach every proposal row
    assert (np.abs(orc.draft_logits(req, 322) - got).max(axis=1) > 1e-8).all()
    req.hist[0] += 1.0
    assert (np.abs(orc.draft_logits(req, 321) - got).max(axis=1) > 1e-8).all()


def test_drafter_parameter_counts_match_paper():
    """Whisper-Flash §3.2 / Table 3: 60.7M trainable parameters with audio and
    history, 47.5M without direct audio, 52.5M without the target history."""
    gold = _load("paper_numbers.json")["drafter_params_millions"]
    s = synth.LARGE_V3
    sizes = dict((n, int(np.prod(sh))) for n, sh in synth.drafter_tensor_shapes(s))
    full = sum(sizes.values())
    cross = sum(v for n, v in sizes.items()
                if any(n.endswith(k) for k in ("w_qc", "w_kvc", "w_oc", "b_qc", "b_vc", "b_oc", "ln2_g", "ln2_b")))
    hist = sizes["fuse_w"] + sizes["lnh_g"] + sizes["lnh_b"]
    tol = gold["printed_precision"]
    assert abs(full / 1e6 - gold["audio_and_history"]) < tol
    assert abs((full - cross) / 1e6 - gold["without_audio"]) < gold["tolerance_without_audio"]
    assert abs((full - hist) / 1e6 - gold["without_history"]) < tol
    shp = _load("paper_numbers.json")["whisper_large_v3_shape"]
    assert list(s.hist_layers) == shp["hist_layers"] and s.n_layers == shp["n_layers"]
    assert s.n_hist * s.d_model == shp["concat_width"]


# ---------------------------------------------------------------- acceptance

def test_figure1_worked_example():
    ex = _load("paper_numbers.json")["figure1_worked_example"]
    words = sorted(set(ex["candidates"]) | set(ex["target_argmax"]))
    ids = {w: i for i, w in enumerate(words)}
    block = [ids["the"]] + [ids[w] for w in ex["candidates"]]
    g = [ids[w] for w in ex["target_argmax"]]
    acc = M.accept_greedy(block, 8, g, budget=100, eos=10 ** 6)
    assert acc.a == ex["accepted"]
    assert acc.emitted == [ids[w] for w in ex["emitted"]]
    assert acc.next_anchor == ids[ex["next_anchor"]]


def test_accept_eos_budget_and_bonus():
    eos = 9
    acc = M.accept_greedy([1, 2, eos, 4], 3, [2, eos, 4, 5], budget=50, eos=eos)
    assert acc.a == 2 and acc.emitted == [2, eos] and acc.done          # no bonus after EOS
    acc = M.accept_greedy([1, 2, 3], 2, [2, 3, 7], budget=50, eos=eos)
    assert acc.a == 2 and acc.emitted == [2, 3, 7] and not acc.done      # bonus
    acc = M.accept_greedy([1, 2, 3], 2, [2, eos, 7], budget=50, eos=eos)
    assert acc.emitted == [2, eos] and acc.done                          # EOS correction
    acc = M.accept_greedy([1, 2, 3], 2, [2, 3, 7], budget=3, eos=eos)
    assert acc.done and len(acc.emitted) == 3                            # budget used up


@pytest.fixture(scope="module")
def small_prompted():
    s = synth.ModelShape("small", 3, 128, 2, 512, vocab=1000, max_pos=96, hist_layers=(0, 2),
                         dtype="f32", eos_id=999, prompt=(990, 991, 992, 993))
    tw = synth.target_weights(s, 12)
    dw = synth.drafter_weights(s, 12, tw)
    return s, M.Oracle(s, tw, dw), synth.encoder_states(s, 12, 0, frames=50)


def test_speculative_equals_ar_for_all_draft_kinds(small_prompted):
    s, orc, A = small_prompted
    budget = 25
    ar = M.greedy_plain(orc, orc.new_request(A), budget)
    traj = list(s.prompt) + ar.tokens
    perfect = lambda req, a, t, n: [traj[t + j] if t + j < len(traj) else 0 for j in range(1, n + 1)]
    wrong = lambda req, a, t, n: [(traj[t + j] + 1) % s.vocab if t + j < len(traj) else 0 for j in range(1, n + 1)]
    plan = synth.corruption_plan(1, s.max_pos, s.K, synth.corruption_p_const(s.K, 0.3), s.vocab, 3)
    corrupt = M.corrupted_proposer(traj, plan.mask[0], plan.tok[0])
    for prop, tau in ((perfect, None), (wrong, 1.0), (corrupt, None), (M.drafter_proposer(orc), None)):
        sp = M.speculative_greedy(orc, orc.new_request(A), budget, prop)
        assert sp.tokens == ar.tokens
        met = M.acceptance_metrics(sp, s.K)
        if tau is not None:
            assert met["tau"] == tau
        # emitted per round = a + 1 (no EOS here): tau = 1 + mean a
        assert abs(met["tau"] - (1 + met["mean_a"])) < 1e-12
    sp = M.speculative_greedy(orc, orc.new_request(A), budget, perfect)
    assert sp.accepted[:2] == [s.K, s.K]          # perfect drafts: K+1 tokens per call
    assert 1 + sum(sp.emitted) == budget          # prefill emits the first token


def test_rollback_keeps_L_plus_1_plus_a(small_prompted):
    s, orc, A = small_prompted
    ar = M.greedy_cached(orc, orc.new_request(A), 10)
    req = orc.new_request(A)
    acc, _ = M.prefill(orc, req, 50)
    assert req.L == len(s.prompt) and acc.next_anchor == ar.tokens[0]
    L0 = req.L
    block = [ar.tokens[0], ar.tokens[1], ar.tokens[2], (ar.tokens[3] + 1) % s.vocab]
    lg = orc.verify(req, block)
    g = [M.argmax_lowest(z) for z in lg]
    acc2 = M.accept_greedy(block, 3, g, 50, s.eos_id)
    assert acc2.a == 2 and acc2.emitted == ar.tokens[1:4]
    req.L += 1 + acc2.a
    assert req.L == L0 + 3
    # re-verifying from the rolled-back cache reproduces the accepted rows
    r2 = orc.new_request(A)
    M.prefill(orc, r2, 50)
    lg3 = orc.verify(r2, block[:3])
    np.testing.assert_allclose(lg3, lg[:3], atol=1e-10)
    # the next round starts at L0 + 3 and overwrites the rejected position
    lg4 = orc.verify(req, [acc2.next_anchor])
    assert M.argmax_lowest(lg4[0]) == ar.tokens[4]


def test_budget_limits_candidates(small_prompted):
    s, orc, A = small_prompted
    seen = []
    def prop(req, a, t, n):
        seen.append(n)
        return [0] * n
    sp = M.speculative_greedy(orc, orc.new_request(A), 5, prop)
    assert len(sp.tokens) == 5
    R = 4
    for n in seen:                                 # n_prop = min(K, R-1)
        assert n == min(s.K, R - 1)
        R -= 1


def test_synthetic_acceptance_closed_form(small_prompted):
    """E[a] = sum_k prod_{j<=k} (1 - p_j) for independently corrupted drafts
    of the target's own trajectory (K = 8, p = 0.2: 3.329)."""
    s, orc, A = small_prompted
    budget = 90
    ar = M.greedy_cached(orc, orc.new_request(A), budget)
    traj = list(s.prompt) + ar.tokens
    pj = synth.corruption_p_const(s.K, 0.2)
    expect = sum(np.prod(1 - pj[:k]) for k in range(1, s.K + 1))
    assert abs(expect - 3.329) < 1e-3
    full_a = []
    for seed in range(6):
        plan = synth.corruption_plan(1, s.max_pos, s.K, pj, s.vocab, 100 + seed)
        sp = M.speculative_greedy(orc, orc.new_request(A), budget,
                                  M.corrupted_proposer(traj, plan.mask[0], plan.tok[0]))
        assert sp.tokens == ar.tokens
        full_a += [a for a, n in zip(sp.accepted, sp.proposed) if n == s.K]
    full_a = np.array(full_a)
    se = full_a.std() / math.sqrt(len(full_a))
    assert abs(full_a.mean() - expect) < 4 * se + 0.05, (full_a.mean(), expect, se)


def test_paper_metric_identities():
    g = _load("paper_numbers.json")
    K = g["table_a4_identity_a_equals_alpha_K"]["K"]
    for r in g["table_a4_identity_a_equals_alpha_K"]["rows"]:
        assert abs(r["alpha"] * K - r["a"]) < g["table_a4_identity_a_equals_alpha_K"]["printed_precision"]
    for r in g["table_a5_tau_bound"]["rows"]:
        assert r["tau"] <= 1 + r["alpha"] * r["K"] + 1e-9


# ---------------------------------------------------------------- rejection rule

def _grid_uniform(n):
    return (np.arange(n) + 0.5) / n


def test_inverse_cdf_and_fp32_softmax_by_hand():
    """Sampling helpers pinned by hand and by brute force: the inverse CDF
    returns the smallest id whose running sum exceeds u * total (zero-weight
    ids are never drawn, u = 0 gives the first id with weight); the FP32
    softmax at temperature T equals torch's float64 softmax of z / T within
    FP32 rounding and gives suppressed ids probability zero."""
    w = np.array([0.0, 1.0, 0.0, 2.0, 0.0])
    # running sums 0, 1, 1, 3, 3: by hand
    assert M.sample_inverse_cdf(w, 0.0) == 1
    assert M.sample_inverse_cdf(w, 0.3) == 1          # 0.9 < 1
    assert M.sample_inverse_cdf(w, 1 / 3 + 1e-9) == 3
    assert M.sample_inverse_cdf(w, 0.999999) == 3
    rng = np.random.default_rng(3)
    for _ in range(200):
        n = int(rng.integers(1, 40))
        ww = rng.random(n) * (rng.random(n) < 0.6)
        if ww.sum() == 0:
            ww[int(rng.integers(0, n))] = 1.0
        u = float(rng.random())
        tgt = u * ww.sum()
        run, want = 0.0, None
        for v in range(n):                             # brute force: first id past the target
            run += ww[v]
            if run > tgt:
                want = v
                break
        assert M.sample_inverse_cdf(ww, u) == want
        assert ww[want] > 0
    z = rng.normal(size=300).astype(np.float32)
    sup = [0, 7, 299]
    for T in (0.7, 1.0, 1.5):
        p = M.probs_fp32(z, T, sup)
        assert p.dtype == np.float32 and np.all(p[sup] == 0)
        zz = torch.tensor(z.astype(np.float64) / T)
        zz[sup] = -math.inf
        ref = torch.softmax(zz, 0).numpy()
        np.testing.assert_allclose(p, ref, rtol=2e-6, atol=1e-9)
        assert abs(float(p.astype(np.float64).sum()) - 1.0) < 1e-5


def test_rejection_rule_preserves_target_distribution_exactly():
    """Quadrature over the acceptance and residual uniforms: the first
    emitted token's distribution equals p (Leviathan et al. / Chen et al.,
    as used in Whisper-Flash §3.1)."""
    V, T = 7, 0.7
    g = np.random.default_rng(8)
    zp, zq = g.standard_normal(V) * 2, g.standard_normal(V) * 2
    p = M.probs_fp32(zp, T).astype(np.float64)
    q = M.probs_fp32(zq, T).astype(np.float64)
    N = 4000
    grid = _grid_uniform(N)
    dist = np.zeros(V)
    for y in range(V):
        for u in grid[::8]:
            for u2 in grid[::40]:
                uni = lambda j, purpose, u=u, u2=u2: u if purpose == philox.PURPOSE_ACCEPT else u2
                acc, _ = M.accept_sampling([0, y], 1, [zp, zp], [zq], T, 0, 0, 0, 10, eos=10 ** 6, uniform=uni)
                dist[acc.emitted[0]] += q[y]
    dist /= len(grid[::8]) * len(grid[::40])
    np.testing.assert_allclose(dist, p, atol=3e-3)


def test_rejection_rule_special_cases():
    V, T = 50, 1.0
    g = np.random.default_rng(9)
    z = g.standard_normal(V)
    # q == p: always accepted
    for rnd in range(40):
        acc, _ = M.accept_sampling([0, 3, 4], 2, [z, z, z], [z, z], T, 5, 0, rnd, 10, 10 ** 6)
        assert acc.a == 2
    # p(y) == 0 (suppressed): never accepted
    for rnd in range(40):
        acc, _ = M.accept_sampling([0, 3], 1, [z, z], [z], T, 5, 0, rnd, 10, 10 ** 6, suppress=[3])
        assert acc.a == 0 and acc.emitted[0] != 3
    # disjoint supports: the residual is p itself
    zp = np.full(V, -np.inf); zp[:10] = g.standard_normal(10)
    zq = np.full(V, -np.inf); zq[20:] = g.standard_normal(30)
    p = M.probs_fp32(zp, T)
    for rnd in range(40):
        acc, det = M.accept_sampling([0, 25], 1, [zp, zp], [zq], T, 5, 0, rnd, 10, 10 ** 6)
        assert acc.a == 0
        assert det[-1][0] == "residual" and det[-1][3] == M.sample_inverse_cdf(p, det[-1][2])
    # T -> 0 reduces to greedy verification
    zt, zd = g.standard_normal(V), g.standard_normal(V)
    acc, _ = M.accept_sampling([0, int(np.argmax(zt))], 1, [zt, zt], [zd], 1e-4, 5, 0, 0, 10, 10 ** 6)
    assert acc.a == 1
    y = (int(np.argmax(zt)) + 1) % V
    acc, _ = M.accept_sampling([0, y], 1, [zt, zt], [zd], 1e-4, 5, 0, 0, 10, 10 ** 6)
    assert acc.a == 0 and acc.emitted == [int(np.argmax(zt))]


def test_first_token_chi_square_montecarlo():
    """Monte Carlo over Philox streams: first emitted token ~ p."""
    V, T = 20, 0.7
    g = np.random.default_rng(10)
    zp = g.standard_normal(V)
    zq = zp + g.standard_normal(V)
    p = M.probs_fp32(zp, T).astype(np.float64)
    n = 6000
    counts = np.zeros(V)
    for r in range(n):
        y = M.sample_draft(zq, T, 7, 0, r, 1)
        acc, _ = M.accept_sampling([0, y], 1, [zp, zp], [zq], T, 7, 0, r, 10, 10 ** 6)
        counts[acc.emitted[0]] += 1
    chi2 = ((counts - n * p) ** 2 / (n * p)).sum()
    assert chi2 < 43.8   # chi-square 99.9% quantile, 19 dof


# ---------------------------------------------------------------- truncated verification, confidence stopping

@pytest.fixture(scope="module")
def small_drafter():
    s = synth.ModelShape("small-d", 2, 128, 2, 256, vocab=300, max_pos=64, hist_layers=(0, 1), dtype="f32",
                         eos_id=299, prompt=(290, 291, 292, 293))
    tw = synth.target_weights(s, 71)
    dw = synth.drafter_weights(s, 71, tw)
    orc = M.Oracle(s, tw, dw)
    A = synth.encoder_states(s, 71, 0, frames=50)
    return s, orc, A


@pytest.mark.parametrize("k_verify,threshold", [(1, 0.0), (2, 0.0), (4, 0.3), (8, 0.0), (8, 0.3), (8, 0.05)])
def test_limited_speculation_is_exact_and_accounts_tau(small_drafter, k_verify, threshold):
    """Truncating the verified block (Whisper-Flash Table A5) and stopping at
    low confidence (Alignment Drift Table 21) keep the output equal to
    autoregressive greedy decoding; tokens per target call follow
    tau = 1 + (accepted per round), <= 1 + alpha K' (Table A5's identity)."""
    s, orc, A = small_drafter
    budget = 30
    ar = M.greedy_cached(orc, orc.new_request(A), budget).tokens
    res = M.speculative_greedy_limited(orc, orc.new_request(A), budget, k_verify, threshold)
    assert res.tokens == ar
    assert max(res.proposed) <= k_verify
    a, prop = sum(res.accepted), sum(res.proposed)
    emitted_rounds = sum(res.emitted)
    assert emitted_rounds == res.rounds + a                 # no EOS: each round = accepted + 1
    tau = emitted_rounds / res.rounds
    alpha = a / max(prop, 1)
    assert tau <= 1 + alpha * k_verify + 1e-12
    if threshold == 0.0 and k_verify == s.K:
        base = M.speculative_greedy(orc, orc.new_request(A), budget, M.drafter_proposer(orc))
        assert base.proposed == res.proposed and base.accepted == res.accepted


def test_confidence_threshold_one_means_no_proposals(small_drafter):
    """No probability reaches a threshold above 1: every round verifies the
    anchor alone, so the loop is autoregressive (one token per target call)."""
    s, orc, A = small_drafter
    res = M.speculative_greedy_limited(orc, orc.new_request(A), 12, s.K, 1.01)
    assert set(res.proposed) == {0}
    assert res.rounds == 11                                 # the prefill emits the first token


def test_proposal_confidence_and_stop_rule_brute_force():
    """The confidence is the drafter's softmax probability of its token
    (torch softmax in float64 agrees to fp32 precision); the limit is the
    first position below the threshold, capped by K' and R - 1."""
    g = np.random.default_rng(14)
    q = g.standard_normal((8, 50)) * 3
    cand = [int(np.argmax(r)) for r in q]
    conf = [M.proposal_confidence(q[j], cand[j], 0.0) for j in range(8)]
    ref = torch.softmax(torch.from_numpy(q), dim=-1).numpy()
    np.testing.assert_allclose(conf, [ref[j, cand[j]] for j in range(8)], rtol=1e-5)
    for thr in (0.0, 0.2, 0.5, 0.9):
        for kv in (1, 3, 8):
            for R in (1, 2, 5, 100):
                n = 0
                while n < min(kv, R - 1) and (thr <= 0 or conf[n] >= thr):
                    n += 1
                assert M.limit_proposals(cand, q, kv, thr, 0.0, R) == n
    # sampling: confidence at the drafter's temperature
    assert abs(M.proposal_confidence(q[0], 3, 0.7) -
               torch.softmax(torch.from_numpy(q[0] / 0.7), -1)[3].item()) < 1e-6


# ---------------------------------------------------------------- verification-attention readout, windowed drafter

def test_attention_peaks_match_torch_head_averaged_weights():
    """The readout is the argmax over frames of torch's head-averaged
    multi-head attention weights (identity projections)."""
    g = np.random.default_rng(21)
    d, heads, R, F_ = 128, 2, 5, 37
    q, k = g.standard_normal((R, d)), g.standard_normal((F_, d))
    orc = M.Oracle(SMALL, synth.target_weights(SMALL, 11), None)
    got = orc.attention_peaks(q, k)
    eye = torch.eye(d, dtype=torch.float64)
    _, w = F.multi_head_attention_forward(
        torch.from_numpy(q)[:, None], torch.from_numpy(k)[:, None], torch.from_numpy(k)[:, None], d, heads,
        in_proj_weight=torch.cat([eye, eye, eye]), in_proj_bias=None, bias_k=None, bias_v=None,
        add_zero_attn=False, dropout_p=0.0, out_proj_weight=eye, out_proj_bias=None, need_weights=True,
        average_attn_weights=True)
    assert got == [int(i) for i in w[0].argmax(dim=-1)]


def test_windowed_drafter_equals_drafter_on_window_frames(small):
    """The windowed drafter cross-attention equals the torch drafter given only
    the window's encoder frames; a window covering every frame is the
    unrestricted drafter."""
    orc, tw, dw, A = small
    req = orc.new_request(A)
    t = 5
    req.hist[:t] = np.random.default_rng(22).standard_normal((t, SMALL.n_hist, SMALL.d_model))
    req.L = t
    req.center = 31
    got = orc.draft_logits(req, 77, half_width=6)
    ref = _torch_drafter_logits(SMALL, tw, dw, req.hist[:t], A[25:38], 77, t)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-9)
    req.center = 2                                       # clipped at frame 0
    np.testing.assert_allclose(orc.draft_logits(req, 77, half_width=6),
                               _torch_drafter_logits(SMALL, tw, dw, req.hist[:t], A[0:9], 77, t), atol=1e-9)
    req.center = 30
    np.testing.assert_array_equal(orc.draft_logits(req, 77, half_width=1000), orc.draft_logits(req, 77))


def test_windowed_speculation_is_exact(small_drafter):
    s, orc, A = small_drafter
    ar = M.greedy_cached(orc, orc.new_request(A), 20).tokens
    res = M.speculative_greedy_windowed(orc, orc.new_request(A), 20, 1, 5)
    assert res.tokens == ar
    assert all(0 <= c < 50 for c in res.margins)


# ---------------------------------------------------------------- tree drafts (Alignment Drift App. E.3)

TREE_PARENT = [-1, 0, 0, 0, 1, 2, 4, 6, 7, 8, 9, 10]      # 11 candidate nodes under the anchor
TREE_RANK = [0, 0, 1, 2, 0, 0, 0, 0, 0, 0, 0, 0]


def test_tree_verify_node_logits_equal_plain_forward_over_root_path(small):
    """Every node's logits equal the plain uncached forward over prompt +
    cache + the tokens on the node's root path (the tree mask is exactly
    'see your ancestors')."""
    orc, _, _, A = small
    req = orc.new_request(A)
    prefix = [5, 6, 7, 8, 9]
    orc.verify(req, prefix)
    req.L = len(prefix)
    toks = [11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22]
    lg = orc.verify_tree(req, toks, TREE_PARENT)
    for j in range(len(toks)):
        path, c = [], j
        while c >= 0:
            path.append(toks[c])
            c = TREE_PARENT[c]
        full, _ = orc.forward_full(orc.new_request(A), prefix + path[::-1])
        np.testing.assert_allclose(lg[j], full[-1], atol=1e-9)


def test_tree_speculation_exact_and_one_branch_is_linear(small_drafter):
    """A candidate tree keeps the output equal to autoregressive greedy
    decoding, and a one-branch tree (a chain of K nodes taking the argmax of
    each mask row) reproduces the linear drafter decode round for round."""
    s, orc, A = small_drafter
    budget = 24
    ar = M.greedy_cached(orc, orc.new_request(A), budget).tokens
    res = M.speculative_greedy_tree(orc, orc.new_request(A), budget, TREE_PARENT, TREE_RANK)
    assert res.tokens == ar
    chain = [-1] + list(range(s.K))
    lin_t = M.speculative_greedy_tree(orc, orc.new_request(A), budget, chain, [0] * (s.K + 1))
    lin = M.speculative_greedy(orc, orc.new_request(A), budget, M.drafter_proposer(orc))
    assert lin_t.tokens == lin.tokens == ar
    # a linear round proposes min(K, R-1); the tree proposes its nodes but accepts at most R-1
    assert lin_t.accepted == lin.accepted and lin_t.rounds == lin.rounds


def test_accept_tree_walk_and_tokens_by_rank():
    g = [50, 60, 0, 0, 70, 0, 55, 0, 0, 0, 0, 0]        # argmax at node j
    toks = [1, 50, 51, 52, 60, 53, 70, 71, 72, 73, 74, 75]
    acc, path = M.accept_tree(toks, TREE_PARENT, g, 100, 999)
    assert path == [0, 1, 4, 6] and acc.emitted == [50, 60, 70, 55] and acc.a == 3
    acc, path = M.accept_tree(toks, TREE_PARENT, g, 3, 999)       # at most R - 1 = 2 candidates
    assert path == [0, 1, 4] and acc.emitted == [50, 60, 70]
    acc, path = M.accept_tree(toks, TREE_PARENT, [51] + g[1:], 100, 999)   # second branch at depth 1
    assert path[:2] == [0, 2]
    q = np.zeros((8, 10)); q[0, [4, 7, 2]] = [3.0, 2.0, 2.0]
    t = M.tree_tokens(q, TREE_PARENT, TREE_RANK, 9)
    assert t[:4] == [9, 4, 2, 7]                                  # ties rank the lower id first


# ---------------------------------------------------------------- audio encoder

from oracle import encoder as ENC

ENC_SMALL = synth.EncoderShape("enc-small", 2, 128, 2, 512, 16, n_frames=48, dtype="f32")


def test_encoder_positions_closed_forms():
    """Sine half and cosine half of one frequency: sin^2 + cos^2 = 1; row 0 is
    (0, ..., 0, 1, ..., 1); the first frequency is 1 rad per position and the
    last 1/10000."""
    P = ENC.sinusoids(1500, 384)
    np.testing.assert_allclose(P[:, :192] ** 2 + P[:, 192:] ** 2, 1.0, atol=1e-12)
    np.testing.assert_array_equal(P[0], np.r_[np.zeros(192), np.ones(192)])
    t = np.arange(1500)
    np.testing.assert_allclose(P[:, 0], np.sin(t), atol=1e-12)
    np.testing.assert_allclose(P[:, 191], np.sin(t / 10000.0), atol=1e-12)
    np.testing.assert_allclose(P[:, 383], np.cos(t / 10000.0), atol=1e-12)


def test_encoder_fp64_equals_torch_modules():
    """The whole fp64 encoder against torch: F.conv1d (padding 1, strides 1
    and 2) with exact GELU, an independently built position table,
    nn.TransformerEncoderLayer(norm_first=True, activation='gelu') holding
    the same weights (key bias zero), and F.layer_norm."""
    e = ENC_SMALL
    w = synth.encoder_weights(e, 3)
    mel = synth.mel_input(e, 3, 0)
    ora = ENC.Encoder(e, w).encode(mel)
    t = {k: torch.tensor(np.asarray(v, dtype=np.float64)) for k, v in w.items()}
    x = torch.tensor(np.asarray(mel, dtype=np.float64))[None]
    x = F.gelu(F.conv1d(x, t["conv1_w"], t["conv1_b"], stride=1, padding=1))
    x = F.gelu(F.conv1d(x, t["conv2_w"], t["conv2_b"], stride=2, padding=1))[0].T
    d, F_ = e.d_model, e.n_frames
    pos = torch.arange(F_, dtype=torch.float64)[:, None]
    inv = 10000.0 ** (-torch.arange(d // 2, dtype=torch.float64) / (d // 2 - 1))
    x = (x + torch.cat([torch.sin(pos * inv), torch.cos(pos * inv)], dim=1))[None]
    for l in range(e.n_layers):
        p = f"layers.{l}."
        layer = torch.nn.TransformerEncoderLayer(d, e.n_heads, e.d_ff, dropout=0.0, activation="gelu",
                                                 norm_first=True, batch_first=True, dtype=torch.float64)
        with torch.no_grad():
            layer.self_attn.in_proj_weight.copy_(t[p + "w_qkv"])
            layer.self_attn.in_proj_bias.copy_(torch.cat([t[p + "b_q"], torch.zeros(d, dtype=torch.float64),
                                                          t[p + "b_v"]]))
            layer.self_attn.out_proj.weight.copy_(t[p + "w_o"])
            layer.self_attn.out_proj.bias.copy_(t[p + "b_o"])
            layer.linear1.weight.copy_(t[p + "w_fc1"]); layer.linear1.bias.copy_(t[p + "b_fc1"])
            layer.linear2.weight.copy_(t[p + "w_fc2"]); layer.linear2.bias.copy_(t[p + "b_fc2"])
            layer.norm1.weight.copy_(t[p + "ln1_g"]); layer.norm1.bias.copy_(t[p + "ln1_b"])
            layer.norm2.weight.copy_(t[p + "ln2_g"]); layer.norm2.bias.copy_(t[p + "ln2_b"])
        layer.eval()
        with torch.no_grad():
            x = layer(x)
    ref = F.layer_norm(x[0], (d,), t["lnp_g"], t["lnp_b"], eps=1e-5).numpy()
    np.testing.assert_allclose(ora, ref, atol=1e-9, rtol=1e-9)


def test_encoder_conv_stem_by_brute_force():
    """Output position t of the stride-2 convolution reads mel frames 2t-1 ..
    2t+1 of the first convolution's output (zero outside): one output value
    summed term by term."""
    e = ENC_SMALL
    w = synth.encoder_weights(e, 4)
    mel = np.asarray(synth.mel_input(e, 4, 1), dtype=np.float64)
    h1 = ENC.conv1d(mel, w["conv1_w"], w["conv1_b"], 1)
    for t, o in ((0, 5), (17, 0), (e.n_frames - 1, 127)):
        s = float(w["conv2_b"][o])
        for k in range(3):
            src = 2 * t + k - 1
            if 0 <= src < 2 * e.n_frames:
                s += sum(float(w["conv2_w"][o, c, k]) * h1[c, src] for c in range(e.d_model))
        assert abs(ENC.conv1d(h1, w["conv2_w"], w["conv2_b"], 2)[o, t] - s) < 1e-12


def test_encoder_bf16_mode_stays_near_fp64():
    """bf16 storage rounding moves the encoder output by far less than the
    2e-2 parity tolerance (relative to the largest output)."""
    e = synth.EncoderShape("enc-small-bf16", 2, 128, 2, 512, 16, n_frames=48, dtype="bf16")
    w = synth.encoder_weights(e, 5)
    mel = synth.mel_input(e, 5, 0)
    a = ENC.Encoder(e, w, bf16=True).encode(mel)
    b = ENC.Encoder(e, w, bf16=False).encode(mel)
    assert np.abs(a - b).max() < 2e-2 * np.abs(b).max()
