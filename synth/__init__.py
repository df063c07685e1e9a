"""Seeded synthetic inputs for speculative Whisper decoding.

This module is the ONLY code shared by the CPU oracle and the CUDA path.  It
draws random numbers and lays them out; it holds none of the method's
arithmetic (no layer norm, attention, softmax, acceptance or sampling).

What it produces
  * model shapes (Whisper large-v3, large-v3-turbo and a tiny 4-layer shape);
  * decoder / drafter weights, N(0, 0.02) random init, one independent PCG64
    stream per tensor so that any tensor can be regenerated on its own;
  * encoder states A = E(x) ~ N(0, 1) for the decoding path (Whisper-Flash
    §3.2 names A as the acoustic memory), and for the audio encoder its
    weights and log-mel stand-ins;
  * workload plans: synthetic draft corruption, transcript budgets, varlen
    frame counts.

Weights for bf16 models are returned as float32 arrays whose values are
exactly representable in bf16 (round-to-nearest-even of the float32 draw),
plus a uint16 view for upload.  That rounding is input formatting, done once
here, not a storage point of the method.

Blob layout (the byte order that ``ws_load_weights`` expects; every tensor is
row-major, [out, in] for matrices, in the model dtype, back to back):

  target blob : tok_emb[V,d], pos_emb[P,d], layer 0..nL-1, lnf_g[d], lnf_b[d]
  drafter blob: fuse_w[d, n_hist*d], lnh_g[d], lnh_b[d], mask_emb[d],
                lnf_g[d], lnf_b[d], layer 0..1
  layer       : w_qkv[3d,d] (rows q|k|v), w_o[d,d], w_qc[d,d],
                w_kvc[2d,d] (rows k|v), w_oc[d,d], w_fc1[f,d], w_fc2[d,f],
                b_q, b_v, b_o, b_qc, b_vc, b_oc [d each], b_fc1[f], b_fc2[d],
                ln1_g, ln1_b, ln2_g, ln2_b, ln3_g, ln3_b [d each]

There is no key bias and no cross-key bias (Whisper convention).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
import numpy as np

# Control-token ids used as the 4-token prompt and the end-of-transcript id.
# They only need to be valid ids < vocab; with random weights EOS is rare.
PROMPT = (50258, 50259, 50360, 50364)
EOS_ID = 50257


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    d_ff: int
    vocab: int = 51866
    max_pos: int = 448
    hist_layers: tuple = (0, 1, 2, 3)
    drafter_layers: int = 2
    K: int = 8
    dtype: str = "f32"           # "f32" or "bf16"
    eos_id: int = EOS_ID
    prompt: tuple = PROMPT

    @property
    def d_head(self) -> int:
        return self.d_model // self.n_heads

    @property
    def n_hist(self) -> int:
        return len(self.hist_layers)


# Whisper large-v3: 32 decoder layers, width 1280, 20 heads, FFN 5120.
LARGE_V3 = ModelShape("large-v3", 32, 1280, 20, 5120,
                      hist_layers=(1, 8, 15, 22, 29), dtype="bf16")
# Whisper large-v3-turbo: the same widths with a 4-layer decoder.
TURBO = ModelShape("large-v3-turbo", 4, 1280, 20, 5120, dtype="bf16")
# Tiny Whisper-style decoder used as the fp32 parity shape.
TINY = ModelShape("tiny", 4, 384, 6, 1536, dtype="f32")

SHAPES = {"large-v3": LARGE_V3, "large-v3-turbo": TURBO, "tiny": TINY}


def with_dtype(shape: ModelShape, dtype: str) -> ModelShape:
    return replace(shape, dtype=dtype)


# ---------------------------------------------------------------- layouts

LAYER_MATS = ("w_qkv", "w_o", "w_qc", "w_kvc", "w_oc", "w_fc1", "w_fc2")
LAYER_VECS = ("b_q", "b_v", "b_o", "b_qc", "b_vc", "b_oc", "b_fc1", "b_fc2",
              "ln1_g", "ln1_b", "ln2_g", "ln2_b", "ln3_g", "ln3_b")


def layer_tensor_shapes(s: ModelShape):
    d, f = s.d_model, s.d_ff
    shp = {"w_qkv": (3 * d, d), "w_o": (d, d), "w_qc": (d, d),
           "w_kvc": (2 * d, d), "w_oc": (d, d), "w_fc1": (f, d),
           "w_fc2": (d, f), "b_fc1": (f,)}
    out = []
    for n in LAYER_MATS + LAYER_VECS:
        out.append((n, shp.get(n, (d,))))
    return out


def target_tensor_shapes(s: ModelShape):
    """(name, shape) in blob order for the target decoder."""
    d = s.d_model
    out = [("tok_emb", (s.vocab, d)), ("pos_emb", (s.max_pos, d))]
    for l in range(s.n_layers):
        out += [(f"layers.{l}.{n}", sh) for n, sh in layer_tensor_shapes(s)]
    out += [("lnf_g", (d,)), ("lnf_b", (d,))]
    return out


def drafter_tensor_shapes(s: ModelShape):
    """(name, shape) in blob order for the parallel drafter."""
    d = s.d_model
    out = [("fuse_w", (d, s.n_hist * d)), ("lnh_g", (d,)), ("lnh_b", (d,)),
           ("mask_emb", (d,)), ("lnf_g", (d,)), ("lnf_b", (d,))]
    for l in range(s.drafter_layers):
        out += [(f"layers.{l}.{n}", sh) for n, sh in layer_tensor_shapes(s)]
    return out


# ---------------------------------------------------------------- rounding

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest-even bf16 value, returned as float32 (input formatting).
    Finite inputs only (uint32 arithmetic cannot overflow below the NaN range)."""
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    r = (u >> 16) & 1
    r += 0x7FFF
    u += r
    u &= np.uint32(0xFFFF0000)
    return u.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16-representable float32 array -> uint16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------- drawing

def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _draw(name: str, shape, seed: int, salt: int) -> np.ndarray:
    """One tensor: N(0, 0.02) for weights/biases, 1 + N(0, 0.02) for LN gains."""
    tag = sum((i + 1) * ord(c) for i, c in enumerate(name)) & 0x7FFFFFFF
    g = _rng(seed, salt, tag, len(name))
    a = g.standard_normal(size=shape, dtype=np.float32) * np.float32(0.02)
    if name.endswith("_g"):
        a += np.float32(1.0)
    return a


def _fmt(a: np.ndarray, dtype: str) -> np.ndarray:
    return round_to_bf16(a) if dtype == "bf16" else a.astype(np.float32, copy=False)


def drafter_weights(s: ModelShape, seed: int, target: dict | None = None) -> dict:
    """Drafter tensors.  Its two layers are copies of target layers 0 and 1
    (Whisper-Flash §3.2: the drafter is initialised from Whisper's first two
    decoder blocks) and its final LN is a copy of the target's; the fusion
    projection and the mask vector are fresh N(0, 0.02) draws."""
    if target is None:
        target = target_weights(s, seed)
    out = {}
    for n, sh in drafter_tensor_shapes(s):
        if n.startswith("layers."):
            out[n] = target[n].copy()
        elif n in ("lnf_g", "lnf_b"):
            out[n] = target[n].copy()
        else:
            out[n] = _fmt(_draw(n, sh, seed, 2), s.dtype)
    return out


def pack_blob(tensors: dict, order) -> np.ndarray:
    """Concatenate tensors in blob order into one flat array (f32 or bf16 bits)."""
    parts = [np.ascontiguousarray(tensors[n]).reshape(-1) for n, _ in order]
    return np.concatenate(parts)


def _threads():
    import os
    return max(1, min(16, os.cpu_count() or 1))


def target_weights(s: ModelShape, seed: int) -> dict:
    """All target tensors (float32 arrays, bf16-valued for bf16 shapes)."""
    from concurrent.futures import ThreadPoolExecutor
    shapes = target_tensor_shapes(s)
    with ThreadPoolExecutor(_threads()) as ex:
        arrs = list(ex.map(lambda ns: _fmt(_draw(ns[0], ns[1], seed, 1), s.dtype), shapes))
    return {n: a for (n, _), a in zip(shapes, arrs)}


def blob_from(tensors: dict, order, dtype: str) -> np.ndarray:
    """Serialise tensors in blob order: uint16 bf16 bits or float32, one flat array."""
    total = sum(int(np.prod(sh)) for _, sh in order)
    out = np.empty(total, dtype=np.uint16 if dtype == "bf16" else np.float32)
    offs, off = [], 0
    for n, sh in order:
        offs.append(off)
        off += int(np.prod(sh))
    from concurrent.futures import ThreadPoolExecutor

    def put(i):
        n, sh = order[i]
        a = np.ascontiguousarray(tensors[n], dtype=np.float32).reshape(-1)
        dst = out[offs[i]:offs[i] + a.size]
        if dtype == "bf16":
            np.right_shift(a.view(np.uint32), 16, out=dst, casting="unsafe")
        else:
            dst[:] = a
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(put, range(len(order))))
    return out


def encode_blob(flat_f32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits(flat_f32)
    return np.ascontiguousarray(flat_f32, dtype=np.float32)


def encoder_states(s: ModelShape, seed: int, request: int, frames: int = 1500) -> np.ndarray:
    """A = E(x) stand-in: [frames, d] ~ N(0, 1), seeded per request."""
    g = _rng(seed + 1000 + request, 3)
    a = g.standard_normal(size=(frames, s.d_model), dtype=np.float32)
    return _fmt(a, s.dtype)


# ---------------------------------------------------------------- audio encoder

@dataclass(frozen=True)
class EncoderShape:
    """Whisper audio encoder: a two-convolution stem over 2 * n_frames mel
    frames, n_layers pre-LN transformer blocks over n_frames positions."""
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    d_ff: int
    n_mels: int
    n_frames: int = 1500
    dtype: str = "bf16"


ENC_LARGE_V3 = EncoderShape("large-v3-encoder", 32, 1280, 20, 5120, 128)
ENC_TINY = EncoderShape("tiny-encoder", 4, 384, 6, 1536, 80)

ENC_LAYER = ("ln1_g", "ln1_b", "w_qkv", "b_q", "b_v", "w_o", "b_o", "ln2_g", "ln2_b",
             "w_fc1", "b_fc1", "w_fc2", "b_fc2")


def encoder_tensor_shapes(e: EncoderShape):
    """(name, shape) in blob order for the audio encoder:
    conv1_w[d, n_mels, 3], conv1_b[d], conv2_w[d, d, 3], conv2_b[d],
    layer 0..n-1 (ENC_LAYER order; w_qkv rows q|k|v, no key bias),
    lnp_g[d], lnp_b[d] (the final layer norm)."""
    d, f = e.d_model, e.d_ff
    shp = {"w_qkv": (3 * d, d), "w_o": (d, d), "w_fc1": (f, d), "w_fc2": (d, f), "b_fc1": (f,)}
    out = [("conv1_w", (d, e.n_mels, 3)), ("conv1_b", (d,)), ("conv2_w", (d, d, 3)), ("conv2_b", (d,))]
    for l in range(e.n_layers):
        out += [(f"layers.{l}.{n}", shp.get(n, (d,))) for n in ENC_LAYER]
    out += [("lnp_g", (d,)), ("lnp_b", (d,))]
    return out


def encoder_weights(e: EncoderShape, seed: int) -> dict:
    """All encoder tensors, N(0, 0.02) (LN gains 1 + N(0, 0.02)), bf16-valued
    for bf16 shapes."""
    from concurrent.futures import ThreadPoolExecutor
    shapes = encoder_tensor_shapes(e)
    with ThreadPoolExecutor(_threads()) as ex:
        arrs = list(ex.map(lambda ns: _fmt(_draw(ns[0], ns[1], seed, 4), e.dtype), shapes))
    return {n: a for (n, _), a in zip(shapes, arrs)}


def mel_input(e: EncoderShape, seed: int, request: int) -> np.ndarray:
    """Log-mel stand-in [n_mels, 2 * n_frames] ~ 0.5 N(0, 1) (normalised
    Whisper features lie within about +-1.5), seeded per request."""
    g = _rng(seed + 2000 + request, 5)
    a = g.standard_normal(size=(e.n_mels, 2 * e.n_frames), dtype=np.float32) * np.float32(0.5)
    return _fmt(a, e.dtype)


# ---------------------------------------------------------------- workloads

@dataclass
class DraftCorruption:
    """Synthetic drafts from a reference trajectory.

    For an anchor at absolute position t and candidate j (1..K) the draft is
    traj[t + j] unless mask[t, j-1] is set, in which case it is tok[t, j-1]
    (uniform over the vocabulary).  Each (request, t, j) has its own draw, so
    proposals are independent across rounds.
    """
    mask: np.ndarray     # [n_req, max_pos, K] uint8
    tok: np.ndarray      # [n_req, max_pos, K] int32


def corruption_plan(n_req: int, max_pos: int, K: int, p: np.ndarray, vocab: int,
                    seed: int) -> DraftCorruption:
    p = np.asarray(p, dtype=np.float64).reshape(1, 1, K)
    g = _rng(seed, 4, n_req, max_pos, K)
    u = g.random(size=(n_req, max_pos, K))
    tok = g.integers(0, vocab, size=(n_req, max_pos, K), dtype=np.int64).astype(np.int32)
    return DraftCorruption((u < p).astype(np.uint8), tok)


def corruption_p_const(K: int, p: float) -> np.ndarray:
    return np.full(K, p)


def corruption_p_linear(K: int, p_first: float = 0.1, p_last: float = 0.5) -> np.ndarray:
    """p_j grows linearly from p_first at j=1 to p_last at j=K."""
    return np.array([p_first + (p_last - p_first) * (j / (K - 1)) for j in range(K)])


def budgets_uniform(n_req: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Transcript lengths drawn uniformly from [lo, hi]."""
    return _rng(seed, 5, n_req).integers(lo, hi + 1, size=n_req).astype(np.int32)


def varlen_frames_and_budgets(n_req: int, seed: int, f_lo: int = 250, f_hi: int = 1500,
                              frames_full: int = 1500, tok_full: int = 200):
    """Valid frame counts F ~ U{f_lo..f_hi} and lengths round(F/1500*200 * s),
    s ~ U[0.8, 1.2] (the +-20 % spread)."""
    g = _rng(seed, 6, n_req)
    F = g.integers(f_lo, f_hi + 1, size=n_req).astype(np.int32)
    sc = g.uniform(0.8, 1.2, size=n_req)
    n = np.floor(F / frames_full * tok_full * sc + 0.5).astype(np.int32)
    return F, np.maximum(n, 1)


def gaussian_noise(shape, seed: int) -> np.ndarray:
    """N(0, 1) noise, used to build the drafter logits of the sampling study."""
    return _rng(seed, 7).standard_normal(size=shape, dtype=np.float32)


def random_tokens(n: int, vocab: int, seed: int) -> np.ndarray:
    return _rng(seed, 8, n).integers(0, vocab, size=n).astype(np.int32)
