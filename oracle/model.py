"""CPU oracle for speculative Whisper decoding — TEST INFRASTRUCTURE ONLY.

Only tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding)
never does, and this package never imports the product path: the two share
no code, only the seeded inputs from ``synth``.

It is a plain, slow numpy implementation in float64 of what the decoding
path computes, written from the pages:

  * Whisper-Flash: Acoustically Conditioned Parallel Drafting for Faster
    Whisper Decoding (arXiv 2609.32869), §3.1 (propose / verify / advance,
    Eq. 1, the rejection rule), §3.2 (drafter input Eq. 2, history and
    acoustic memories), Appendix A.1 (anchor, cache, budget), A.2 (drafter
    architecture, RoPE), A.4 (sampling in FP32), A.5 (per-request acoustic
    K/V).
  * The target is a standard pre-LN Whisper decoder (token + learned position
    embedding; per layer causal self-attention, cross-attention over the
    encoder states, GELU FFN; final LN; LM head tied to the token embedding).

Numeric modes
  bf16=False : pure float64 (the fp32 model shape is compared against this).
  bf16=True  : the same float64 arithmetic, but values are rounded to bf16
               (through float32, nearest-even) at the points where the bf16
               model stores them: layer-norm outputs, q/k/v, the self and
               cross K/V caches, attention outputs, GELU outputs, the history
               features fed to the fusion projection, the fused history
               state.  The residual stream, logits, softmax and every
               accumulation stay wide.

Readings taken where the pages are silent (each also listed in the design
notes): LN eps 1e-5; exact-erf GELU; no bias on k (self and cross); scores
scaled by 1/sqrt(d_head); RoPE on drafter q/k only, interleaved pairs
(2i, 2i+1), theta_i = 10000^(-2i/d_head) rounded to fp32, phase
fp32(pos * theta_i); history feature h = LN_h(W_f concat(resid)) with no
further LN before the drafter's K/V projections; the drafter's mask rows get
no absolute position embedding; argmax ties go to the lowest token id.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
from scipy.special import erf

from . import philox

LN_EPS = 1e-5


# ------------------------------------------------------------------ helpers

def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 -> bf16 (round to nearest even), returned as float64."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def layer_norm(x: np.ndarray, g: np.ndarray, b: np.ndarray) -> np.ndarray:
    """LayerNorm over the last axis with biased variance and eps 1e-5."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + LN_EPS) * g + b


def gelu(x: np.ndarray) -> np.ndarray:
    """GELU with the exact Gaussian CDF: x * Phi(x)."""
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=axis, keepdims=True)


def rope_theta(d_head: int) -> np.ndarray:
    """Per-pair inverse frequencies theta_i = 10000^(-2i/d_head), as fp32 values."""
    i = np.arange(d_head // 2, dtype=np.float64)
    return (10000.0 ** (-2.0 * i / d_head)).astype(np.float32)


def rope(x: np.ndarray, pos: np.ndarray, n_heads: int) -> np.ndarray:
    """Rotary position embedding (RoFormer) on rows x[r] at absolute text
    positions pos[r]; pairs (2i, 2i+1) inside each head rotate by
    fp32(pos * theta_i) (Whisper-Flash Appendix A.2: base 10,000, FP32 phases,
    explicit text positions)."""
    R, d = x.shape
    dh = d // n_heads
    th = rope_theta(dh)                                              # [dh/2] fp32
    ang = (np.asarray(pos, dtype=np.float32)[:, None] * th[None, :]).astype(np.float32)
    c = np.cos(ang.astype(np.float64))[:, None, :]                   # [R,1,dh/2]
    s = np.sin(ang.astype(np.float64))[:, None, :]
    xr = x.reshape(R, n_heads, dh // 2, 2)
    x0, x1 = xr[..., 0], xr[..., 1]
    out = np.empty_like(xr)
    out[..., 0] = x0 * c - x1 * s
    out[..., 1] = x0 * s + x1 * c
    return out.reshape(R, d)


def mha(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_heads: int,
        mask: np.ndarray | None = None) -> np.ndarray:
    """Scaled dot-product attention, per head.  q [R,d], k/v [S,d],
    mask [R,S] boolean (True = key visible) or None."""
    R, d = q.shape
    S = k.shape[0]
    dh = d // n_heads
    qh = q.reshape(R, n_heads, dh).transpose(1, 0, 2)
    kh = k.reshape(S, n_heads, dh).transpose(1, 0, 2)
    vh = v.reshape(S, n_heads, dh).transpose(1, 0, 2)
    s = np.einsum("hrd,hsd->hrs", qh, kh) / math.sqrt(dh)
    if mask is not None:
        s = np.where(mask[None, :, :], s, -np.inf)
    p = softmax(s, axis=-1)
    o = np.einsum("hrs,hsd->hrd", p, vh)
    return o.transpose(1, 0, 2).reshape(R, d)


def argmax_lowest(z: np.ndarray) -> int:
    """Greedy choice (Eq. 1); np.argmax returns the first (lowest-id) maximum."""
    return int(np.argmax(z))


def top2_margin(z: np.ndarray) -> float:
    t = np.partition(z, -2)[-2:]
    return float(t[1] - t[0])


# ------------------------------------------------------------------ model

@dataclass
class Request:
    """Per-request decoder state (Appendix A.1: before a round with anchor at
    position t the caches hold exactly the positions before t)."""
    frames: int
    ck: list            # target cross K per layer [F, d]
    cv: list
    dck: list           # drafter cross K per drafter layer [F, d]
    dcv: list
    sk: list            # target self K cache per layer [max_pos, d]
    sv: list
    hist: np.ndarray    # residual streams at the history layers [max_pos, n_hist, d]
    L: int = 0          # target cache length
    peaks: list = field(default_factory=list)   # readout: per block row, the head-averaged attention peak frame
    center: int = -1    # centre of the drafter's cross-attention window (-1: no window yet)


class Oracle:
    def __init__(self, shape, target: dict, drafter: dict | None = None, bf16: bool | None = None):
        self.s = shape
        self.bf16 = (shape.dtype == "bf16") if bf16 is None else bf16
        f64 = lambda a: np.asarray(a, dtype=np.float64)
        self.t = {k: f64(v) for k, v in target.items()}
        self.dr = {k: f64(v) for k, v in drafter.items()} if drafter is not None else None
        self.d = shape.d_model
        self.H = shape.n_heads

    # storage-point rounding
    def rb(self, x):
        return round_bf16(x) if self.bf16 else x

    # ---------------------------------------------------- acoustic K/V (A.5)
    def cross_kv_layer(self, A: np.ndarray, w: dict, pre: str):
        """K_c = A W_k^T, V_c = A W_v^T + b_v for one layer's cross-attention."""
        d = self.d
        wkv = w[pre + "w_kvc"]
        Ad = np.asarray(A, dtype=np.float64)
        k = self.rb(Ad @ wkv[:d].T)
        v = self.rb(Ad @ wkv[d:].T + w[pre + "b_vc"])
        return k, v

    def new_request(self, A: np.ndarray, frames: int | None = None) -> Request:
        """Set up one request: refresh the acoustic K/V of target and drafter
        from its encoder states (Appendix A.5).  Frames >= `frames` are masked."""
        F = A.shape[0] if frames is None else frames
        A = A[:F]
        ck, cv, dck, dcv = [], [], [], []
        for l in range(self.s.n_layers):
            k, v = self.cross_kv_layer(A, self.t, f"layers.{l}.")
            ck.append(k); cv.append(v)
        if self.dr is not None:
            for l in range(self.s.drafter_layers):
                k, v = self.cross_kv_layer(A, self.dr, f"layers.{l}.")
                dck.append(k); dcv.append(v)
        P, d = self.s.max_pos, self.d
        return Request(F, ck, cv, dck, dcv,
                       [np.zeros((P, d)) for _ in range(self.s.n_layers)],
                       [np.zeros((P, d)) for _ in range(self.s.n_layers)],
                       np.zeros((P, self.s.n_hist, d)))

    # ---------------------------------------------------- verification-attention readout
    def attention_peaks(self, qc: np.ndarray, ck: np.ndarray) -> list:
        """Alignment Drift §5 / App. D.2: the target's audio attention of each
        query row at one layer, averaged over heads (softmax per head of
        q k^T / sqrt(d_head) over the valid frames), and its peak frame
        (lowest frame on ties)."""
        R, d = qc.shape
        dh = d // self.H
        qh = qc.reshape(R, self.H, dh).transpose(1, 0, 2)
        kh = ck.reshape(ck.shape[0], self.H, dh).transpose(1, 0, 2)
        p = softmax(np.einsum("hrd,hsd->hrs", qh, kh) / math.sqrt(dh), axis=-1)
        return [int(np.argmax(row)) for row in p.mean(axis=0)]

    # ---------------------------------------------------- target decoder
    def _layer(self, x, l, q_rows_attend, ck, cv, readout=None):
        """One pre-LN decoder layer.  `q_rows_attend(q, k, v)` does the
        self-attention (cached or full)."""
        w, p, d = self.t, f"layers.{l}.", self.d
        h = self.rb(layer_norm(x, w[p + "ln1_g"], w[p + "ln1_b"]))
        qkv = h @ w[p + "w_qkv"].T
        q = self.rb(qkv[:, :d] + w[p + "b_q"])
        k = self.rb(qkv[:, d:2 * d])
        v = self.rb(qkv[:, 2 * d:] + w[p + "b_v"])
        o = self.rb(q_rows_attend(l, q, k, v))
        x = x + (o @ w[p + "w_o"].T + w[p + "b_o"])
        h2 = self.rb(layer_norm(x, w[p + "ln2_g"], w[p + "ln2_b"]))
        qc = self.rb(h2 @ w[p + "w_qc"].T + w[p + "b_qc"])
        if readout is not None:
            readout.extend(self.attention_peaks(qc, ck))
        oc = self.rb(mha(qc, ck, cv, self.H))
        x = x + (oc @ w[p + "w_oc"].T + w[p + "b_oc"])
        h3 = self.rb(layer_norm(x, w[p + "ln3_g"], w[p + "ln3_b"]))
        f = self.rb(gelu(h3 @ w[p + "w_fc1"].T + w[p + "b_fc1"]))
        x = x + (f @ w[p + "w_fc2"].T + w[p + "b_fc2"])
        return x

    def _head(self, x):
        hf = self.rb(layer_norm(x, self.t["lnf_g"], self.t["lnf_b"]))
        return hf @ self.t["tok_emb"].T

    def _embed(self, tokens, pos):
        return self.t["tok_emb"][np.asarray(tokens)] + self.t["pos_emb"][np.asarray(pos)]

    def forward_full(self, req: Request, tokens) -> tuple[np.ndarray, np.ndarray]:
        """The plain definition: the whole sequence at positions 0..n-1 in one
        pass with a causal mask and no cache.  Returns logits [n, V] and the
        residual streams at the history layers [n, n_hist, d]."""
        n = len(tokens)
        pos = np.arange(n)
        x = self._embed(tokens, pos)
        causal = np.tril(np.ones((n, n), dtype=bool))
        hist = []

        def attend(l, q, k, v):
            return mha(q, k, v, self.H, causal)

        for l in range(self.s.n_layers):
            x = self._layer(x, l, attend, req.ck[l][:req.frames], req.cv[l][:req.frames])
            if l in self.s.hist_layers:
                hist.append(x.copy())
        return self._head(x), np.stack(hist, axis=1)

    def verify(self, req: Request, block, readout_layer: int | None = None) -> np.ndarray:
        """One causal target pass over the block [anchor, candidates...] at
        positions L..L+H-1 (Whisper-Flash §3.1).  Writes the block's K/V into
        the cache and its history-layer residuals into req.hist; does not
        move L (rollback / advance is the acceptor's job).  Returns logits [H, V]."""
        H = len(block)
        pos = req.L + np.arange(H)
        assert pos[-1] < self.s.max_pos, "position beyond the decoder context"
        x = self._embed(block, pos)
        hist = []

        def attend(l, q, k, v):
            req.sk[l][pos] = k
            req.sv[l][pos] = v
            last = pos[-1] + 1
            vis = np.arange(last)[None, :] <= pos[:, None]
            return mha(q, req.sk[l][:last], req.sv[l][:last], self.H, vis)

        peaks = []
        for l in range(self.s.n_layers):
            x = self._layer(x, l, attend, req.ck[l][:req.frames], req.cv[l][:req.frames],
                            peaks if l == readout_layer else None)
            if l in self.s.hist_layers:
                hist.append(x.copy())
        req.hist[pos] = np.stack(hist, axis=1)
        req.peaks = peaks
        return self._head(x)

    # ---------------------------------------------------- tree verification (Alignment Drift App. E.3)
    def verify_tree(self, req: Request, tokens, parent) -> np.ndarray:
        """One target pass over a candidate tree: node j (0 = the anchor, the
        root; parent[j] < j) sits at position L + depth(j) and attends to the
        cache positions before L and to its own ancestors (itself included) --
        a tree attention mask.  Node j's keys and values are stored at cache
        slot L + j until acceptance commits a path.  Returns logits [N, V]."""
        N = len(tokens)
        depth = [0] * N
        anc = [[j] for j in range(N)]
        for j in range(1, N):
            depth[j] = depth[parent[j]] + 1
            anc[j] = anc[parent[j]] + [j]
        L = req.L
        assert L + N <= self.s.max_pos, "tree beyond the decoder context"
        x = self._embed(tokens, L + np.asarray(depth))
        vis = np.zeros((N, L + N), dtype=bool)
        vis[:, :L] = True
        for j in range(N):
            vis[j, [L + m for m in anc[j]]] = True
        slots = L + np.arange(N)

        def attend(l, q, k, v):
            req.sk[l][slots] = k
            req.sv[l][slots] = v
            return mha(q, req.sk[l][:L + N], req.sv[l][:L + N], self.H, vis)

        hist = []
        for l in range(self.s.n_layers):
            x = self._layer(x, l, attend, req.ck[l][:req.frames], req.cv[l][:req.frames])
            if l in self.s.hist_layers:
                hist.append(x.copy())
        req.hist[slots] = np.stack(hist, axis=1)
        return self._head(x)

    def commit_path(self, req: Request, path) -> None:
        """Move the accepted path's keys, values and history rows from their
        node slots L + path[j] to positions L + j."""
        L = req.L
        for j, node in enumerate(path):
            for l in range(self.s.n_layers):
                req.sk[l][L + j] = req.sk[l][L + node]
                req.sv[l][L + j] = req.sv[l][L + node]
            req.hist[L + j] = req.hist[L + node]

    # ---------------------------------------------------- drafter (§3.2, A.2)
    def history_features(self, resid: np.ndarray) -> np.ndarray:
        """History memory H_<t: the residual streams of the history layers,
        concatenated (n_hist*d) and projected to the drafter width, then
        LN_h.  resid [n, n_hist, d] -> h [n, d]."""
        dr = self.dr
        n = resid.shape[0]
        if n == 0:
            return np.zeros((0, self.d))
        feat = self.rb(resid.reshape(n, -1))
        return self.rb(layer_norm(feat @ dr["fuse_w"].T, dr["lnh_g"], dr["lnh_b"]))

    def drafter_layer(self, x, l: int, pos, h_hist, pos_hist, dck, dcv, window=None):
        """One drafter layer.  Block rows x [R, d] at RoPE positions `pos`;
        history features h_hist [S, d] at positions `pos_hist`.  The block's
        queries attend to [history ; block] in one softmax with no mask
        inside the block (Whisper-Flash §3.2, Appendix A.2); history keys are
        RoPE(W_k h) and values W_v h + b_v, with this layer's projections.
        Then cross-attention to the drafter's own acoustic K/V and the FFN."""
        dr, d, p = self.dr, self.d, f"layers.{l}."
        w = dr[p + "w_qkv"]
        hk = self.rb(rope(h_hist @ w[d:2 * d].T, pos_hist, self.H))
        hv = self.rb(h_hist @ w[2 * d:].T + dr[p + "b_v"])
        h = self.rb(layer_norm(x, dr[p + "ln1_g"], dr[p + "ln1_b"]))
        qkv = h @ w.T
        q = self.rb(rope(qkv[:, :d] + dr[p + "b_q"], pos, self.H))
        k = self.rb(rope(qkv[:, d:2 * d], pos, self.H))
        v = self.rb(qkv[:, 2 * d:] + dr[p + "b_v"])
        o = self.rb(mha(q, np.concatenate([hk, k]), np.concatenate([hv, v]), self.H))
        x = x + (o @ dr[p + "w_o"].T + dr[p + "b_o"])
        h2 = self.rb(layer_norm(x, dr[p + "ln2_g"], dr[p + "ln2_b"]))
        qc = self.rb(h2 @ dr[p + "w_qc"].T + dr[p + "b_qc"])
        vis = None
        if window is not None:            # windowed cross-attention: frames lo <= f < hi only
            f = np.arange(dck.shape[0])
            vis = np.broadcast_to(((f >= window[0]) & (f < window[1]))[None, :], (qc.shape[0], dck.shape[0]))
        oc = self.rb(mha(qc, dck, dcv, self.H, vis))
        x = x + (oc @ dr[p + "w_oc"].T + dr[p + "b_oc"])
        h3 = self.rb(layer_norm(x, dr[p + "ln3_g"], dr[p + "ln3_b"]))
        f = self.rb(gelu(h3 @ dr[p + "w_fc1"].T + dr[p + "b_fc1"]))
        return x + (f @ dr[p + "w_fc2"].T + dr[p + "b_fc2"])

    def draft_logits(self, req: Request, anchor: int, half_width: int = 0) -> np.ndarray:
        """Drafter forward for the anchor at position t = L: input
        X_t = [Emb(y_t), m, ..., m] (Eq. 2) at RoPE positions t..t+K, history =
        accepted positions < t (never at or beyond the anchor, Appendix A.2).
        Returns the logits of the K mask rows [K, V] (the anchor row's output
        is not a proposal).  half_width > 0: the drafter's cross-attention sees
        only the frames within half_width of req.center (Alignment Drift App.
        A.2, a fixed-width window; ±400 ms is ±20 Whisper frames), clipped to
        the valid frames."""
        dr, K = self.dr, self.s.K
        t = req.L
        pos = t + np.arange(K + 1)
        x = np.concatenate([self.t["tok_emb"][[anchor]], np.repeat(dr["mask_emb"][None, :], K, 0)])
        h_hist = self.history_features(req.hist[:t])
        window = None
        if half_width > 0 and req.center >= 0:
            window = (max(0, req.center - half_width), min(req.frames, req.center + half_width + 1))
        for l in range(self.s.drafter_layers):
            x = self.drafter_layer(x, l, pos, h_hist, np.arange(t),
                                   req.dck[l][:req.frames], req.dcv[l][:req.frames], window)
        hf = self.rb(layer_norm(x[1:], dr["lnf_g"], dr["lnf_b"]))
        return hf @ self.t["tok_emb"].T


# ------------------------------------------------------------------ acceptance

@dataclass
class Accepted:
    a: int              # accepted candidates
    emitted: list       # tokens appended to the transcript this round
    next_anchor: int
    done: bool
    margins: list = field(default_factory=list)   # sampling: decision margin per emitted token


def accept_greedy(block, n_prop: int, g, budget: int, eos: int) -> Accepted:
    """Greedy verification (Whisper-Flash §3.1, Appendix A.1): keep candidates
    while they equal the target's argmax at the previous position; emit the
    target's token at the first disagreement, or the bonus token after all
    n_prop agree.  An accepted EOS ends the transcript with no bonus.
    `g[i]` is the target argmax of block row i."""
    a, out = 0, []
    for j in range(1, n_prop + 1):
        if int(block[j]) != int(g[j - 1]):
            break
        a += 1
        out.append(int(block[j]))
        if int(block[j]) == eos:
            return Accepted(a, out, int(block[j]), True)
    out.append(int(g[a]))
    return Accepted(a, out, int(g[a]), out[-1] == eos or len(out) >= budget)


def accept_tree(tokens, parent, g, budget: int, eos: int):
    """Greedy acceptance on a candidate tree: from the root, move to the
    child whose token equals the target's argmax at the current node, while
    one exists (at most budget - 1 candidates); emit the accepted tokens and
    the target's token at the last accepted node (none after an accepted
    EOS).  Returns (Accepted, path of node indices from the root)."""
    children = {}
    for j in range(1, len(tokens)):
        children.setdefault(parent[j], []).append(j)
    cur, path, out = 0, [0], []
    while len(out) < budget - 1:
        nxt = [c for c in children.get(cur, []) if int(tokens[c]) == int(g[cur])]
        if not nxt:
            break
        cur = nxt[0]
        path.append(cur)
        out.append(int(tokens[cur]))
        if int(tokens[cur]) == eos:
            return Accepted(len(out), out, int(tokens[cur]), True), path
    out.append(int(g[cur]))
    a = len(path) - 1
    return Accepted(a, out, int(g[cur]), out[-1] == eos or len(out) >= budget), path


def tree_tokens(q_logits, parent, rank, anchor: int) -> list:
    """Candidate tokens of a fixed tree from the parallel drafter: node j at
    depth k takes the rank[j]-th most likely token of mask row k (rank 0 =
    argmax; equal logits rank the lower id first); node 0 is the anchor."""
    out = [int(anchor)]
    depth = [0] * len(parent)
    for j in range(1, len(parent)):
        depth[j] = depth[parent[j]] + 1
        row = np.asarray(q_logits[depth[j] - 1])
        order = np.lexsort((np.arange(len(row)), -row))
        out.append(int(order[rank[j]]))
    return out


def speculative_greedy_tree(orc: Oracle, req: Request, budget: int, parent, rank, log=None) -> DecodeResult:
    """Propose / verify / advance with a candidate tree (Alignment Drift
    App. E.3): the drafter's ranked tokens fill a fixed tree, the target
    verifies every node in one pass under the tree mask, the longest
    matching root path is accepted and committed to the cache.  Rows that
    would pass the decoder's last position are left out (the tree's first
    rows form a tree).  log: per round (drafter logits, tokens, target
    logits, path) appended when given."""
    eos = orc.s.eos_id
    acc, logits = prefill(orc, req, budget)
    out = list(acc.emitted)
    res = DecodeResult(out, margins=[top2_margin(logits[-1])])
    done, anchor = acc.done, acc.next_anchor
    while not done:
        R = budget - len(out)
        n = min(len(parent), orc.s.max_pos - req.L)
        q = orc.draft_logits(req, anchor)
        toks = tree_tokens(q, parent[:n], rank[:n], anchor)
        lg = orc.verify_tree(req, toks, parent[:n])
        g = [argmax_lowest(z) for z in lg]
        acc, path = accept_tree(toks, parent[:n], g, R, eos)
        if log is not None:
            log.append((q, toks, lg, path))
        orc.commit_path(req, path)
        req.L += 1 + acc.a
        out += acc.emitted
        res.rounds += 1
        res.accepted.append(acc.a)
        res.proposed.append(len(toks) - 1)
        res.emitted.append(len(acc.emitted))
        done, anchor = acc.done, acc.next_anchor
    return res


def accept_forced(n_prop: int, g, budget: int, eos: int) -> Accepted:
    """Teacher-forced block (the prompt prefill of Appendix A.1): every block
    token is given, the target's argmax after the last one is emitted."""
    tok = int(g[n_prop])
    return Accepted(n_prop, [tok], tok, tok == eos or budget <= 1)


def probs_fp32(z: np.ndarray, T: float, suppress=None) -> np.ndarray:
    """softmax(z / T) in float32 (Appendix A.4: softmax and acceptance
    probabilities in FP32), suppressed ids set to probability 0."""
    z = np.asarray(z, dtype=np.float32) / np.float32(T)
    if suppress is not None and len(suppress):
        z = z.copy()
        z[np.asarray(suppress)] = -np.inf
    m = np.max(z)
    e = np.exp(z - m, dtype=np.float32)
    return (e / np.sum(e, dtype=np.float32)).astype(np.float32)


def sample_inverse_cdf(w: np.ndarray, u: float) -> int:
    """Smallest id v with cumsum(w)[v] > u * sum(w) (ids in ascending order)."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    tgt = float(u) * c[-1]
    v = int(np.searchsorted(c, tgt, side="right"))
    if v >= len(c):
        v = int(np.nonzero(w > 0)[0][-1])
    return v


def cdf_margin(w: np.ndarray, u: float) -> float:
    """How far u * sum(w) lies from the nearest boundary of the inverse-CDF
    draw, as a fraction of sum(w): the size of a perturbation of the weights
    that could change the drawn id."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    t = float(u) * c[-1]
    v = min(int(np.searchsorted(c, t, side="right")), len(c) - 1)
    lo = c[v - 1] if v > 0 else 0.0
    return float(min(t - lo, c[v] - t) / c[-1])


def accept_sampling(block, n_prop: int, p_logits, q_logits, T: float, seed: int, slot: int,
                    rnd: int, budget: int, eos: int, suppress=None, uniform=None, cand_margins=None):
    """Rejection rule with per-token decision margins: `cand_margins[j-1]` is
    the margin of the draw that produced candidate j (if known); the margin
    of an emitted token is the smallest margin among the decisions that led
    to it."""
    acc, det = _accept_sampling(block, n_prop, p_logits, q_logits, T, seed, slot, rnd, budget, eos, suppress,
                                uniform)
    # (acceptance margin, inverse-CDF margin) of the decision chain so far
    ca, cc = float("inf"), float("inf")
    margins = []
    for d in det:
        if d[0] == "accept":
            _, j, u, qv, pv, ok = d
            ca = min(ca, abs(u * qv - pv) / max(pv, 1e-30))
            if cand_margins is not None:
                cc = min(cc, cand_margins[j - 1])
            if ok:
                margins.append((ca, cc))
        else:
            _, j, u2, tok = d
            if d[0] == "residual":
                p = probs_fp32(p_logits[j - 1], T, suppress)
                q = probs_fp32(q_logits[j - 1], T, suppress)
                w = np.maximum(p - q, np.float32(0))
                w = w if np.any(w > 0) else p
            else:
                w = probs_fp32(p_logits[j - 1], T, suppress)
            margins.append((ca, min(cc, cdf_margin(w, u2))))
    acc.margins = margins
    return acc, det


def _accept_sampling(block, n_prop: int, p_logits, q_logits, T: float, seed: int, slot: int,
                     rnd: int, budget: int, eos: int, suppress=None, uniform=None):
    """Speculative rejection rule (Whisper-Flash §3.1; Leviathan et al.,
    Chen et al.): candidate j is accepted iff u_j * q_j(y_j) < p_j(y_j)
    (probability min(1, p/q)); at the first rejection a token is drawn from
    the normalised residual (p_j - q_j)_+; after a fully accepted block the
    bonus is drawn from p_{n+1}.  p_j is the target row j-1, q_j the draft
    row j-1.  `uniform(j, purpose)` overrides the Philox uniforms (tests).
    Returns (Accepted, detail) where detail records the decisions."""
    if uniform is None:
        uniform = lambda j, purpose: philox.uniform(seed, slot, rnd, j, purpose)
    a, out, detail = 0, [], []
    for j in range(1, n_prop + 1):
        y = int(block[j])
        p = probs_fp32(p_logits[j - 1], T, suppress)
        q = probs_fp32(q_logits[j - 1], T, suppress)
        u = uniform(j, philox.PURPOSE_ACCEPT)
        acc = bool(np.float32(u) * q[y] < p[y])
        detail.append(("accept", j, float(u), float(q[y]), float(p[y]), acc))
        if acc:
            a += 1
            out.append(y)
            if y == eos:
                return Accepted(a, out, y, True), detail
            continue
        r = np.maximum(p - q, np.float32(0)).astype(np.float32)
        if not np.any(r > 0):
            r = p
        u2 = uniform(j, philox.PURPOSE_RESIDUAL)
        tok = sample_inverse_cdf(r, u2)
        detail.append(("residual", j, float(u2), tok))
        out.append(tok)
        return Accepted(a, out, tok, tok == eos or len(out) >= budget), detail
    p = probs_fp32(p_logits[n_prop], T, suppress)
    u2 = uniform(n_prop + 1, philox.PURPOSE_RESIDUAL)
    tok = sample_inverse_cdf(p, u2)
    detail.append(("bonus", n_prop + 1, float(u2), tok))
    out.append(tok)
    return Accepted(a, out, tok, tok == eos or len(out) >= budget), detail


def sample_draft(q_logits_row, T: float, seed: int, slot: int, rnd: int, j: int, suppress=None) -> int:
    """Each mask position is sampled independently from its draft
    distribution (Appendix A.4)."""
    q = probs_fp32(q_logits_row, T, suppress)
    return sample_inverse_cdf(q, philox.uniform(seed, slot, rnd, j, philox.PURPOSE_DRAFT))


# ------------------------------------------------------------------ decoding loops

@dataclass
class DecodeResult:
    tokens: list                     # emitted transcript (prompt excluded)
    rounds: int = 0                  # target calls after prefill
    accepted: list = field(default_factory=list)   # a per round
    proposed: list = field(default_factory=list)   # n_prop per round
    margins: list = field(default_factory=list)    # oracle top-2 margin per emitted greedy token
    emitted: list = field(default_factory=list)    # tokens emitted per round


def greedy_plain(orc: Oracle, req: Request, budget: int) -> DecodeResult:
    """Eq. 1 taken literally: every new token is the argmax of a full
    uncached forward over prompt + transcript so far."""
    seq = list(orc.s.prompt)
    out = []
    margins = []
    while len(out) < budget:
        logits, _ = orc.forward_full(req, seq)
        z = logits[-1]
        tok = argmax_lowest(z)
        margins.append(top2_margin(z))
        out.append(tok)
        seq.append(tok)
        if tok == orc.s.eos_id:
            break
    return DecodeResult(out, rounds=len(out), margins=margins)


def prefill(orc: Oracle, req: Request, budget: int, T: float = 0.0, seed: int = 0, slot: int = 0):
    """Prompt pass: processes the prompt and emits the first transcript token,
    which becomes the first anchor (Appendix A.1).  With T > 0 that token is
    drawn from softmax(z/T) of the last prompt row (counter (slot, 0, n, 2))."""
    prompt = list(orc.s.prompt)
    logits = orc.verify(req, prompt)
    g = [argmax_lowest(z) for z in logits]
    n_prop = len(prompt) - 1
    margin = top2_margin(logits[n_prop])
    if T > 0:
        u = philox.uniform(seed, slot, 0, n_prop + 1, philox.PURPOSE_RESIDUAL)
        p = probs_fp32(logits[n_prop], T)
        g[n_prop] = sample_inverse_cdf(p, u)
        margin = (float("inf"), cdf_margin(p, u))
    acc = accept_forced(n_prop, g, budget, orc.s.eos_id)
    acc.margins = [margin]
    req.L += 1 + acc.a
    return acc, logits


def greedy_cached(orc: Oracle, req: Request, budget: int) -> DecodeResult:
    """Autoregressive greedy through the cached verify with blocks of height 1."""
    acc, logits = prefill(orc, req, budget)
    out = list(acc.emitted)
    margins = [top2_margin(logits[-1])]
    done, anchor, rounds = acc.done, acc.next_anchor, 0
    while not done:
        lg = orc.verify(req, [anchor])
        g = [argmax_lowest(lg[0])]
        margins.append(top2_margin(lg[0]))
        acc = accept_greedy([anchor], 0, g, budget - len(out), orc.s.eos_id)
        req.L += 1 + acc.a
        out += acc.emitted
        done, anchor = acc.done, acc.next_anchor
        rounds += 1
    return DecodeResult(out, rounds=rounds, margins=margins)


def speculative_greedy(orc: Oracle, req: Request, budget: int, propose) -> DecodeResult:
    """Propose / verify / advance (Whisper-Flash §3.1, Appendix A.1).
    `propose(req, anchor, t, n_prop) -> list of n_prop candidate ids`."""
    K, eos = orc.s.K, orc.s.eos_id
    acc, logits = prefill(orc, req, budget)
    out = list(acc.emitted)
    res = DecodeResult(out, margins=[top2_margin(logits[-1])])
    done, anchor = acc.done, acc.next_anchor
    while not done:
        R = budget - len(out)
        n_prop = min(K, R - 1)
        cand = list(propose(req, anchor, req.L, n_prop))[:n_prop] if n_prop > 0 else []
        block = [anchor] + cand
        lg = orc.verify(req, block)
        g = [argmax_lowest(z) for z in lg]
        acc = accept_greedy(block, n_prop, g, R, eos)
        res.margins += [top2_margin(lg[i]) for i in range(len(acc.emitted))]
        req.L += 1 + acc.a
        out += acc.emitted
        res.rounds += 1
        res.accepted.append(acc.a)
        res.proposed.append(n_prop)
        res.emitted.append(len(acc.emitted))
        done, anchor = acc.done, acc.next_anchor
    return res


def proposal_confidence(q_logits_row, tok: int, T: float, suppress=None) -> float:
    """Confidence of a drafted token: its probability under the drafter's own
    softmax (FP32, Appendix A.4), at temperature T when sampling, T = 1 for
    greedy proposals."""
    return float(probs_fp32(q_logits_row, T if T > 0 else 1.0, suppress)[int(tok)])


def limit_proposals(cand, q_logits, k_verify: int, threshold: float, T: float, R: int, suppress=None) -> int:
    """How many of the drafted candidates go to verification: truncated
    verification keeps only the first k_verify (Whisper-Flash Table A5), a
    confidence threshold stops drafting before the first position whose
    confidence is below it (Alignment Drift Table 21), and at most R - 1 are
    proposed when R output tokens remain (Appendix A.1)."""
    n = max(0, min(k_verify, len(cand), R - 1))
    if threshold > 0:
        for j in range(n):
            if proposal_confidence(q_logits[j], cand[j], T, suppress) < threshold:
                return j
    return n


def speculative_greedy_limited(orc: Oracle, req: Request, budget: int, k_verify: int, threshold: float,
                               conf_log: list | None = None) -> DecodeResult:
    """Propose / verify / advance with the parallel drafter's greedy proposals,
    verifying only the first k_verify of them and stopping at the first one
    below the confidence threshold.  conf_log, when given, receives each
    round's confidences of the K drafted tokens."""
    eos = orc.s.eos_id
    acc, logits = prefill(orc, req, budget)
    out = list(acc.emitted)
    res = DecodeResult(out, margins=[top2_margin(logits[-1])])
    done, anchor = acc.done, acc.next_anchor
    while not done:
        R = budget - len(out)
        q = orc.draft_logits(req, anchor)
        cand = [argmax_lowest(q[j]) for j in range(orc.s.K)]
        if conf_log is not None:
            conf_log.append([proposal_confidence(q[j], cand[j], 0.0) for j in range(orc.s.K)])
        n_prop = limit_proposals(cand, q, k_verify, threshold, 0.0, R)
        block = [anchor] + cand[:n_prop]
        lg = orc.verify(req, block)
        g = [argmax_lowest(z) for z in lg]
        acc = accept_greedy(block, n_prop, g, R, eos)
        res.margins += [top2_margin(lg[i]) for i in range(len(acc.emitted))]
        req.L += 1 + acc.a
        out += acc.emitted
        res.rounds += 1
        res.accepted.append(acc.a)
        res.proposed.append(n_prop)
        res.emitted.append(len(acc.emitted))
        done, anchor = acc.done, acc.next_anchor
    return res


def speculative_greedy_windowed(orc: Oracle, req: Request, budget: int, readout_layer: int,
                                half_width: int) -> DecodeResult:
    """Verification-attention correction (Alignment Drift §5, App. D.2):
    every target pass also reads its head-averaged audio attention at
    `readout_layer`; the peak frame of the row that produced the next anchor
    centres the drafter's cross-attention window for the next round (the
    prompt pass sets the first centre).  Proposals are the drafter's greedy
    tokens; acceptance is unchanged, so the output is greedy decoding's."""
    K, eos = orc.s.K, orc.s.eos_id
    prompt = list(orc.s.prompt)
    logits = orc.verify(req, prompt, readout_layer)
    g = [argmax_lowest(z) for z in logits]
    acc = accept_forced(len(prompt) - 1, g, budget, eos)
    req.center = req.peaks[acc.a]
    req.L += 1 + acc.a
    out = list(acc.emitted)
    res = DecodeResult(out)
    done, anchor = acc.done, acc.next_anchor
    centers = [req.center]
    while not done:
        R = budget - len(out)
        n_prop = min(K, R - 1)
        q = orc.draft_logits(req, anchor, half_width)
        cand = [argmax_lowest(q[j]) for j in range(n_prop)]
        block = [anchor] + cand
        lg = orc.verify(req, block, readout_layer)
        g = [argmax_lowest(z) for z in lg]
        acc = accept_greedy(block, n_prop, g, R, eos)
        req.center = req.peaks[acc.a]
        centers.append(req.center)
        req.L += 1 + acc.a
        out += acc.emitted
        res.rounds += 1
        res.accepted.append(acc.a)
        res.proposed.append(n_prop)
        res.emitted.append(len(acc.emitted))
        done, anchor = acc.done, acc.next_anchor
    res.margins = centers            # the window centre used by each round (prompt's first)
    return res


def drafter_proposer(orc: Oracle):
    """Greedy proposals from the parallel drafter (argmax of each mask row)."""
    def propose(req, anchor, t, n_prop):
        z = orc.draft_logits(req, anchor)
        return [argmax_lowest(z[j]) for j in range(n_prop)]
    return propose


def corrupted_proposer(traj_with_prompt, mask, tok):
    """Synthetic drafts: candidate j for an anchor at position t is
    traj[t + j] unless the corruption plan replaces it."""
    def propose(req, anchor, t, n_prop):
        out = []
        for j in range(1, n_prop + 1):
            if mask[t, j - 1]:
                out.append(int(tok[t, j - 1]))
            else:
                p = t + j
                out.append(int(traj_with_prompt[p]) if p < len(traj_with_prompt) else int(tok[t, j - 1]))
        return out
    return propose


def sampling_plain(orc: Oracle, req: Request, budget: int, T: float, seed: int, slot: int,
                   suppress=None) -> DecodeResult:
    """Autoregressive sampling from the target at temperature T: after the
    prompt, every round verifies the anchor alone and draws the next token
    from softmax(z/T) (the rejection rule with no candidates reduces to the
    bonus draw; Philox counter (slot, round, 1, 2))."""
    acc, logits = prefill(orc, req, budget, T, seed, slot)
    out, done, anchor, rnd = list(acc.emitted), acc.done, acc.next_anchor, 0
    res = DecodeResult(out, margins=list(acc.margins))
    while not done:
        rnd += 1
        lg = orc.verify(req, [anchor])
        acc, _ = accept_sampling([anchor], 0, lg, None, T, seed, slot, rnd, budget - len(out), orc.s.eos_id,
                                 suppress)
        req.L += 1 + acc.a
        out += acc.emitted
        res.margins += acc.margins
        done, anchor = acc.done, acc.next_anchor
        res.rounds += 1
    return res


def speculative_sampling(orc: Oracle, req: Request, budget: int, T: float, seed: int, slot: int,
                         suppress=None) -> DecodeResult:
    """Speculative sampling with the parallel drafter (Whisper-Flash §3.1,
    Appendix A.4): each mask row is sampled independently from its draft
    distribution (counter (slot, round, j, 0)), the target verifies the block,
    the rejection rule accepts or resamples."""
    K, eos = orc.s.K, orc.s.eos_id
    acc, logits = prefill(orc, req, budget, T, seed, slot)
    out, done, anchor, rnd = list(acc.emitted), acc.done, acc.next_anchor, 0
    res = DecodeResult(out, margins=list(acc.margins))
    while not done:
        rnd += 1
        R = budget - len(out)
        n_prop = min(K, R - 1)
        q = orc.draft_logits(req, anchor)
        cand = [sample_draft(q[j], T, seed, slot, rnd, j + 1, suppress) for j in range(K)]
        cmarg = [cdf_margin(probs_fp32(q[j], T, suppress),
                            philox.uniform(seed, slot, rnd, j + 1, philox.PURPOSE_DRAFT)) for j in range(K)]
        block = [anchor] + cand[:n_prop]
        lg = orc.verify(req, block)
        acc, _ = accept_sampling(block, n_prop, lg, q, T, seed, slot, rnd, R, eos, suppress, cand_margins=cmarg)
        req.L += 1 + acc.a
        out += acc.emitted
        res.margins += acc.margins
        res.rounds += 1
        res.accepted.append(acc.a)
        res.proposed.append(n_prop)
        res.emitted.append(len(acc.emitted))
        done, anchor = acc.done, acc.next_anchor
    return res


def acceptance_metrics(res: DecodeResult, K: int) -> dict:
    """alpha = accepted / proposed, tau = emitted per target call, mean a,
    cumulative survival s_k (Alignment Drift §3 'Speculative Loop')."""
    prop = np.asarray(res.proposed)
    acc = np.asarray(res.accepted)
    n_round = max(len(acc), 1)
    s = [float(np.mean(acc >= k)) if len(acc) else 0.0 for k in range(1, K + 1)]
    return {"alpha": float(acc.sum() / max(prop.sum(), 1)),
            "tau": float(np.sum(res.emitted) / max(res.rounds, 1)),
            "mean_a": float(acc.mean()) if len(acc) else 0.0,
            "survival": s, "rounds": res.rounds}
