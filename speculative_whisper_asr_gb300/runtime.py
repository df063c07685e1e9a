"""Host driver for libws: device buffers (PyTorch), weight upload and the
propose / verify / accept loop.  Every step of the decoding path runs in the
library's CUDA kernels; this module only allocates memory, marshals
arguments and decides when the loop stops.

Loop (Whisper-Flash §3.1, Appendix A.1):
  prefill   : ws_verify(prompt) + ws_accept(FORCED) -> first anchor
  each round: ws_draft (or ws_draft_synthetic) -> ws_verify(K+1 rows)
              -> ws_accept (greedy or rejection rule) -> next anchor
  AR greedy : ws_verify(1 row) + ws_accept with no proposals
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from . import binding as B


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


@dataclass
class RunStats:
    rounds: int = 0
    proposed: int = 0
    accepted: int = 0
    emitted: int = 0
    per_round_acc: list = field(default_factory=list)


class Decoder:
    """One libws context on the current CUDA device."""

    def __init__(self, shape: synth.ModelShape, target: dict, drafter: dict | None, max_batch: int,
                 max_frames: int = 1500, gemm: int = B.WS_GEMM_AUTO, max_block: int | None = None):
        if not torch.cuda.is_available():
            raise RuntimeError("libws needs a CUDA device")
        self.s = shape
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.max_batch = max_batch
        self.max_frames = max_frames
        self.K = shape.K
        self.V = shape.vocab
        self.dtype = B.WS_BF16 if shape.dtype == "bf16" else B.WS_F32
        self.tdtype = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
        self.readout = False
        self.tree = None
        dl = shape.drafter_layers if drafter is not None else 0
        self.max_block = max_block or max(shape.K + 1, len(shape.prompt))
        self.desc = B.make_desc(shape.n_layers, shape.d_model, shape.n_heads, shape.d_ff, shape.vocab,
                                shape.max_pos, dl, shape.hist_layers, shape.K, self.dtype, max_batch, max_frames,
                                self.max_block, shape.eos_id, gemm)
        nbytes = B.ws_query_workspace(self.desc)
        if nbytes == 0:
            raise ValueError("invalid model description")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        tblob = self._blob(target, synth.target_tensor_shapes(shape))
        dblob = self._blob(drafter, synth.drafter_tensor_shapes(shape)) if dl else None
        self.ctx = B.ws_load_weights(self.desc, self.workspace.data_ptr(), nbytes, tblob.data_ptr(),
                                     _ptr(dblob), _stream())
        del tblob, dblob
        self.engine = B.ws_gemm_engine(self.ctx)

    def __del__(self):
        ctx = getattr(self, "ctx", None)
        if ctx:
            B.ws_free(ctx)
            self.ctx = None

    def _blob(self, tensors, order):
        t = torch.from_numpy(synth.blob_from(tensors, order, self.s.dtype))
        if self.s.dtype == "bf16":
            t = t.view(torch.int16)
        return t.to(self.dev)

    def enc_tensor(self, A: np.ndarray) -> torch.Tensor:
        """Encoder states (already in the model's value set) as a device tensor."""
        if self.s.dtype == "bf16":
            return torch.from_numpy(synth.bf16_bits(A)).view(torch.int16).to(self.dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(A, dtype=np.float32)).to(self.dev)

    # ------------------------------------------------------------------ raw calls
    def slots(self, ids) -> torch.Tensor:
        return torch.as_tensor(np.asarray(ids, dtype=np.int32), device=self.dev)

    def reset(self, req):
        B.ws_reset(self.ctx, req.numel(), req.data_ptr(), _stream())

    def cross_kv(self, req, enc_packed: torch.Tensor, frames, valid=None):
        frames = np.asarray(frames, dtype=np.int32)
        cu = torch.as_tensor(np.concatenate([[0], np.cumsum(frames)]).astype(np.int32), device=self.dev)
        vt = None if valid is None else torch.as_tensor(np.asarray(valid, dtype=np.int32), device=self.dev)
        B.ws_cross_kv(self.ctx, req.numel(), req.data_ptr(), enc_packed.data_ptr(), cu.data_ptr(), _ptr(vt),
                      int(frames.max()), int(frames.sum()), _stream())
        return cu, vt

    def verify(self, req, block, block_len, target, logits=None):
        n, H = block.shape
        B.ws_verify(self.ctx, n, req.data_ptr(), H, block.data_ptr(), block_len.data_ptr(), target.data_ptr(),
                    _ptr(logits), _stream())

    def draft(self, req, block, temperature=0.0, seed=0, rnd=0, q_logits=None):
        B.ws_draft(self.ctx, req.numel(), req.data_ptr(), block.data_ptr(), float(temperature), seed, rnd,
                   _ptr(q_logits), _stream())

    def sample(self, req, logits, temperature, seed, rnd, out):
        n, rows = out.shape
        B.ws_sample(self.ctx, n, req.data_ptr(), logits.data_ptr(), rows, float(temperature), seed, rnd,
                    out.data_ptr(), _stream())

    def lengths(self, req) -> np.ndarray:
        out = torch.empty(req.numel(), dtype=torch.int32, device=self.dev)
        B.ws_get_lengths(self.ctx, req.numel(), req.data_ptr(), out.data_ptr(), _stream())
        return out.cpu().numpy()

    def status(self) -> int:
        return B.ws_status(self.ctx, _stream())

    def set_readout(self, layer: int, half_width: int):
        """Verification-attention readout at `layer` centring a +-half_width
        frame window on the drafter's cross-attention (layer -1: off)."""
        B.ws_set_readout(self.ctx, layer, half_width)
        self.readout = layer >= 0

    def set_tree(self, parent=(), rank=()):
        """Candidate tree of block rows for tree verification (Alignment Drift
        App. E.3): parent[j] < j (parent[0] = -1), rank[j] = which of the
        drafter's ranked tokens row j takes at its depth; empty: no tree."""
        B.ws_set_tree(self.ctx, list(parent), list(rank))
        self.tree = (tuple(parent), tuple(rank)) if len(parent) else None

    def centers(self, req) -> np.ndarray:
        out = torch.empty(req.numel(), dtype=torch.int32, device=self.dev)
        B.ws_get_centers(self.ctx, req.numel(), req.data_ptr(), out.data_ptr(), _stream())
        return out.cpu().numpy()

    # ------------------------------------------------------------------ batch state
    def new_batch(self, req, budgets, tcap: int | None = None, sampling: bool = False,
                  draft_logits: bool = False) -> "Batch":
        """draft_logits: keep the drafter's logits also for greedy decoding
        (needed by a confidence threshold)."""
        return Batch(self, req, budgets, tcap or self.s.max_pos, sampling, draft_logits)


class Batch:
    """Device arrays of one decoding batch (request slots `req`)."""

    def __init__(self, dec: Decoder, req: torch.Tensor, budgets, tcap: int, sampling: bool,
                 draft_logits: bool = False):
        self.dec = dec
        self.req = req
        n = req.numel()
        self.n = n
        dev, K = dec.dev, dec.K
        i32 = dict(dtype=torch.int32, device=dev)
        self.block = torch.zeros(n, K + 1, **i32)
        self.blen = torch.zeros(n, **i32)
        self.target = torch.zeros(n, K + 1, **i32)
        self.block1 = torch.zeros(n, 1, **i32)
        self.target1 = torch.zeros(n, 1, **i32)
        self.prompt = torch.as_tensor(np.tile(np.asarray(dec.s.prompt, dtype=np.int32), (n, 1)), device=dev)
        self.plen = torch.full((n,), len(dec.s.prompt), **i32)
        self.ptarget = torch.zeros(n, len(dec.s.prompt), **i32)
        self.budget = torch.as_tensor(np.asarray(budgets, dtype=np.int32), device=dev).clone()
        self.done = torch.zeros(n, **i32)
        self.n_acc = torch.zeros(n, **i32)
        self.n_emit = torch.zeros(n, **i32)
        self.transcript = torch.full((n, tcap), -1, **i32)
        self.out_len = torch.zeros(n, **i32)
        self.n_done = torch.zeros(1, **i32)
        self.tcap = tcap
        self.acc_sum = torch.zeros(n, dtype=torch.int64, device=dev)
        self.prop_sum = torch.zeros(n, dtype=torch.int64, device=dev)
        self.p_logits = self.q_logits = self.p_logits1 = None
        if sampling:
            self.p_logits = torch.empty(n, K + 1, dec.V, dtype=torch.float32, device=dev)
        if sampling or draft_logits or dec.tree is not None:
            self.q_logits = torch.empty(n, K, dec.V, dtype=torch.float32, device=dev)
        self.vblock = torch.zeros(n, K + 1, **i32)      # the block as verified (truncated proposals)
        self.tblock = torch.zeros(n, dec.max_block, **i32)    # a candidate tree's tokens
        self.ttarget = torch.zeros(n, dec.max_block, **i32)
        self.host_done = torch.zeros(1, dtype=torch.int32).pin_memory()
        self.graphs = {}

    def __del__(self):
        for g in getattr(self, "graphs", {}).values():
            B.ws_graph_free(g)

    def replay(self, key, fn):
        """Run `fn` (a fixed sequence of ws_* calls) through a CUDA graph
        captured on first use; later calls replay it."""
        g = self.graphs.get(key)
        s = _stream()
        if g is None:
            B.ws_capture_begin(self.dec.ctx, s)
            try:
                fn()
            finally:
                g = B.ws_capture_end(self.dec.ctx, s)
            self.graphs[key] = g
        B.ws_graph_launch(g, s)

    def _args(self, mode, H, block, blen, target, next_block, next_len, p_logits=None, q_logits=None,
              temperature=0.0, seed=0, rnd=0) -> B.AcceptArgs:
        a = B.AcceptArgs()
        a.mode, a.H = mode, H
        a.block, a.block_len, a.target = block.data_ptr(), blen.data_ptr(), _ptr(target)
        a.p_logits, a.q_logits = _ptr(p_logits), _ptr(q_logits)
        a.temperature, a.seed, a.round = float(temperature), int(seed), int(rnd)
        a.budget, a.done, a.n_acc, a.n_emit = (self.budget.data_ptr(), self.done.data_ptr(),
                                               self.n_acc.data_ptr(), self.n_emit.data_ptr())
        a.next_block, a.next_stride, a.next_len = next_block.data_ptr(), next_block.shape[1], next_len.data_ptr()
        a.transcript, a.out_len, a.tcap = self.transcript.data_ptr(), self.out_len.data_ptr(), self.tcap
        a.n_done = self.n_done.data_ptr()
        return a

    def prefill(self, ar: bool = False, temperature: float = 0.0, seed: int = 0):
        """Prompt pass: emits the first transcript token (the first anchor)."""
        d = self.dec
        d.reset(self.req)
        sampled = temperature > 0.0 and self.p_logits is not None
        d.verify(self.req, self.prompt, self.plen, self.ptarget, self.p_logits if sampled else None)
        nb = self.block1 if ar else self.block
        a = self._args(B.WS_ACCEPT_FORCED, self.prompt.shape[1], self.prompt, self.plen, self.ptarget, nb,
                       self.blen, self.p_logits if sampled else None, None, temperature if sampled else 0.0,
                       seed, 0)
        B.ws_accept(d.ctx, self.n, self.req.data_ptr(), a, _stream())
        if d.readout and not ar:
            B.ws_readout(d.ctx, self.n, self.req.data_ptr(), self.n_acc.data_ptr(), _stream())

    def ar_step(self, graph: bool = True):
        d = self.dec

        def calls():
            d.verify(self.req, self.block1, self.blen, self.target1)
            a = self._args(B.WS_ACCEPT_GREEDY, 1, self.block1, self.blen, self.target1, self.block1, self.blen)
            B.ws_accept(d.ctx, self.n, self.req.data_ptr(), a, _stream())
        if graph:
            self.replay(("ar",), calls)
        else:
            calls()

    def ar_sample_step(self, rnd: int, temperature: float, seed: int):
        """Autoregressive sampling round: verify the anchor, draw from softmax(z/T)."""
        d = self.dec
        d.verify(self.req, self.block1, self.blen, self.target1, self.p_logits)
        a = self._args(B.WS_ACCEPT_SAMPLE, 1, self.block1, self.blen, self.target1, self.block1, self.blen,
                       self.p_logits, self.q_logits, temperature, seed, rnd)
        B.ws_accept(d.ctx, self.n, self.req.data_ptr(), a, _stream())

    def spec_step(self, rnd: int, synthetic=None, temperature: float = 0.0, seed: int = 0, run_drafter=True,
                  graph: bool = True, k_verify: int | None = None, threshold: float = 0.0, tree: bool = False):
        """One propose / verify / accept round.  `synthetic` = (traj, cmask, ctok) device tensors.
        k_verify / threshold: verify only the first k_verify proposals, stopping
        before the first one whose drafter confidence is below threshold
        (ws_draft_limit).  Greedy rounds replay one captured graph per
        (proposal source, verify length, threshold): their calls do not depend
        on the round.  tree: the drafter's ranked tokens fill the decoder's
        candidate tree (set_tree), verified in one pass and accepted along
        the longest matching root path (greedy only)."""
        if tree:
            if temperature > 0.0 or synthetic is not None or not run_drafter or self.dec.tree is None:
                raise ValueError("tree rounds need set_tree, the drafter and greedy decoding")
            if graph:
                self.replay(("tree", self.dec.tree), self._tree_calls)
            else:
                self._tree_calls()
        elif graph and temperature <= 0.0:
            self.replay(("spec", synthetic is not None, run_drafter, k_verify, threshold),
                        lambda: self._spec_calls(0, synthetic, 0.0, 0, run_drafter, k_verify, threshold))
        else:
            self._spec_calls(rnd, synthetic, temperature, seed, run_drafter, k_verify, threshold)

    def _tree_calls(self):
        d = self.dec
        N = len(d.tree[0])
        req = self.req.data_ptr()
        d.draft(self.req, self.block, 0.0, 0, 0, self.q_logits)
        B.ws_tree_tokens(d.ctx, self.n, req, self.block.data_ptr(), d.K + 1, self.q_logits.data_ptr(),
                         self.tblock.data_ptr(), N, self.blen.data_ptr(), _stream())
        B.ws_verify_tree(d.ctx, self.n, req, N, self.tblock.data_ptr(), self.blen.data_ptr(),
                         self.ttarget.data_ptr(), 0, _stream())
        a = self._args(B.WS_ACCEPT_TREE, N, self.tblock, self.blen, self.ttarget, self.block, self.blen)
        B.ws_accept(d.ctx, self.n, req, a, _stream())
        if d.readout:              # the path's rows are in block order after acceptance
            B.ws_readout(d.ctx, self.n, req, self.n_acc.data_ptr(), _stream())

    def _spec_calls(self, rnd, synthetic, temperature, seed, run_drafter, k_verify=None, threshold=0.0):
        d = self.dec
        sampling = temperature > 0.0
        K = d.K
        limited = k_verify is not None and (k_verify < K or threshold > 0.0)
        if run_drafter:
            d.draft(self.req, self.block, temperature, seed, rnd,
                    self.q_logits if (sampling or threshold > 0.0) else None)
        if synthetic is not None:
            traj, cmask, ctok = synthetic
            B.ws_draft_synthetic(d.ctx, self.n, self.req.data_ptr(), self.block.data_ptr(), traj.data_ptr(),
                                 traj.shape[1], cmask.data_ptr(), ctok.data_ptr(), _stream())
        H, vb = K + 1, self.block
        if limited:
            H, vb = k_verify + 1, self.vblock
            B.ws_draft_limit(d.ctx, self.n, self.req.data_ptr(), self.block.data_ptr(), K + 1,
                             _ptr(self.q_logits) if threshold > 0.0 else 0, k_verify, threshold, temperature,
                             vb.data_ptr(), H, self.blen.data_ptr(), _stream())
        B.ws_verify(d.ctx, self.n, self.req.data_ptr(), H, vb.data_ptr(), self.blen.data_ptr(),
                    self.target.data_ptr(), _ptr(self.p_logits) if sampling else 0, _stream())
        mode = B.WS_ACCEPT_SAMPLE if sampling else B.WS_ACCEPT_GREEDY
        a = self._args(mode, H, vb, self.blen, self.target, self.block, self.blen,
                       self.p_logits, self.q_logits, temperature, seed, rnd)
        B.ws_accept(d.ctx, self.n, self.req.data_ptr(), a, _stream())
        if d.readout:              # the row that produced the next anchor centres the next draft window
            B.ws_readout(d.ctx, self.n, self.req.data_ptr(), self.n_acc.data_ptr(), _stream())

    def poll_done(self) -> int:
        self.host_done.copy_(self.n_done, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return int(self.host_done.item())

    def transcripts(self):
        t = self.transcript.cpu().numpy()
        n = self.out_len.cpu().numpy()
        return [list(map(int, t[i, :n[i]])) for i in range(self.n)]


def run_ar(dec: Decoder, batch: Batch, max_rounds: int = 100000) -> int:
    batch.prefill(ar=True)
    rounds = 0
    while batch.poll_done() < batch.n and rounds < max_rounds:
        batch.ar_step()
        rounds += 1
    return rounds


def run_spec(dec: Decoder, batch: Batch, synthetic=None, temperature=0.0, seed=0, max_rounds=100000,
             run_drafter=True, graph=True, k_verify=None, threshold=0.0, tree=False) -> int:
    batch.prefill(temperature=temperature, seed=seed)
    rounds = 0
    while batch.poll_done() < batch.n and rounds < max_rounds:
        batch.spec_step(rounds + 1, synthetic, temperature, seed, run_drafter, graph=graph, k_verify=k_verify,
                        threshold=threshold, tree=tree)
        rounds += 1
    return rounds


def run_ar_sampling(dec: Decoder, batch: Batch, temperature: float, seed: int, max_rounds=100000) -> int:
    batch.prefill(ar=True, temperature=temperature, seed=seed)
    rounds = 0
    while batch.poll_done() < batch.n and rounds < max_rounds:
        rounds += 1
        batch.ar_sample_step(rounds, temperature, seed)
    return rounds


def run_spec_packed(dec: Decoder, req_all: torch.Tensor, budgets, synthetic=None, max_rounds=100000,
                    live_rounds: list | None = None):
    """Varlen batch without padding rows: after every round the requests that
    finished are dropped from the slot list, so later rounds only carry live
    requests (their rows, attention and acceptance).  Returns (transcripts,
    rounds, rows processed); `live_rounds`, when given, receives the number
    of rounds each request took part in."""
    n_all = req_all.numel()
    alive = list(range(n_all))
    out = [None] * n_all
    live = [0] * n_all
    budgets = np.asarray(budgets, dtype=np.int32)
    b = dec.new_batch(req_all, budgets)
    b.prefill()
    rounds, rows = 0, 0
    syn_all = synthetic
    while rounds < max_rounds:
        done = b.done.cpu().numpy()
        if done.any():
            tr = b.transcripts()
            keep = [k for k in range(len(alive)) if not done[k]]
            for k in range(len(alive)):
                if done[k]:
                    out[alive[k]] = tr[k]
            if not keep:
                break
            idx = torch.as_tensor(keep, device=dec.dev, dtype=torch.long)
            nb = dec.new_batch(b.req[idx].contiguous(), b.budget[idx].cpu().numpy(), b.tcap)
            for name in ("block", "blen", "budget", "done", "out_len", "transcript"):
                getattr(nb, name).copy_(getattr(b, name)[idx])
            if syn_all is not None:
                syn_all = tuple(t[idx].contiguous() for t in syn_all)
            alive = [alive[k] for k in keep]
            b = nb
        rounds += 1
        rows += b.n * (dec.K + 1)
        for k in alive:
            live[k] += 1
        b.spec_step(rounds, syn_all, graph=False)
    if live_rounds is not None:
        live_rounds[:] = live
    return out, rounds, rows


class Encoder:
    """libws audio encoder on the current CUDA device (bf16): log-mel windows
    [n, n_mels, 2F] -> encoder states [n, F, d], the input of Decoder.cross_kv."""

    def __init__(self, shape: synth.EncoderShape, weights: dict, max_batch: int):
        if not torch.cuda.is_available():
            raise RuntimeError("libws needs a CUDA device")
        if shape.dtype != "bf16":
            raise ValueError("the encoder runs in bf16")
        self.s = shape
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.max_batch = max_batch
        self.desc = B.make_encoder_desc(shape.n_layers, shape.d_model, shape.n_heads, shape.d_ff, shape.n_mels,
                                        shape.n_frames, max_batch)
        nbytes = B.ws_encoder_workspace(self.desc)
        if nbytes == 0:
            raise ValueError("invalid encoder description")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        blob = torch.from_numpy(synth.blob_from(weights, synth.encoder_tensor_shapes(shape), "bf16"))
        blob = blob.view(torch.int16).to(self.dev)
        self.enc = B.ws_encoder_load(self.desc, self.workspace.data_ptr(), nbytes, blob.data_ptr(), _stream())
        del blob

    def __del__(self):
        enc = getattr(self, "enc", None)
        if enc:
            B.ws_encoder_free(enc)
            self.enc = None

    def mel_tensor(self, mels) -> torch.Tensor:
        """Stack bf16-valued log-mel arrays [n_mels, 2F] into one device tensor."""
        a = np.stack([np.asarray(m, dtype=np.float32) for m in mels])
        return torch.from_numpy(synth.bf16_bits(a)).view(torch.int16).to(self.dev).view(torch.bfloat16)

    def encode(self, mel: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
        n = mel.shape[0]
        if out is None:
            out = torch.empty(n, self.s.n_frames, self.s.d_model, dtype=torch.bfloat16, device=self.dev)
        B.ws_encode(self.enc, n, mel.data_ptr(), out.data_ptr(), _stream())
        return out

    def status(self) -> int:
        return B.ws_encoder_status(self.enc, _stream())

    def set_attention(self, tcgen05: bool):
        """Attention kernel: tcgen05 flash attention (default) or the legacy mma.sync one."""
        B.ws_encoder_attention(self.enc, 1 if tcgen05 else 0)
