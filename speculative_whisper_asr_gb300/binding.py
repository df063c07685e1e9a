"""ctypes binding of libws (include/ws.h): argument marshalling only.

Every function has the name of the C entry point it calls and takes plain
integers for device pointers (e.g. ``tensor.data_ptr()``) and for the CUDA
stream (``torch.cuda.current_stream().cuda_stream``).  A negative return code
raises ``WSError`` with the library's message.  There is no fallback: if the
shared library has not been built this module fails to import.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libws.so")

WS_OK, WS_EINVAL, WS_ENOSPACE, WS_EPOS, WS_ECUDA, WS_EDEVICE, WS_EUNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
WS_F32, WS_BF16 = 0, 1
WS_GEMM_AUTO, WS_GEMM_SIMT, WS_GEMM_TC = 0, 1, 2
WS_ACCEPT_GREEDY, WS_ACCEPT_SAMPLE, WS_ACCEPT_FORCED, WS_ACCEPT_TREE = 0, 1, 2, 3

EXPORTS = ("ws_query_workspace", "ws_load_weights", "ws_reset", "ws_cross_kv", "ws_verify", "ws_draft",
           "ws_accept", "ws_draft_synthetic", "ws_sample", "ws_set_suppress", "ws_get_lengths", "ws_status",
           "ws_gemm_engine", "ws_launch_count", "ws_last_error", "ws_free", "ws_capture_begin",
           "ws_capture_end", "ws_graph_launch", "ws_graph_free", "ws_argmax_rows_noalloc", "ws_fused_verify", "ws_draft_limit", "ws_set_readout", "ws_readout",
           "ws_get_centers", "ws_set_tree", "ws_tree_tokens", "ws_verify_tree",
           "ws_encoder_workspace", "ws_encoder_load", "ws_encode", "ws_encoder_status", "ws_encoder_error",
           "ws_encoder_free", "ws_encoder_attention",
           "ws_fused_layernorm")


class WSError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"ws error {code}: {msg}")
        self.code = code


class ModelDesc(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32), ("d_ff", C.c_int32),
                ("vocab", C.c_int32), ("max_pos", C.c_int32), ("drafter_layers", C.c_int32),
                ("n_hist", C.c_int32), ("hist_layers", C.c_int32 * 8), ("K", C.c_int32), ("dtype", C.c_int32),
                ("max_batch", C.c_int32), ("max_frames", C.c_int32), ("max_block", C.c_int32),
                ("eos_id", C.c_int32), ("gemm", C.c_int32)]


class AcceptArgs(C.Structure):
    _fields_ = [("mode", C.c_int32), ("H", C.c_int32), ("block", C.c_void_p), ("block_len", C.c_void_p),
                ("target", C.c_void_p), ("p_logits", C.c_void_p), ("q_logits", C.c_void_p),
                ("temperature", C.c_float), ("seed", C.c_uint64), ("round", C.c_uint64),
                ("budget", C.c_void_p), ("done", C.c_void_p), ("n_acc", C.c_void_p), ("n_emit", C.c_void_p),
                ("next_block", C.c_void_p), ("next_stride", C.c_int32), ("next_len", C.c_void_p),
                ("transcript", C.c_void_p), ("out_len", C.c_void_p), ("tcap", C.c_int32),
                ("n_done", C.c_void_p)]


class EncoderDesc(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32), ("d_ff", C.c_int32),
                ("n_mels", C.c_int32), ("n_frames", C.c_int32), ("max_batch", C.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = C.CDLL(LIB_PATH)
    P, I, U64, F, S = C.c_void_p, C.c_int, C.c_uint64, C.c_float, C.c_void_p
    sig = {
        "ws_query_workspace": (C.c_size_t, [C.POINTER(ModelDesc)]),
        "ws_load_weights": (I, [C.POINTER(P), C.POINTER(ModelDesc), P, C.c_size_t, P, P, S]),
        "ws_reset": (I, [P, I, P, S]),
        "ws_cross_kv": (I, [P, I, P, P, P, P, I, I, S]),
        "ws_verify": (I, [P, I, P, I, P, P, P, P, S]),
        "ws_draft": (I, [P, I, P, P, F, U64, U64, P, S]),
        "ws_accept": (I, [P, I, P, C.POINTER(AcceptArgs), S]),
        "ws_draft_synthetic": (I, [P, I, P, P, P, I, P, P, S]),
        "ws_sample": (I, [P, I, P, P, I, F, U64, U64, P, S]),
        "ws_set_suppress": (I, [P, P]),
        "ws_get_lengths": (I, [P, I, P, P, S]),
        "ws_status": (I, [P, S, C.POINTER(C.c_int32)]),
        "ws_gemm_engine": (C.c_char_p, [P]),
        "ws_fused_verify": (C.c_int, [P, C.c_int]),
        "ws_fused_layernorm": (C.c_int, [P, C.c_int]),
        "ws_launch_count": (C.c_ulonglong, []),
        "ws_last_error": (C.c_char_p, [P]),
        "ws_free": (None, [P]),
        "ws_capture_begin": (I, [P, S]),
        "ws_capture_end": (I, [P, S, C.POINTER(P)]),
        "ws_graph_launch": (I, [P, S]),
        "ws_graph_free": (None, [P]),
        "ws_argmax_rows_noalloc": (I, [P, I, I, P, P, S]),
        "ws_draft_limit": (I, [P, I, P, P, I, P, I, C.c_float, C.c_float, P, I, P, S]),
        "ws_set_readout": (I, [P, I, I]),
        "ws_readout": (I, [P, I, P, P, S]),
        "ws_get_centers": (I, [P, I, P, P, S]),
        "ws_set_tree": (I, [P, I, P, P]),
        "ws_tree_tokens": (I, [P, I, P, P, I, P, P, I, P, S]),
        "ws_verify_tree": (I, [P, I, P, I, P, P, P, P, S]),
        "ws_encoder_workspace": (C.c_size_t, [C.POINTER(EncoderDesc)]),
        "ws_encoder_load": (I, [C.POINTER(P), C.POINTER(EncoderDesc), P, C.c_size_t, P, S]),
        "ws_encode": (I, [P, I, P, P, S]),
        "ws_encoder_status": (I, [P, S, C.POINTER(C.c_int32)]),
        "ws_encoder_error": (C.c_char_p, [P]),
        "ws_encoder_free": (None, [P]),
        "ws_encoder_attention": (I, [P, I]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _check(ctx, rc: int) -> int:
    if rc < 0:
        raise WSError(rc, lib.ws_last_error(ctx).decode())
    return rc


def make_desc(n_layers, d_model, n_heads, d_ff, vocab, max_pos, drafter_layers, hist_layers, K, dtype,
              max_batch, max_frames, max_block, eos_id, gemm=WS_GEMM_AUTO) -> ModelDesc:
    d = ModelDesc()
    d.n_layers, d.d_model, d.n_heads, d.d_ff, d.vocab, d.max_pos = n_layers, d_model, n_heads, d_ff, vocab, max_pos
    d.drafter_layers = drafter_layers
    d.n_hist = len(hist_layers)
    for i, l in enumerate(hist_layers):
        d.hist_layers[i] = l
    d.K, d.dtype, d.max_batch, d.max_frames, d.max_block, d.eos_id, d.gemm = (
        K, dtype, max_batch, max_frames, max_block, eos_id, gemm)
    return d


def ws_query_workspace(desc: ModelDesc) -> int:
    return int(lib.ws_query_workspace(C.byref(desc)))


def ws_load_weights(desc: ModelDesc, workspace: int, nbytes: int, target_blob: int, drafter_blob: int,
                    stream: int) -> int:
    h = C.c_void_p()
    _check(None, lib.ws_load_weights(C.byref(h), C.byref(desc), workspace, nbytes, target_blob,
                                     drafter_blob or None, stream))
    return h.value


def ws_reset(ctx, n, req_ids, stream):
    return _check(ctx, lib.ws_reset(ctx, n, req_ids, stream))


def ws_cross_kv(ctx, n, req_ids, enc, cu_frames, valid_frames, max_frames_call, total_frames, stream):
    return _check(ctx, lib.ws_cross_kv(ctx, n, req_ids, enc, cu_frames, valid_frames or None, max_frames_call,
                                       total_frames, stream))


def ws_verify(ctx, n, req_ids, H, block, block_len, target, logits, stream):
    return _check(ctx, lib.ws_verify(ctx, n, req_ids, H, block, block_len, target, logits or None, stream))


def ws_draft(ctx, n, req_ids, block, temperature, seed, rnd, q_logits, stream):
    return _check(ctx, lib.ws_draft(ctx, n, req_ids, block, temperature, seed, rnd, q_logits or None, stream))


def ws_accept(ctx, n, req_ids, args: AcceptArgs, stream):
    return _check(ctx, lib.ws_accept(ctx, n, req_ids, C.byref(args), stream))


def ws_draft_synthetic(ctx, n, req_ids, block, traj, tlen, cmask, ctok, stream):
    return _check(ctx, lib.ws_draft_synthetic(ctx, n, req_ids, block, traj, tlen, cmask, ctok, stream))


def ws_sample(ctx, n, req_ids, logits, rows, temperature, seed, rnd, out, stream):
    return _check(ctx, lib.ws_sample(ctx, n, req_ids, logits, rows, temperature, seed, rnd, out, stream))


def ws_set_suppress(ctx, mask):
    return _check(ctx, lib.ws_set_suppress(ctx, mask or None))


def ws_get_lengths(ctx, n, req_ids, out, stream):
    return _check(ctx, lib.ws_get_lengths(ctx, n, req_ids, out, stream))


def ws_status(ctx, stream) -> int:
    v = C.c_int32(0)
    rc = lib.ws_status(ctx, stream, C.byref(v))
    if rc < 0 and rc != WS_EDEVICE:
        _check(ctx, rc)
    return int(v.value)


def ws_gemm_engine(ctx) -> str:
    return lib.ws_gemm_engine(ctx).decode()


def ws_fused_verify(ctx, enable: int = -1) -> int:
    """Switch the persistent verify path (1 on, 0 off, -1 query); returns 1 when in use."""
    r = lib.ws_fused_verify(ctx, enable)
    if r < 0:
        raise WSError(r, lib.ws_last_error(ctx).decode())
    return r


def ws_fused_layernorm(ctx, enable: int = -1) -> int:
    """Switch layer norm inside eligible GEMMs (1 on, 0 off, -1 query); returns 1 when on."""
    r = lib.ws_fused_layernorm(ctx, enable)
    if r < 0:
        raise WSError(r, lib.ws_last_error(ctx).decode())
    return r


def ws_launch_count() -> int:
    return int(lib.ws_launch_count())


def ws_last_error(ctx=None) -> str:
    return lib.ws_last_error(ctx).decode()


def ws_free(ctx):
    lib.ws_free(ctx)


def ws_capture_begin(ctx, stream):
    return _check(ctx, lib.ws_capture_begin(ctx, stream))


def ws_capture_end(ctx, stream) -> int:
    g = C.c_void_p()
    _check(ctx, lib.ws_capture_end(ctx, stream, C.byref(g)))
    return g.value


def ws_graph_launch(graph, stream):
    return _check(None, lib.ws_graph_launch(graph, stream))


def ws_graph_free(graph):
    lib.ws_graph_free(graph)


def ws_draft_limit(ctx, n, req, block, stride_in, q_logits, k_verify, threshold, temperature, block_out,
                   stride_out, block_len, stream):
    return _check(ctx, lib.ws_draft_limit(ctx, n, req, block, stride_in, q_logits or None, k_verify,
                                          float(threshold), float(temperature), block_out, stride_out, block_len,
                                          stream))


def ws_set_readout(ctx, layer, half_width):
    return _check(ctx, lib.ws_set_readout(ctx, layer, half_width))


def ws_readout(ctx, n, req, row, stream):
    return _check(ctx, lib.ws_readout(ctx, n, req, row, stream))


def ws_get_centers(ctx, n, req, out, stream):
    return _check(ctx, lib.ws_get_centers(ctx, n, req, out, stream))


def ws_set_tree(ctx, parent, rank):
    """parent, rank: host sequences of the tree's rows (empty = no tree)."""
    n = len(parent)
    pa = (C.c_int32 * max(n, 1))(*parent)
    ra = (C.c_int32 * max(n, 1))(*rank)
    return _check(ctx, lib.ws_set_tree(ctx, n, pa if n else None, ra if n else None))


def ws_tree_tokens(ctx, n, req, block, stride_in, q_logits, block_out, stride_out, block_len, stream):
    return _check(ctx, lib.ws_tree_tokens(ctx, n, req, block, stride_in, q_logits, block_out, stride_out, block_len,
                                          stream))


def ws_verify_tree(ctx, n, req_ids, H, block, block_len, target, logits, stream):
    return _check(ctx, lib.ws_verify_tree(ctx, n, req_ids, H, block, block_len, target, logits or None, stream))


def _echeck(enc, rc: int) -> int:
    if rc < 0:
        raise WSError(rc, lib.ws_encoder_error(enc).decode())
    return rc


def make_encoder_desc(n_layers, d_model, n_heads, d_ff, n_mels, n_frames, max_batch) -> EncoderDesc:
    d = EncoderDesc()
    d.n_layers, d.d_model, d.n_heads, d.d_ff, d.n_mels, d.n_frames, d.max_batch = (
        n_layers, d_model, n_heads, d_ff, n_mels, n_frames, max_batch)
    return d


def ws_encoder_workspace(desc: EncoderDesc) -> int:
    return int(lib.ws_encoder_workspace(C.byref(desc)))


def ws_encoder_load(desc: EncoderDesc, workspace: int, nbytes: int, blob: int, stream: int) -> int:
    h = C.c_void_p()
    _echeck(None, lib.ws_encoder_load(C.byref(h), C.byref(desc), workspace, nbytes, blob, stream))
    return h.value


def ws_encode(enc, n, mel, out, stream):
    return _echeck(enc, lib.ws_encode(enc, n, mel, out, stream))


def ws_encoder_status(enc, stream) -> int:
    v = C.c_int32(0)
    _echeck(enc, lib.ws_encoder_status(enc, stream, C.byref(v)))
    return v.value


def ws_encoder_attention(enc, mode: int) -> int:
    return _echeck(enc, lib.ws_encoder_attention(enc, mode))


def ws_encoder_free(enc):
    lib.ws_encoder_free(enc)


def ws_argmax_rows_noalloc(logits, rows, vocab, suppress, out, stream):
    return _check(None, lib.ws_argmax_rows_noalloc(logits, rows, vocab, suppress or None, out, stream))
