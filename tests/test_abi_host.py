"""Host-side checks of the C ABI: the library loads, every entry point that
include/ws.h declares is exported, and argument validation that needs no GPU
returns the documented error codes."""
import ctypes as C
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding
    return binding


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(ws_[a-z_0-9]+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported(B):
    declared = _declared()
    assert {"ws_load_weights", "ws_cross_kv", "ws_draft", "ws_verify", "ws_accept"} <= declared
    lib = C.CDLL(B.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert set(B.EXPORTS) == declared


def _desc(B, s, **kw):
    args = dict(n_layers=s.n_layers, d_model=s.d_model, n_heads=s.n_heads, d_ff=s.d_ff, vocab=s.vocab,
                max_pos=s.max_pos, drafter_layers=2, hist_layers=s.hist_layers, K=s.K,
                dtype=B.WS_BF16 if s.dtype == "bf16" else B.WS_F32, max_batch=4, max_frames=1500, max_block=9,
                eos_id=s.eos_id)
    args.update(kw)
    return B.make_desc(**args)


def test_query_workspace_sizes(B):
    tiny = B.ws_query_workspace(_desc(B, synth.TINY))
    lv3 = B.ws_query_workspace(_desc(B, synth.LARGE_V3, max_batch=1))
    assert tiny > 0 and lv3 > 0
    # large-v3 bf16: target 1.6 GB + drafter 0.3 GB + 34 layers of acoustic K/V (261 MB / request)
    assert 2.0e9 < lv3 < 2.6e9, lv3
    b96 = B.ws_query_workspace(_desc(B, synth.LARGE_V3, max_batch=96))
    assert b96 > 30e9       # acoustic K/V for 96 requests alone is 25 GB


@pytest.mark.parametrize("bad", [dict(d_model=100), dict(n_heads=5), dict(K=0), dict(K=16),
                                 dict(max_block=3), dict(dtype=7), dict(eos_id=10 ** 6), dict(vocab=51867), dict(vocab=65538),
                                 dict(hist_layers=(0, 9)), dict(max_frames=0), dict(gemm=9)])
def test_invalid_descriptions_rejected(B, bad):
    assert B.ws_query_workspace(_desc(B, synth.TINY, **bad)) == 0


def test_load_weights_argument_errors(B):
    d = _desc(B, synth.TINY)
    with pytest.raises(B.WSError) as e:
        B.ws_load_weights(d, 0, 1 << 30, 1, 1, 0)
    assert e.value.code == B.WS_EINVAL
    with pytest.raises(B.WSError) as e:
        B.ws_load_weights(d, 4096, 10, 1, 1, 0)        # too small workspace
    assert e.value.code == B.WS_ENOSPACE
    with pytest.raises(B.WSError) as e:
        B.ws_load_weights(d, 4097, 1 << 40, 1, 1, 0)   # misaligned workspace
    assert e.value.code == B.WS_EINVAL


def test_null_context_calls_fail_cleanly(B):
    for rc in (B.lib.ws_verify(None, 1, 1, 1, 1, 1, 1, None, None),
               B.lib.ws_draft(None, 1, 1, 1, 0.0, 0, 0, None, None),
               B.lib.ws_reset(None, 1, 1, None),
               B.lib.ws_cross_kv(None, 1, 1, 1, 1, None, 10, 10, None),
               B.lib.ws_fused_verify(None, 1),
               B.lib.ws_fused_layernorm(None, -1)):
        assert rc == B.WS_EINVAL
    assert "context" in B.ws_last_error()
    assert B.ws_gemm_engine(None) == "none"


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "speculative_whisper_asr_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "oracle" not in re.findall(r"^\s*(?:from|import)\s+([\w.]+)", src, flags=re.M), fn
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith(".py"):
            src = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "speculative_whisper_asr_gb300" not in src, fn


def _enc_desc(B, **kw):
    s = synth.ENC_LARGE_V3
    args = dict(n_layers=s.n_layers, d_model=s.d_model, n_heads=s.n_heads, d_ff=s.d_ff, n_mels=s.n_mels,
                n_frames=s.n_frames, max_batch=16)
    args.update(kw)
    return B.make_encoder_desc(**args)


def test_encoder_workspace_size():
    """Large-v3 encoder, 16 windows: 0.64 G bf16 weights plus the activations
    of 24,000 rows (a few GB), well inside one GPU."""
    from speculative_whisper_asr_gb300 import binding as B
    n = B.ws_encoder_workspace(_enc_desc(B))
    assert 1.0e9 < n < 8.0e9, n


@pytest.mark.parametrize("bad", [dict(d_model=100), dict(d_model=2176, n_heads=34), dict(n_heads=7),
                                 dict(d_ff=100), dict(n_layers=0), dict(n_mels=0), dict(n_frames=0),
                                 dict(max_batch=0)])
def test_invalid_encoder_descriptions_rejected(bad):
    from speculative_whisper_asr_gb300 import binding as B
    assert B.ws_encoder_workspace(_enc_desc(B, **bad)) == 0
