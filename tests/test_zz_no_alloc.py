"""The allocation-free greedy choice (ws_argmax_rows_noalloc) against the
existing entry point: for the logits that ws_verify writes, the ids it
returns must equal ws_verify's own `target` output, on two calls in a row.

This file is collected last so that a run stopping at the first failure has
already run every other test; it builds its own decoder, so it also passes
alone in a fresh process."""
import numpy as np
import pytest
import torch

import synth
from gpu_common import dev_i32, small_shape

pytestmark = pytest.mark.gpu


def test_noalloc_argmax_matches_verify_targets_twice():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding as B
    from speculative_whisper_asr_gb300 import runtime as R

    s = small_shape("bf16", n_layers=2)
    tw = synth.target_weights(s, 41)
    As = [synth.encoder_states(s, 41, i, frames=96) for i in range(3)]
    dec = R.Decoder(s, tw, None, max_batch=3, max_frames=96)
    req = dec.slots([0, 1, 2])
    dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in As]), [96] * 3)
    stream = torch.cuda.current_stream().cuda_stream
    H = len(s.prompt)
    for call in range(2):
        dec.reset(req)
        block = dev_i32([s.prompt] * 3) if call == 0 else dev_i32(
            np.random.default_rng(call).integers(0, s.vocab, size=(3, H)))
        tgt = torch.full((3, H), -7, dtype=torch.int32, device="cuda")
        lg = torch.empty(3, H, s.vocab, device="cuda")
        dec.verify(req, block, dev_i32([H] * 3), tgt, lg)
        out = torch.full((3 * H,), -9, dtype=torch.int32, device="cuda")
        B.ws_argmax_rows_noalloc(lg.data_ptr(), 3 * H, s.vocab, None, out.data_ptr(), stream)
        torch.cuda.synchronize()
        assert torch.equal(out.view(3, H), tgt), call
        # independent check of the same choice: lowest id among the maxima
        ref = lg.view(3 * H, s.vocab).argmax(dim=1).to(torch.int32)
        assert torch.equal(out, ref)
    with pytest.raises(B.WSError) as e:
        B.ws_argmax_rows_noalloc(lg.data_ptr(), 1025, s.vocab, None, out.data_ptr(), stream)
    assert e.value.code == B.WS_EINVAL and "capacity" in B.ws_last_error()
