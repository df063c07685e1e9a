"""The allocation-free greedy choice (ws_argmax_rows_noalloc) against the
existing entry point: for the logits that ws_verify writes, the ids it
returns must equal ws_verify's own `target` output, on two calls in a row;
and on given logits it must equal the lowest-id maximum (torch.argmax) with
and without a suppression mask, at the 1024-row capacity and for a
vocabulary smaller than its 32 column chunks (empty chunks).

This file is collected last so that a run stopping at the first failure has
already run every other test; it builds its own decoder, so it also passes
alone in a fresh process."""
import numpy as np
import pytest
import torch

import synth
from gpu_common import dev_i32, small_shape

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import binding
    return binding


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_noalloc_argmax_matches_verify_targets_twice(B):
    from speculative_whisper_asr_gb300 import runtime as R

    s = small_shape("bf16", n_layers=2)
    tw = synth.target_weights(s, 41)
    As = [synth.encoder_states(s, 41, i, frames=96) for i in range(3)]
    dec = R.Decoder(s, tw, None, max_batch=3, max_frames=96)
    req = dec.slots([0, 1, 2])
    dec.cross_kv(req, torch.cat([dec.enc_tensor(a) for a in As]), [96] * 3)
    H = len(s.prompt)
    for call in range(2):
        dec.reset(req)
        block = dev_i32([s.prompt] * 3) if call == 0 else dev_i32(
            np.random.default_rng(call).integers(0, s.vocab, size=(3, H)))
        tgt = torch.full((3, H), -7, dtype=torch.int32, device="cuda")
        lg = torch.empty(3, H, s.vocab, device="cuda")
        dec.verify(req, block, dev_i32([H] * 3), tgt, lg)
        out = torch.full((3 * H,), -9, dtype=torch.int32, device="cuda")
        B.ws_argmax_rows_noalloc(lg.data_ptr(), 3 * H, s.vocab, None, out.data_ptr(), _stream())
        torch.cuda.synchronize()
        assert torch.equal(out.view(3, H), tgt), call
        # independent check of the same choice: lowest id among the maxima
        ref = lg.view(3 * H, s.vocab).argmax(dim=1).to(torch.int32)
        assert torch.equal(out, ref)
    with pytest.raises(B.WSError) as e:
        B.ws_argmax_rows_noalloc(lg.data_ptr(), 1025, s.vocab, None, out.data_ptr(), _stream())
    assert e.value.code == B.WS_EINVAL and "capacity" in B.ws_last_error()


@pytest.mark.parametrize("rows,vocab,suppressed", [(1024, 1000, False), (37, 20, False), (64, 5000, True),
                                                    (5, 31, True)])
def test_noalloc_argmax_given_logits_twice(B, rows, vocab, suppressed):
    g = torch.Generator(device="cpu").manual_seed(rows * 7 + vocab)
    z = torch.randn(rows, vocab, generator=g)
    z[:, ::7] = torch.round(z[:, ::7])                 # exact ties between ids
    z[0] = -0.0
    z[0, vocab // 2] = 0.0                             # a row whose maximum is 0 with both signs
    mask, ref_in = None, z.clone()
    if suppressed:
        # suppress every row's true argmax and every fifth id: the choice must move
        ids = set(z.argmax(dim=1).tolist()) | set(range(1, vocab, 5))
        words = np.zeros((vocab + 31) // 32, dtype=np.uint64)
        for v in ids:
            words[v >> 5] |= np.uint64(1) << np.uint64(v & 31)
        mask = torch.as_tensor(words.astype(np.uint32).view(np.int32), device="cuda")
        ref_in[:, sorted(ids)] = -float("inf")
    zd = z.cuda()
    zero_ties = (ref_in[0] == 0).nonzero()
    ref = ref_in.argmax(dim=1).to(torch.int32)
    if len(zero_ties) and ref_in[0].max() == 0:
        assert ref[0].item() == zero_ties[0].item()        # lowest id among +0 / -0
    for _ in range(2):
        out = torch.full((rows,), -9, dtype=torch.int32, device="cuda")
        B.ws_argmax_rows_noalloc(zd.data_ptr(), rows, vocab, 0 if mask is None else mask.data_ptr(),
                                 out.data_ptr(), _stream())
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), ref)
