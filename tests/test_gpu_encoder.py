"""GPU parity for the audio encoder (the step before the decoding path,
Whisper-Flash App. B.2): tcgen05 GEMMs for both convolutions and every
projection, the flash-attention kernel, layer norms, against the
bf16-emulating oracle encoder, element by element (2e-2 of the row's
largest value, the bf16 tolerance)."""
import numpy as np
import pytest
import torch

import synth
from oracle import encoder as ENC
from gpu_common import logits_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    import __graft_entry__ as g
    g.build()
    from speculative_whisper_asr_gb300 import runtime
    return runtime


def _run(R, shape, seed, n):
    w = synth.encoder_weights(shape, seed)
    mels = [synth.mel_input(shape, seed, i) for i in range(n)]
    enc = R.Encoder(shape, w, max_batch=n)
    out = enc.encode(enc.mel_tensor(mels))
    torch.cuda.synchronize()
    assert enc.status() == 0
    return w, mels, out.float().cpu().numpy()


def test_tiny_encoder_three_windows_vs_oracle(R):
    """Tiny Whisper encoder shape (4 layers, d 384, 80 mels, 1500 frames), three
    windows in one call (4,500 rows: the layer norms take their many-row
    kernel): each window equals the oracle's encoding of it."""
    s = synth.ENC_TINY
    w, mels, got = _run(R, s, 7, 3)
    orc = ENC.Encoder(s, w)
    for i in range(3):
        logits_close(got[i], orc.encode(mels[i]), 2e-2)


def test_short_windows_key_tiles_cross_window_boundaries(R):
    """100-frame windows (200 mel frames): the second key tile of window 0
    holds window 1's first rows, which must stay masked; three windows, the
    last one's tile runs past the matrix."""
    s = synth.EncoderShape("tiny-encoder-100", 2, 384, 6, 1536, 80, n_frames=100)
    w, mels, got = _run(R, s, 8, 3)
    orc = ENC.Encoder(s, w)
    for i in range(3):
        logits_close(got[i], orc.encode(mels[i]), 2e-2)


def test_large_v3_width_two_layers_vs_oracle(R):
    """Large-v3 widths at full size (d 1280, 20 heads, FFN 5120, 128 mels,
    3000 -> 1500 frames) with the first two blocks: the stem GEMMs (K = 384
    and 3840), the 1500-key attention and the 5120-wide FFN against the
    oracle."""
    s = synth.EncoderShape("large-v3-encoder-2l", 2, 1280, 20, 5120, 128)
    w, mels, got = _run(R, s, 9, 1)
    logits_close(got[0], ENC.Encoder(s, w).encode(mels[0]), 2e-2)


def test_tcgen05_and_legacy_attention_agree_with_oracle(R):
    """The tcgen05 flash attention (default) and the legacy mma.sync kernel
    both match the oracle on two 100-frame windows (key tiles of 64 and 128
    query rows cross the windows' ends)."""
    s = synth.EncoderShape("tiny-encoder-100", 2, 384, 6, 1536, 80, n_frames=100)
    w = synth.encoder_weights(s, 12)
    mels = [synth.mel_input(s, 12, i) for i in range(2)]
    enc = R.Encoder(s, w, max_batch=2)
    mel = enc.mel_tensor(mels)
    outs = []
    for tc in (True, False):
        enc.set_attention(tc)
        outs.append(enc.encode(mel).float().cpu().numpy())
    assert enc.status() == 0
    orc = ENC.Encoder(s, w)
    for i in range(2):
        ref = orc.encode(mels[i])
        logits_close(outs[0][i], ref, 2e-2)
        logits_close(outs[1][i], ref, 2e-2)
