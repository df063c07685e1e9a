"""CPU oracle of the Whisper audio encoder: the step before the decoding path.

TEST INFRASTRUCTURE.  Only tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does, and
this module never imports the product path.

Why it is here: once speculation removes most decoder calls, the fixed
encoder cost becomes visible (Whisper-Flash App. B.2, Table A2: 15-34% of
request time at batch one, about half at batch 32 and 96), so the encoder
runs on the GPU too and needs an oracle of its own.

The pages name the encoder and its output A but do not print its layers;
this restates the published Whisper audio encoder, the plainest reading:

  conv1   1-D convolution n_mels -> d, kernel 3, stride 1, padding 1, + bias, GELU
  conv2   1-D convolution d -> d, kernel 3, stride 2, padding 1, + bias, GELU
          (2F mel frames -> F positions, 20 ms each)
  + P     sinusoidal positions: P[t, i] = sin(t w_i), P[t, d/2 + i] = cos(t w_i),
          w_i = 10000^(-i / (d/2 - 1)), i < d/2
  blocks  n_layers pre-LN blocks over all F positions (no mask):
          x += W_o MHA(LN1(x)) + b_o,  x += W_2 GELU(W_1 LN2(x) + b_1) + b_2
          (biases on q, v, o, fc1, fc2; none on k; scale 1/sqrt(64); exact-erf GELU)
  LN_p    a final layer norm; its output is A [F, d].

Floating point: fp64.  With bf16=True values are rounded (nearest even) to
bf16 where the GPU path stores them: the mel input, both convolution outputs,
LN outputs, q / k / v, the attention output, the GELU output and the encoder
output; the residual stream, softmax and accumulations stay fp64.

Pins (tests/test_oracle.py): the whole fp64 encoder against torch's conv1d,
TransformerEncoderLayer (norm_first) and layer_norm with the same weights;
the position table's closed forms.
"""
from __future__ import annotations

import math

import numpy as np

from .model import gelu, layer_norm, mha, round_bf16


def sinusoids(length: int, channels: int) -> np.ndarray:
    """Position table [length, channels]: sines of t w_i in the first half,
    cosines in the second, w_i geometric from 1 down to 1/10000."""
    half = channels // 2
    w = np.exp(-np.arange(half) * (math.log(10000.0) / (half - 1)))
    t = np.arange(length)[:, None] * w[None, :]
    return np.concatenate([np.sin(t), np.cos(t)], axis=1)


def conv1d(x: np.ndarray, w: np.ndarray, b: np.ndarray, stride: int) -> np.ndarray:
    """x [C_in, T], w [C_out, C_in, 3], padding 1 -> [C_out, T_out]:
    out[:, t] = b + sum_k w[:, :, k] x[:, stride t + k - 1] (zeros outside)."""
    C_in, T = x.shape
    T_out = (T + 2 - 3) // stride + 1
    xp = np.zeros((C_in, T + 2))
    xp[:, 1:T + 1] = x
    out = np.repeat(np.asarray(b, dtype=np.float64)[:, None], T_out, axis=1)
    for k in range(3):
        out += w[:, :, k] @ xp[:, k:k + stride * (T_out - 1) + 1:stride]
    return out


class Encoder:
    """Weights from synth.encoder_weights (float arrays), shape an EncoderShape."""

    def __init__(self, shape, weights: dict, bf16: bool | None = None):
        self.s = shape
        self.w = {k: np.asarray(v, dtype=np.float64) for k, v in weights.items()}
        self.bf16 = (shape.dtype == "bf16") if bf16 is None else bf16
        self.H = shape.n_heads

    def rb(self, x):
        return round_bf16(x) if self.bf16 else x

    def stem(self, mel: np.ndarray) -> np.ndarray:
        """[n_mels, 2F] -> residual stream [F, d] (convolutions, GELU, + P)."""
        w = self.w
        h = self.rb(gelu(conv1d(self.rb(np.asarray(mel, dtype=np.float64)), w["conv1_w"], w["conv1_b"], 1)))
        h = self.rb(gelu(conv1d(h, w["conv2_w"], w["conv2_b"], 2)))
        x = h.T
        return x + sinusoids(x.shape[0], x.shape[1])

    def block(self, x: np.ndarray, l: int) -> np.ndarray:
        w, p, d = self.w, f"layers.{l}.", self.s.d_model
        h = self.rb(layer_norm(x, w[p + "ln1_g"], w[p + "ln1_b"]))
        qkv = h @ w[p + "w_qkv"].T
        q = self.rb(qkv[:, :d] + w[p + "b_q"])
        k = self.rb(qkv[:, d:2 * d])
        v = self.rb(qkv[:, 2 * d:] + w[p + "b_v"])
        o = self.rb(mha(q, k, v, self.H))
        x = x + (o @ w[p + "w_o"].T + w[p + "b_o"])
        h2 = self.rb(layer_norm(x, w[p + "ln2_g"], w[p + "ln2_b"]))
        f = self.rb(gelu(h2 @ w[p + "w_fc1"].T + w[p + "b_fc1"]))
        return x + (f @ w[p + "w_fc2"].T + w[p + "b_fc2"])

    def encode(self, mel: np.ndarray, n_layers: int | None = None) -> np.ndarray:
        """Encoder output A [F, d] of one window (the first n_layers blocks
        when given)."""
        x = self.stem(mel)
        for l in range(self.s.n_layers if n_layers is None else n_layers):
            x = self.block(x, l)
        return self.rb(layer_norm(x, self.w["lnp_g"], self.w["lnp_b"]))
