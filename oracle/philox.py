"""Philox4x32-10 counter-based generator — oracle side (test infrastructure only).

Written from the published definition: J. K. Salmon, M. A. Moraes,
R. O. Dror, D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
SC'11, §4 (the Philox S-box: two 32x32->64 multiplies per round, a Weyl key
schedule, 10 rounds for the 4x32 variant).  The CUDA library implements the
same published definition independently; the two share no code.

Counter discipline used by the decoding method (our choice; the pages only
say the drafter samples each candidate and the verifier accepts with
probability min(1, p/q), Whisper-Flash §3.1 and Appendix A.4):
  key     = (seed & 0xffffffff, seed >> 32)
  counter = (request slot, round & 0xffffffff, position j, purpose)
  purpose : 0 = draft sample, 1 = acceptance uniform, 2 = residual / bonus sample
  uniform = (word0 >> 8) * 2**-24  in [0, 1)
"""
from __future__ import annotations

import numpy as np

_M0 = 0xD2511F53
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF

PURPOSE_DRAFT = 0
PURPOSE_ACCEPT = 1
PURPOSE_RESIDUAL = 2


def philox4x32_10(ctr, key):
    """One block: ctr = 4 uint32, key = 2 uint32 -> 4 uint32 (Python ints)."""
    c0, c1, c2, c3 = (int(v) & _MASK for v in ctr)
    k0, k1 = (int(v) & _MASK for v in key)
    for _ in range(10):
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> 32, p0 & _MASK
        hi1, lo1 = p1 >> 32, p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & _MASK, lo1, (hi0 ^ c3 ^ k1) & _MASK, lo0
        k0 = (k0 + _W0) & _MASK
        k1 = (k1 + _W1) & _MASK
    return (c0, c1, c2, c3)


def uniform(seed: int, slot: int, rnd: int, j: int, purpose: int) -> np.float32:
    """The method's uniform in [0, 1) for one (request, round, position, purpose)."""
    key = (seed & _MASK, (seed >> 32) & _MASK)
    w0 = philox4x32_10((slot, rnd & _MASK, j, purpose), key)[0]
    return np.float32((w0 >> 8) * (1.0 / 16777216.0))
