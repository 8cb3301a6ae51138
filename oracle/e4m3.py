"""Exact FP8 E4M3 encode / decode -- test infrastructure.

Format facts used (stated on "4.3 FlashAttention 2 & 3: Work Partitioning,
Warp Specialization & FP8", section "Why FP8 attention is hard", and on
"FlashAttention-3: How Warp Specialization, Asynchronous TMA Tiling, and FP8
Hardware Acceleration Scale Attention on Hopper GPUs", section 4): one sign
bit, four exponent bits, three mantissa bits, largest finite magnitude 448.
The rest is the usual E4M3 ("fn") layout: exponent bias 7, exponent field 0
holds subnormals m/8 * 2^-6, there are no infinities, and S.1111.111 is NaN,
so exponent field 15 with mantissa 0..6 is a normal number.

Encoding rounds to the nearest representable value, ties to the even code
(even mantissa), keeps the sign of values that round to zero, and saturates
finite magnitudes above 448 to 448 (the "satfinite" behaviour).  NaN maps to
0x7F / 0xFF.
"""
from __future__ import annotations

import math

import numpy as np

MAX_FINITE = 448.0


def decode_code(code: int) -> float:
    """Value of one E4M3 code (0..255) from the bit fields."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.copysign(float("nan"), sign)
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# Magnitudes of the 127 non-negative finite codes 0x00..0x7E, ascending.
_POS = np.array([decode_code(c) for c in range(0x7F)], dtype=np.float64)
_DECODE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)


def decode(codes) -> np.ndarray:
    """Decode an array of uint8 codes to float64."""
    return _DECODE[np.asarray(codes, dtype=np.uint8)]


def encode(x) -> np.ndarray:
    """Round float64 values to E4M3 codes (uint8): RNE, saturating, signed zero."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, np.minimum(a, MAX_FINITE))
    # hi: first table entry >= a; lo: the entry below it.
    hi = np.searchsorted(_POS, a, side="left")
    hi = np.minimum(hi, _POS.size - 1)
    lo = np.maximum(hi - 1, 0)
    exact = _POS[hi] == a
    d_lo = a - _POS[lo]
    d_hi = _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(exact, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    code = np.where(neg, mag | 0x80, mag).astype(np.uint8)
    return np.where(nan, np.where(neg, 0xFF, 0x7F), code).astype(np.uint8)
