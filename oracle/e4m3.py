"""FP8 E4M3 (the ``float8_e4m3fn`` format) decoded from its bit definition.

Code layout: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
Exponent 0 is subnormal: (m / 8) * 2**-6. The all-ones code S.1111.111 is NaN;
the format has no infinity, so its largest finite magnitude is
(1 + 6/8) * 2**8 = 448. Query and cache are stored in this format
(drafter-attention page, ``cake_supported``: FP8 query and cache).
"""
from __future__ import annotations

import math

import numpy as np


def decode_code(c: int) -> float:
    """One E4M3 code (0..255) -> its real value (NaN for the two NaN codes)."""
    sign = -1.0 if c & 0x80 else 1.0
    e = (c >> 3) & 0xF
    m = c & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)
NAN_CODES = (0x7F, 0xFF)


def decode(codes) -> np.ndarray:
    """Array of uint8 E4M3 codes -> float64 values (same shape).

    Inputs never carry NaN codes (the generator clips before casting); the
    oracle refuses them rather than propagate NaN silently.
    """
    a = np.asarray(codes)
    if a.dtype != np.uint8:
        raise TypeError("E4M3 codes must be uint8")
    if np.isin(a, NAN_CODES).any():
        raise ValueError("E4M3 NaN code in the input")
    return TABLE[a]
