"""E4M3 codes of an 8-bit KV cache, from the format's definition (test
infrastructure only, like the rest of ``oracle``).

E4M3 (the "FN" variant of the 8-bit floating-point formats): one sign bit,
four exponent bits with bias 7, three mantissa bits.  Exponent field 0 holds
subnormals m/8 * 2^-6; fields 1..15 hold (1 + m/8) * 2^(e-7); field 15 with
mantissa 7 is NaN; there are no infinities, so the largest finite value is
1.75 * 2^8 = 448.

Encoding rounds to the nearest code, ties to the code with an even mantissa,
and saturates finite values beyond +-448 to +-448 (the "satfinite" rule).
A cache entry is code * scale with one fp32 scale per kv head (K and V have
their own); quantization divides by the scale in fp32 first.
"""
from __future__ import annotations

import numpy as np


def _positive_table() -> np.ndarray:
    """Values of the codes 0x00..0x7E (sign 0, finite), increasing."""
    vals = np.empty(127, np.float64)
    for c in range(127):
        e, m = c >> 3, c & 7
        vals[c] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_POS = _positive_table()
MAX_FINITE = float(_POS[-1])  # 448


def decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    mag = c & 0x7F
    out = np.where(mag == 0x7F, np.nan, _POS[np.minimum(mag, 126)])
    return np.where(c & 0x80, -out, out)


def encode(x) -> np.ndarray:
    """float values -> uint8 codes: round to nearest, ties to even mantissa,
    saturate beyond +-448, NaN -> 0x7F."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    # index of the largest table value <= a (the table starts at 0)
    lo = np.clip(np.searchsorted(_POS, a, side="right") - 1, 0, 126)
    hi = np.minimum(lo + 1, 126)
    d_lo, d_hi = a - _POS[lo], _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= MAX_FINITE, 126, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize(x, scale) -> np.ndarray:
    """Codes of x / scale, the division done in fp32 (as the append kernel does)."""
    y = np.asarray(x, np.float32) / np.float32(scale)
    return encode(y.astype(np.float32))


def dequantize(codes, scale) -> np.ndarray:
    """code * scale in float64."""
    return decode(codes) * float(np.float32(scale))
