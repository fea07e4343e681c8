"""Oracle for FP8 (e4m3) operands (test infrastructure only).

The e4m3 format (OCP 8-bit floating point, "E4M3"): 1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
m/8 * 2^-6; the code with exponent 15 and mantissa 7 is NaN; no infinities;
the largest finite magnitude is 448.

Row quantisation used by the FP8 forward: for a row x (fp32 values),
  amax = max |x|,  scale = amax / 448,  inv = 448 / amax  (fp32, rounded to
  nearest), q = e4m3(x * inv) rounded to nearest-even with results beyond
  448 clamped to 448; an all-zero row uses scale = inv = 1.
The dequantised value of code q in that row is decode(q) * scale.
"""
from __future__ import annotations

import numpy as np


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each e4m3 code (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


_POS_CODES = np.arange(0, 0x7F, dtype=np.uint8)          # 0 .. 126: the finite non-negatives
_POS_VALS = e4m3_decode(_POS_CODES)                       # ascending


def e4m3_encode_rne(x) -> np.ndarray:
    """Nearest e4m3 code of each value (ties to the even code, magnitudes
    above 448 clamped to 448; NaN -> 0x7F)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    i = np.clip(np.searchsorted(_POS_VALS, a, side="left"), 1, len(_POS_VALS) - 1)
    lo, hi = _POS_VALS[i - 1], _POS_VALS[i]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((_POS_CODES[i] & 1) == 0))
    code = np.where(pick_hi, _POS_CODES[i], _POS_CODES[i - 1]).astype(np.uint8)
    code = np.where(a == _POS_VALS[i - 1], _POS_CODES[i - 1], code).astype(np.uint8)
    code = np.where(np.signbit(x) & (code != 0), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize_rows_e4m3(x):
    """Per-row e4m3 quantisation (see the module docstring).  x: [R, H]
    array of fp32-representable values.  Returns (codes uint8 [R, H],
    scales float32 [R])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=1).astype(np.float32)
    zero = amax == 0
    safe = np.where(zero, np.float32(1), amax).astype(np.float32)
    scale = np.where(zero, np.float32(1), safe / np.float32(448)).astype(np.float32)
    inv = np.where(zero, np.float32(1), np.float32(448) / safe).astype(np.float32)
    y = (x * inv[:, None]).astype(np.float32)
    return e4m3_encode_rne(y), scale


def dequantize_rows_e4m3(codes, scales) -> np.ndarray:
    """float64 value of each quantised element: decode(q) * scale of its row."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]
