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


# ----------------------------------------------------------------------------
# Backward of the e4m3 forward
#
# The pages give no FP8 backward; this is the reading the e4m3 training path
# implements.  The d-logits are those of the logits the e4m3 forward computes
# (z' = hq Wq^T with the row-dequantised operands hq, Wq), so they agree with
# the lse and entropy that forward returned; they are then projected with the
# unquantised operands, as the bf16 backward does:
#   dZ' = g_lp (onehot(t) - p') - g_H p' (z' - lse' + H'),  p' = softmax(z'),
#   dHidden = dZ' W,   dW = dZ'^T hidden.
# Rows with mask 0 contribute nothing.
# ----------------------------------------------------------------------------

def dequantized_rows(x) -> np.ndarray:
    """float64 values the e4m3 path computes with for a [R, H] operand:
    per-row quantised (quantize_rows_e4m3) and dequantised."""
    return dequantize_rows_e4m3(*quantize_rows_e4m3(np.asarray(x, dtype=np.float32)))


def lmhead_backward_e4m3_rows_weighted(hidden_rows, W, Wq, t_rows, g_lp_rows, g_h_rows,
                                       block: int = 256):
    """dHidden rows and the dW contribution of a row subset under the reading
    above; Wq = dequantized_rows(W) is passed in so that large W is quantised
    once.  hidden_rows and W are the unquantised values."""
    from .lmhead import lmhead_dlogits_rows
    h = np.asarray(hidden_rows, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    hq = dequantized_rows(h)
    dh = np.zeros_like(h)
    dW = np.zeros_like(W)
    n = h.shape[0]
    for b in range(0, n, block):
        sl = slice(b, min(n, b + block))
        dz = lmhead_dlogits_rows(hq[sl], Wq, np.asarray(t_rows)[sl],
                                 np.asarray(g_lp_rows)[sl], np.asarray(g_h_rows)[sl])
        dh[sl] = dz @ W
        dW += dz.T @ h[sl]
    return dh, dW


def lmhead_backward_e4m3(hidden, W, targets, mask, g_lp, g_h):
    """dHidden [T, H] and dW [V, H] of the e4m3 path (reading above)."""
    hidden = np.asarray(hidden, dtype=np.float64)
    act = np.flatnonzero(np.asarray(mask).reshape(-1) != 0)
    dhidden = np.zeros_like(hidden)
    Wq = dequantized_rows(W)
    dh, dW = lmhead_backward_e4m3_rows_weighted(hidden[act], W, Wq, np.asarray(targets)[act],
                                                np.asarray(g_lp)[act], np.asarray(g_h)[act])
    dhidden[act] = dh
    return dhidden, dW
