"""Oracle for the fused LM-head forward and backward (test infrastructure only).

Source: "perf(megatron): add block-sparse fused LM-head backward" (SkyRL PR
#2376).  "What does this PR do?" / "How it works": the forward returns the
target log-probability (and, from the entropy layer #2374 it builds on, the
softmax entropy) for tokens the loss mask marks active; the backward builds
d-logits only for active tiles and projects them to dHidden and dW.  The page
prints no formulas; the ones below are the textbook definitions it names:

  z      = W h                       (logits, W is [V, H] as in nn.Linear)
  lse    = max(z) + log sum_v exp(z_v - max(z))
  logp   = z_t - lse                 (t = target token)
  p      = exp(z - lse)              (softmax)
  H      = lse - sum_v p_v z_v       (= -sum_v p_v log p_v)

and, for the loss L = sum_i mask_i (g_lp,i logp_i + g_H,i H_i):

  dL/dz  = g_lp (onehot(t) - p) - g_H p (z - lse + H)
  dHidden = dZ W,   dW = dZ^T hidden.

Rows whose mask bit is 0 get logp = H = lse = 0 and a zero gradient row,
chosen by selection, never by multiplying (so NaN/Inf in g on those rows
cannot leak).  Everything is float64; matmul is NumPy's.  Rows are processed
in blocks only to bound memory; blocking changes nothing in the arithmetic
of a row.
"""
from __future__ import annotations

import numpy as np

_BLOCK = 256


def _as64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def lmhead_forward_rows(h_rows, W, t_rows):
    """logp, entropy, lse of the given rows (all treated as active)."""
    h_rows, W = _as64(h_rows), _as64(W)
    t_rows = np.asarray(t_rows, dtype=np.int64)
    z = h_rows @ W.T
    zmax = z.max(axis=1, keepdims=True)
    lse = zmax[:, 0] + np.log(np.exp(z - zmax).sum(axis=1))
    p = np.exp(z - lse[:, None])
    ent = lse - (p * z).sum(axis=1)
    logp = z[np.arange(z.shape[0]), t_rows] - lse
    return logp, ent, lse


def lmhead_dlogits_rows(h_rows, W, t_rows, g_lp_rows, g_h_rows):
    """d-logits dL/dz of the given rows (all treated as active), shape [n, V]."""
    h_rows, W = _as64(h_rows), _as64(W)
    t_rows = np.asarray(t_rows, dtype=np.int64)
    g_lp_rows, g_h_rows = _as64(g_lp_rows), _as64(g_h_rows)
    z = h_rows @ W.T
    zmax = z.max(axis=1, keepdims=True)
    lse = zmax[:, 0] + np.log(np.exp(z - zmax).sum(axis=1))
    p = np.exp(z - lse[:, None])
    ent = lse - (p * z).sum(axis=1)
    onehot = np.zeros_like(z)
    onehot[np.arange(z.shape[0]), t_rows] = 1.0
    dz = g_lp_rows[:, None] * (onehot - p) \
        - g_h_rows[:, None] * p * (z - lse[:, None] + ent[:, None])
    return dz


def lmhead_forward(hidden, W, targets, mask, block: int = _BLOCK):
    """logp, entropy, lse for every token; zero where mask == 0."""
    hidden = _as64(hidden)
    mask = np.asarray(mask).reshape(-1) != 0
    T = hidden.shape[0]
    logp, ent, lse = (np.zeros(T) for _ in range(3))
    act = np.flatnonzero(mask)
    for b in range(0, len(act), block):
        r = act[b:b + block]
        lp_b, h_b, l_b = lmhead_forward_rows(hidden[r], W, np.asarray(targets)[r])
        logp[r], ent[r], lse[r] = lp_b, h_b, l_b
    return logp, ent, lse


def lmhead_backward(hidden, W, targets, mask, g_lp, g_h, block: int = _BLOCK):
    """dHidden [T, H] and dW [V, H] of L; rows with mask == 0 contribute nothing."""
    hidden, W = _as64(hidden), _as64(W)
    mask = np.asarray(mask).reshape(-1) != 0
    dhidden = np.zeros_like(hidden)
    dW = np.zeros_like(W)
    act = np.flatnonzero(mask)
    for b in range(0, len(act), block):
        r = act[b:b + block]
        dz = lmhead_dlogits_rows(hidden[r], W, np.asarray(targets)[r],
                                 np.asarray(g_lp)[r], np.asarray(g_h)[r])
        dhidden[r] = dz @ W
        dW += dz.T @ hidden[r]
    return dhidden, dW


def lmhead_backward_rows_weighted(hidden_rows, W, t_rows, g_lp_rows, g_h_rows,
                                  block: int = _BLOCK):
    """dHidden rows and the dW contribution sum_r dZ_r^T h_r of a row subset.

    When g_lp and g_H vanish on every other row, this subset's contribution is
    the whole of dW, so it can be checked at any problem size."""
    hidden_rows, W = _as64(hidden_rows), _as64(W)
    dh = np.zeros_like(hidden_rows)
    dW = np.zeros_like(W)
    n = hidden_rows.shape[0]
    for b in range(0, n, block):
        sl = slice(b, min(n, b + block))
        dz = lmhead_dlogits_rows(hidden_rows[sl], W, np.asarray(t_rows)[sl],
                                 np.asarray(g_lp_rows)[sl], np.asarray(g_h_rows)[sl])
        dh[sl] = dz @ W
        dW += dz.T @ hidden_rows[sl]
    return dh, dW


def loss_value(hidden, W, targets, mask, g_lp, g_h) -> float:
    """L = sum over active rows of g_lp * logp + g_H * entropy (float64)."""
    logp, ent, _ = lmhead_forward(hidden, W, targets, mask)
    m = np.asarray(mask).reshape(-1) != 0
    return float(np.sum(np.where(m, _as64(g_lp) * logp + _as64(g_h) * ent, 0.0)))
