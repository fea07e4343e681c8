"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case patches one plausible error into the oracle's d-logits or forward
(a dropped entropy term, a flipped sign, a wrong target index, a transposed
weight) and checks that the finite-difference or closed-form pin rejects it.
"""
import numpy as np
import pytest
import scipy.special

import oracle.lmhead as L
from test_oracle_lmhead import fd_grad, rand_problem


def _dlogits_variant(kind):
    def f(h_rows, W, t_rows, g_lp_rows, g_h_rows):
        h_rows, W = np.asarray(h_rows, float), np.asarray(W, float)
        z = h_rows @ W.T
        lse = scipy.special.logsumexp(z, axis=1)
        p = np.exp(z - lse[:, None])
        ent = lse - (p * z).sum(axis=1)
        onehot = np.zeros_like(z)
        tt = np.asarray(t_rows)
        if kind == "target_off_by_one":
            tt = (tt + 1) % z.shape[1]
        onehot[np.arange(z.shape[0]), tt] = 1.0
        ent_term = p * (z - lse[:, None] + ent[:, None])
        if kind == "drop_entropy_term":
            ent_term = 0 * ent_term
        if kind == "entropy_sign":
            ent_term = -ent_term
        lp_term = onehot - p
        if kind == "nll_sign":
            lp_term = -lp_term
        return np.asarray(g_lp_rows)[:, None] * lp_term - np.asarray(g_h_rows)[:, None] * ent_term
    return f


@pytest.mark.parametrize("kind", ["target_off_by_one", "drop_entropy_term",
                                  "entropy_sign", "nll_sign"])
def test_fd_pin_rejects_planted_dlogits_mistake(kind, monkeypatch):
    hidden, W, t, mask, g_lp, g_h = rand_problem(T=5, H=4, V=7, scale=1.5, seed=3,
                                                 inactive=(1,))
    fd = fd_grad(lambda: L.loss_value(hidden, W, t, mask, g_lp, g_h), W, eps=1e-5)
    monkeypatch.setattr(L, "lmhead_dlogits_rows", _dlogits_variant(kind))
    _, dW = L.lmhead_backward(hidden, W, t, mask, g_lp, g_h)
    assert not np.allclose(dW, fd, rtol=1e-6, atol=5e-7)
    monkeypatch.undo()
    _, dW = L.lmhead_backward(hidden, W, t, mask, g_lp, g_h)
    np.testing.assert_allclose(dW, fd, rtol=1e-6, atol=5e-7)


def test_scipy_pin_rejects_transposed_weight():
    rng = np.random.default_rng(0)
    H = V = 6
    hidden = rng.standard_normal((3, H))
    W = rng.standard_normal((V, H))
    t = np.array([0, 3, 5])
    lp_wrong, _, _ = L.lmhead_forward_rows(hidden, W.T, t)
    lp_right, _, _ = L.lmhead_forward_rows(hidden, W, t)
    ref = np.array([scipy.special.log_softmax(W @ hidden[i])[t[i]] for i in range(3)])
    assert not np.allclose(lp_wrong, ref, atol=1e-6)
    np.testing.assert_allclose(lp_right, ref, atol=1e-12)
