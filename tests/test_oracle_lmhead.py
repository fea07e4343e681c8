"""Pins for the LM-head oracle (CPU only).

Each check is tied to something other than the oracle's own formula:
central finite differences of the loss (gradients), SciPy's log_softmax and
entropy routines (forward), closed forms for degenerate weights, and
invariants of the softmax.  The functions checked follow the textbook
definitions that "perf(megatron): add block-sparse fused LM-head backward"
(SkyRL PR #2376) names: target log-probability, softmax entropy and their
gradients through d-logits, restricted to rows the loss mask marks active.
"""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

from oracle import (lmhead_backward, lmhead_backward_rows_weighted,
                    lmhead_dlogits_rows, lmhead_forward, loss_value)


def rand_problem(T=7, H=5, V=11, scale=1.0, seed=0, inactive=(1, 4)):
    rng = np.random.default_rng(seed)
    hidden = rng.standard_normal((T, H)) * scale
    W = rng.standard_normal((V, H)) * scale
    targets = rng.integers(0, V, T)
    mask = np.ones(T, np.uint8)
    mask[list(inactive)] = 0
    g_lp = rng.standard_normal(T)
    g_h = rng.standard_normal(T) * 0.7
    return hidden, W, targets, mask, g_lp, g_h


def test_forward_matches_scipy():
    hidden, W, targets, mask, *_ = rand_problem(T=9, H=6, V=17, scale=1.3, seed=1)
    lp, ent, lse = lmhead_forward(hidden, W, targets, mask)
    for i in range(len(mask)):
        if not mask[i]:
            assert lp[i] == 0 and ent[i] == 0 and lse[i] == 0
            continue
        z = W @ hidden[i]
        ls = scipy.special.log_softmax(z)
        assert lp[i] == pytest.approx(ls[targets[i]], abs=1e-12)
        assert ent[i] == pytest.approx(scipy.stats.entropy(scipy.special.softmax(z)), abs=1e-12)
        assert lse[i] == pytest.approx(scipy.special.logsumexp(z), abs=1e-12)


def test_identity_weight_is_log_softmax_of_hidden():
    rng = np.random.default_rng(3)
    V = 13
    hidden = rng.standard_normal((4, V)) * 3
    W = np.eye(V)
    t = rng.integers(0, V, 4)
    lp, ent, _ = lmhead_forward(hidden, W, t, np.ones(4))
    for i in range(4):
        z = hidden[i]
        lse = max(z) + math.log(math.fsum(math.exp(v - max(z)) for v in z))
        assert lp[i] == pytest.approx(z[t[i]] - lse, abs=1e-12)
        p = [math.exp(v - lse) for v in z]
        assert ent[i] == pytest.approx(-math.fsum(pi * math.log(pi) for pi in p), abs=1e-12)


@pytest.mark.parametrize("V", [1, 2, 7, 1024])
def test_identical_rows_closed_form(V):
    rng = np.random.default_rng(V)
    H = 8
    c = rng.standard_normal(H)
    W = np.tile(c, (V, 1))
    hidden = rng.standard_normal((5, H))
    t = rng.integers(0, V, 5)
    g_lp, g_h = rng.standard_normal(5), rng.standard_normal(5)
    lp, ent, lse = lmhead_forward(hidden, W, t, np.ones(5))
    np.testing.assert_allclose(lp, -math.log(V), atol=1e-12)
    np.testing.assert_allclose(ent, math.log(V), atol=1e-12)
    np.testing.assert_allclose(lse, hidden @ c + math.log(V), atol=1e-12)
    # d-logits reduce to g_lp (onehot - 1/V); the entropy term vanishes
    dz = lmhead_dlogits_rows(hidden, W, t, g_lp, g_h)
    expect = -np.tile(g_lp[:, None] / V, (1, V))
    expect[np.arange(5), t] += g_lp
    np.testing.assert_allclose(dz, expect, atol=1e-12)


def test_zero_weight():
    V = 50
    lp, ent, lse = lmhead_forward(np.ones((3, 4)), np.zeros((V, 4)), [0, 7, 49], np.ones(3))
    np.testing.assert_allclose(lp, -math.log(V), atol=1e-13)
    np.testing.assert_allclose(ent, math.log(V), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(V), atol=1e-13)


def test_two_way_logistic():
    rng = np.random.default_rng(5)
    hidden = rng.standard_normal((6, 3)) * 2
    W = rng.standard_normal((2, 3))
    t = np.array([0, 1, 0, 1, 1, 0])
    lp, ent, _ = lmhead_forward(hidden, W, t, np.ones(6))
    for i in range(6):
        z = W @ hidden[i]
        d = z[t[i]] - z[1 - t[i]]
        assert lp[i] == pytest.approx(-math.log1p(math.exp(-d)), abs=1e-12)
        q = 1 / (1 + math.exp(-(z[0] - z[1])))
        assert ent[i] == pytest.approx(-(q * math.log(q) + (1 - q) * math.log(1 - q)), abs=1e-12)


def test_shift_invariance():
    hidden, W, t, mask, g_lp, g_h = rand_problem(seed=9, scale=1.5)
    c = np.random.default_rng(1).standard_normal(W.shape[1])
    lp0, ent0, lse0 = lmhead_forward(hidden, W, t, mask)
    lp1, ent1, lse1 = lmhead_forward(hidden, W + c, t, mask)
    np.testing.assert_allclose(lp1, lp0, atol=1e-12)
    np.testing.assert_allclose(ent1, ent0, atol=1e-12)
    np.testing.assert_allclose(lse1 - lse0, np.where(mask != 0, hidden @ c, 0), atol=1e-12)
    dh0, _ = lmhead_backward(hidden, W, t, mask, g_lp, g_h)
    dh1, _ = lmhead_backward(hidden, W + c, t, mask, g_lp, g_h)
    np.testing.assert_allclose(dh1, dh0, atol=1e-12)


def test_dlogits_rows_sum_to_zero():
    hidden, W, t, mask, g_lp, g_h = rand_problem(T=12, V=31, seed=4, scale=2.0)
    dz = lmhead_dlogits_rows(hidden, W, t, g_lp, g_h)
    np.testing.assert_allclose(dz.sum(axis=1), 0, atol=1e-12)


def fd_grad(f, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + eps
        fp = f()
        x[i] = old - eps
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * eps)
    return g


@pytest.mark.parametrize("scale,seed", [(0.5, 0), (1.5, 1), (3.0, 2)])
def test_gradients_match_finite_differences(scale, seed):
    hidden, W, t, mask, g_lp, g_h = rand_problem(T=6, H=5, V=9, scale=scale, seed=seed,
                                                 inactive=(2,))
    dh, dW = lmhead_backward(hidden, W, t, mask, g_lp, g_h)

    def L():
        return loss_value(hidden, W, t, mask, g_lp, g_h)

    # step 1e-5: truncation error ~1e-10 * L''' while the rounding error of L
    # (|L| ~ 1e2 at scale 3) stays ~1e-13 / 1e-5; any dropped term or flipped
    # sign moves entries by ~1e-2 or more.
    fd_h = fd_grad(L, hidden, eps=1e-5)
    fd_W = fd_grad(L, W, eps=1e-5)
    np.testing.assert_allclose(dh, fd_h, rtol=1e-6, atol=5e-7)
    np.testing.assert_allclose(dW, fd_W, rtol=1e-6, atol=5e-7)


def test_entropy_only_and_logprob_only_gradients():
    """Each of the two terms of dZ checked on its own against finite differences."""
    hidden, W, t, mask, g_lp, g_h = rand_problem(T=4, H=3, V=6, scale=2.0, seed=8,
                                                 inactive=())
    for glp, gh in ((g_lp, 0 * g_h), (0 * g_lp, g_h)):
        dh, dW = lmhead_backward(hidden, W, t, mask, glp, gh)
        fd = fd_grad(lambda: loss_value(hidden, W, t, mask, glp, gh), W)
        np.testing.assert_allclose(dW, fd, rtol=1e-6, atol=1e-8)


def test_inactive_rows_zero_even_with_nan_upstream():
    hidden, W, t, mask, g_lp, g_h = rand_problem(seed=12)
    g_lp = g_lp.copy()
    g_h = g_h.copy()
    g_lp[mask == 0] = np.nan
    g_h[mask == 0] = np.inf
    dh, dW = lmhead_backward(hidden, W, t, mask, g_lp, g_h)
    assert np.all(dh[mask == 0] == 0)
    assert np.all(np.isfinite(dW))
    lp, ent, lse = lmhead_forward(hidden, W, t, mask)
    assert np.all(lp[mask == 0] == 0) and np.all(ent[mask == 0] == 0)


def test_row_subset_contribution_equals_full_when_g_vanishes_elsewhere():
    hidden, W, t, mask, g_lp, g_h = rand_problem(T=20, H=6, V=14, seed=21, inactive=(3, 9))
    sub = np.array([0, 5, 11, 19])
    gl = np.zeros_like(g_lp)
    gh = np.zeros_like(g_h)
    gl[sub], gh[sub] = g_lp[sub], g_h[sub]
    dh_full, dW_full = lmhead_backward(hidden, W, t, mask, gl, gh)
    dh_sub, dW_sub = lmhead_backward_rows_weighted(hidden[sub], W, t[sub], g_lp[sub], g_h[sub])
    np.testing.assert_allclose(dW_sub, dW_full, atol=1e-12)
    np.testing.assert_allclose(dh_sub, dh_full[sub], atol=1e-12)
