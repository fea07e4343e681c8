"""Pins for the e4m3 oracle (CPU only): decoding and round-to-nearest-even
encoding checked against PyTorch's float8_e4m3fn type (an independent
implementation of the same format), plus the quantiser's invariants."""
import numpy as np
import pytest
import torch

from oracle import dequantize_rows_e4m3, e4m3_decode, e4m3_encode_rne, quantize_rows_e4m3


def test_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = e4m3_decode(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert e4m3_decode([0x7E])[0] == 448.0 and e4m3_decode([0x01])[0] == 2.0 ** -9


def test_encode_rne_matches_torch_in_range():
    rng = np.random.default_rng(0)
    finite = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (finite[1:] + finite[:-1]) / 2                          # exact ties
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 5000),
                        finite, -finite, mids, -mids, [0.0, -0.0, 448.0]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3_encode_rne(x)
    same = (got == ref) | ((got & 0x7F) == 0) & ((ref & 0x7F) == 0)   # +0 / -0 both zero
    assert np.all(same), x[~same][:10]


def test_encode_saturates():
    assert e4m3_encode_rne([500.0, -1e9, 449.0])[:2].tolist() == [0x7E, 0xFE]
    assert e4m3_encode_rne([np.nan])[0] == 0x7F


def test_quantize_rows_roundtrip_and_amax():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((50, 96)) * rng.uniform(1e-3, 1e3, (50, 1))).astype(np.float32)
    x[7] = 0
    q, s = quantize_rows_e4m3(x)
    deq = dequantize_rows_e4m3(q, s)
    # the largest magnitude of every nonzero row lands on the top code 448
    for r in range(50):
        if r == 7:
            assert np.all(q[r] & 0x7F == 0) and s[r] == 1
            continue
        assert np.max(q[r] & 0x7F) == 0x7E
    # relative error of a normal e4m3 value is at most 2^-4
    big = np.abs(x) > np.abs(x).max(axis=1, keepdims=True) * 2.0 ** -6
    rel = np.abs(deq - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)


# ---------------------------------------------------------------- backward
#
# The e4m3 backward takes its d-logits from the logits the e4m3 forward
# computes (row-quantised operands) and projects them with the unquantised
# operands.  Three special cases pin it to the bf16 oracle, itself pinned by
# finite differences and closed forms:
#   both operands on the e4m3 grid (quantisation exact): the bf16 backward;
#   W on the grid: dHidden is the bf16 oracle's at hidden' = dequantised
#     hidden, and dW differs from that oracle's by dZ^T (hidden - hidden');
#   hidden on the grid: dW is the bf16 oracle's at W' = dequantised W, and
#     dHidden differs from that oracle's by dZ (W - W').
# Planted mistakes (logits from unquantised operands, projection with the
# quantised ones) fail these pins.

import oracle  # noqa: E402


def _grid_rows(rng, R, H):
    """Rows of values on the e4m3 grid, each holding +-448 so that its scale
    is 1 and quantisation returns every value unchanged."""
    codes = rng.integers(0, 0x7F, size=(R, H)).astype(np.uint8)          # finite codes
    codes |= (rng.integers(0, 2, size=(R, H)).astype(np.uint8) << 7)     # signs
    x = e4m3_decode(codes)
    x[:, 0] = np.where(rng.integers(0, 2, R) == 1, 448.0, -448.0)
    return x / 64.0 * 64.0                                               # exact


def _problem(seed, T=7, H=8, V=11, w_grid=False, h_grid=False):
    rng = np.random.default_rng(seed)
    hidden = _grid_rows(rng, T, H) / 256.0 if h_grid else rng.standard_normal((T, H)) * 0.7
    W = _grid_rows(rng, V, H) / 256.0 if w_grid else rng.standard_normal((V, H)) * 0.9
    # scaling a grid row by a power of two keeps it exactly quantisable (its
    # scale becomes that power of two)
    t = rng.integers(0, V, T)
    mask = np.ones(T, np.uint8)
    mask[2] = 0
    g_lp, g_h = rng.standard_normal(T), 0.5 * rng.standard_normal(T)
    return hidden, W, t, mask, g_lp, g_h


def _pin_exact(fn):
    hidden, W, t, mask, g_lp, g_h = _problem(1, w_grid=True, h_grid=True)
    assert np.array_equal(oracle.dequantized_rows(hidden), hidden)
    assert np.array_equal(oracle.dequantized_rows(W), W)
    dh, dW = fn(hidden, W, t, mask, g_lp, g_h)
    rdh, rdW = oracle.lmhead_backward(hidden, W, t, mask, g_lp, g_h)
    np.testing.assert_allclose(dh, rdh, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dW, rdW, rtol=1e-12, atol=1e-14)


def _pin_hidden_quantised(fn):
    hidden, W, t, mask, g_lp, g_h = _problem(2, w_grid=True)
    hq = oracle.dequantized_rows(hidden)
    assert not np.array_equal(hq, hidden)
    dh, dW = fn(hidden, W, t, mask, g_lp, g_h)
    rdh, rdW = oracle.lmhead_backward(hq, W, t, mask, g_lp, g_h)
    act = mask != 0
    dz = oracle.lmhead_dlogits_rows(hq[act], W, t[act], g_lp[act], g_h[act])
    np.testing.assert_allclose(dh, rdh, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dW, rdW + dz.T @ (hidden[act] - hq[act]), rtol=1e-12, atol=1e-14)


def _pin_weight_quantised(fn):
    hidden, W, t, mask, g_lp, g_h = _problem(3, h_grid=True)
    Wq = oracle.dequantized_rows(W)
    assert not np.array_equal(Wq, W)
    dh, dW = fn(hidden, W, t, mask, g_lp, g_h)
    rdh, rdW = oracle.lmhead_backward(hidden, Wq, t, mask, g_lp, g_h)
    act = mask != 0
    dz = oracle.lmhead_dlogits_rows(hidden[act], Wq, t[act], g_lp[act], g_h[act])
    np.testing.assert_allclose(dW, rdW, rtol=1e-12, atol=1e-14)
    exp_dh = rdh.copy()
    exp_dh[act] += dz @ (W - Wq)
    np.testing.assert_allclose(dh, exp_dh, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("pin", [_pin_exact, _pin_hidden_quantised, _pin_weight_quantised])
def test_e4m3_backward_pins(pin):
    pin(oracle.lmhead_backward_e4m3)


def _mistake(kind):
    """The e4m3 backward with one plausible mistake planted."""
    def fn(hidden, W, t, mask, g_lp, g_h):
        h, Wf = np.asarray(hidden, float), np.asarray(W, float)
        hq, Wq = oracle.dequantized_rows(h), oracle.dequantized_rows(Wf)
        act = np.asarray(mask) != 0
        zh, zw = (h, Wf) if kind == "logits_unquantised" else (hq, Wq)
        dz = oracle.lmhead_dlogits_rows(zh[act], zw, t[act], g_lp[act], g_h[act])
        dh = np.zeros_like(h)
        dh[act] = dz @ (Wq if kind == "project_with_quantised" else Wf)
        dW = dz.T @ (hq[act] if kind == "project_with_quantised" else h[act])
        return dh, dW
    return fn


@pytest.mark.parametrize("kind", ["logits_unquantised", "project_with_quantised"])
def test_e4m3_backward_pins_reject_planted_mistakes(kind):
    caught = 0
    for pin in (_pin_exact, _pin_hidden_quantised, _pin_weight_quantised):
        try:
            pin(_mistake(kind))
        except AssertionError:
            caught += 1
    assert caught >= 1
    # the unmutated composition passes all three
    for pin in (_pin_exact, _pin_hidden_quantised, _pin_weight_quantised):
        pin(_mistake("none"))
