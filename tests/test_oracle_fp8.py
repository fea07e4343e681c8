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
