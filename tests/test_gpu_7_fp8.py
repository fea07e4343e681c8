"""e4m3 (FP8) operands: the device quantiser must give the oracle's codes and
scales bit for bit, and the FP8 forward must match the fp64 oracle run on the
dequantised operands (the quantisation itself is the oracle's, so the only
difference left is fp32 accumulation) within the forward tolerance."""
import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import workloads as W
from gpu_helpers import BF16_TOL, small_inputs, to_dev
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_quantizer_bit_exact(dtype):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((300, 384)) * rng.uniform(1e-4, 1e4, (300, 1))).astype(np.float32)
    x[5] = 0
    x[9, 17] = -x[9].__abs__().max() * 3                  # a negative amax
    if dtype == "bf16":
        bits = W.f32_to_bf16_bits(x)
        xd = to_dev(bits)
        x = W.bf16_bits_to_f32(bits)
    else:
        xd = to_dev(x)
    q, s = eas.quantize_rows_e4m3(xd)
    rq, rs = oracle.quantize_rows_e4m3(x)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("T,H,V,w_std", [(700, 256, 1000, 3.0), (300, 128, 257, 8.0),
                                         (2048, 512, 5000, 2.0)])
def test_fp8_forward_matches_oracle(T, H, V, w_std):
    inp = small_inputs(T, H, V, seed=T + H, mask_kind="bernoulli0.6", w_std=w_std)
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    h8, hs = eas.quantize_rows_e4m3(h)
    w8, wsc = eas.quantize_rows_e4m3(w)
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd_fp8(h8, hs, w8, wsc, t, m, spans, ns)
    hq = oracle.dequantize_rows_e4m3(h8.cpu().numpy(), hs.cpu().numpy())
    wq = oracle.dequantize_rows_e4m3(w8.cpu().numpy(), wsc.cpu().numpy())
    rlp, rent, rlse = oracle.lmhead_forward(hq, wq, inp["targets"], inp["mask"])
    assert np.max(np.abs(lp.cpu().numpy() - rlp)) <= BF16_TOL["lp"]
    assert np.max(np.abs(ent.cpu().numpy() - rent)) <= BF16_TOL["ent"]
    assert np.max(np.abs(lse.cpu().numpy() - rlse)) <= BF16_TOL["lp"]
    inactive = inp["mask"] == 0
    assert np.all(lp.cpu().numpy()[inactive] == 0)
