"""Seeded random sweep of small problems against the oracle.

Each case draws its dtype, hidden width, token count, vocabulary size,
vocabulary chunk (including widths that are not multiples of the 256-column
tile or of the 64-element k-block), mask kind, span gap, row policy and W
scale from a fixed seed, then runs spans, forward and backward through the
binding and compares every output with the fp64 oracle: logprob, entropy
and lse within 2e-3, dHidden and dW within the relative-Frobenius bound of
the dtype, inactive rows exactly zero, spans bit-exact.
"""
import numpy as np
import pytest

import entropy_active_span_gb300 as eas
from gpu_helpers import BF16_TOL, FP32_TOL, run_gpu, small_inputs
from test_gpu_2_lmhead import check, oracle_all
import oracle
import torch

pytestmark = pytest.mark.gpu

MASKS = ("bernoulli0.1", "bernoulli0.5", "bernoulli0.9", "sparse_short", "dense")


def draw(i):
    rng = np.random.default_rng(9000 + i)
    fp32 = rng.random() < 0.2
    H = int(rng.choice([4, 12, 36, 64, 132])) if fp32 else int(rng.choice([64, 128, 192, 256,
                                                                             320, 448]))
    T = int(rng.integers(1, 700))
    V = int(rng.integers(3, 3000))
    chunk = int(rng.choice([0, 256, 384, 1000, 1537, 2048]))
    return dict(dtype="fp32" if fp32 else "bf16", T=T, H=H, V=V, chunk=chunk,
                mask=str(rng.choice(MASKS)), max_gap=int(rng.choice([0, 1, 17, 128, 1000])),
                flags=int(rng.choice([eas.EAS_ROWS_ACTIVE, eas.EAS_ROWS_SPAN])),
                w_std=[None, 2.0, 5.0][int(rng.integers(0, 3))], seed=int(rng.integers(1, 1 << 30)))


@pytest.mark.parametrize("i", range(120))
def test_random_problem_matches_oracle(i):
    c = draw(i)
    inp = small_inputs(c["T"], c["H"], c["V"], dtype=c["dtype"], seed=c["seed"],
                       mask_kind=c["mask"], w_std=c["w_std"])
    got = run_gpu(inp, max_gap=c["max_gap"], flags=c["flags"], vocab_chunk=c["chunk"])
    check(got, oracle_all(inp), inp["mask"], FP32_TOL if c["dtype"] == "fp32" else BF16_TOL)
    m = torch.from_numpy(inp["mask"].astype(np.uint8)).cuda()
    spans, ns = eas.build_active_spans(m, c["max_gap"])
    n = int(ns.item())
    np.testing.assert_array_equal(spans[:n].cpu().numpy(),
                                  oracle.active_spans(inp["mask"], c["max_gap"]))
