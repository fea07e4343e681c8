"""The stored span fixtures and tiny forward values still follow from the
seeded generators and the oracle (CPU only)."""
import os

import numpy as np
import pytest

from entropy_active_span_gb300 import workloads
from oracle import active_spans, lmhead_forward

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_spans(name, g):
    a = np.loadtxt(os.path.join(GOLDEN, f"spans_{name}_g{g}.txt"), dtype=np.int64, ndmin=2)
    return a.reshape(-1, 2)


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
@pytest.mark.parametrize("g", [0, 128])
def test_span_fixtures(name, g):
    mask = workloads.make_mask(workloads.WORKLOADS[name])
    np.testing.assert_array_equal(active_spans(mask, g), load_spans(name, g))


def test_tiny_forward_fixture():
    inp = workloads.make_inputs("tiny_fp32")
    lp, ent, lse = lmhead_forward(workloads.to_f64(inp["hidden"]), workloads.to_f64(inp["weight"]),
                                  inp["targets"], inp["mask"])
    ref = np.loadtxt(os.path.join(GOLDEN, "tiny_fp32_forward.txt"))
    np.testing.assert_allclose(lp, ref[:, 1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ent, ref[:, 2], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref[:, 3], rtol=0, atol=1e-12)
