"""Failure detection without a GPU fault: a bounded pipeline wait that nothing
completes runs out and reports EAS_ERR_TIMEOUT through the status word, and
the device stays usable afterwards."""
import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import _lib
from gpu_helpers import BF16_TOL, run_gpu, small_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_device_stays_usable(libeas):
    ws = eas.workspace(64, "cuda")
    st = libeas.eas_selftest_wait_timeout(2_000_000, ws.data_ptr(), ws.numel(),
                                          torch.cuda.current_stream().cuda_stream)
    assert st == _lib.EAS_OK
    assert eas.read_device_status(ws) == _lib.EAS_ERR_TIMEOUT
    # the context is intact: a normal forward + backward still runs and checks out
    inp = small_inputs(300, 128, 400, mask_kind="bernoulli0.5", w_std=2.0)
    got = run_gpu(inp)
    assert np.all(np.isfinite(got["logprob"]))
    assert np.all(got["dhidden"][inp["mask"] == 0] == 0)


def test_selftest_rejects_bad_arguments(libeas):
    ws = eas.workspace(64, "cuda")
    assert libeas.eas_selftest_wait_timeout(0, ws.data_ptr(), 64, None) == _lib.EAS_ERR_INVALID_ARG
    assert libeas.eas_selftest_wait_timeout(1000, ws.data_ptr(), 4, None) == _lib.EAS_ERR_WORKSPACE
