"""The allocation-free forward (eas_lmhead_fwd_noalloc) agrees with the
workspace forward (eas_lmhead_fwd).

That entry point is for callers that cannot allocate device memory when they
run the forward (a pool allocator that owns the whole GPU, a host that forbids
allocation after start-up, a plugin interface that passes only the input and
output buffers); its scratch is a static 64 MiB device array shared by every
call.  The test calls it through the C ABI twice in a row on different problems
(so a call that leaned on what the previous one left in the shared array would
show), and compares each result with eas_lmhead_fwd's within the forward
tolerance of the other tests (2e-3 absolute; inactive rows exactly zero).
"""
import ctypes

import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import _lib
from entropy_active_span_gb300 import workloads as W
from gpu_helpers import small_inputs, to_dev

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _problem(inp):
    hidden, weight = to_dev(inp["hidden"]), to_dev(inp["weight"])
    targets, mask = to_dev(inp["targets"]), to_dev(inp["mask"].astype(np.uint8))
    spans, ns = eas.build_active_spans(mask, 128)
    return hidden, weight, targets, mask, spans, ns


def _noalloc(lib, hidden, weight, targets, mask, spans, ns):
    T, H = hidden.shape
    V = weight.shape[0]
    dt = _lib.EAS_BF16 if hidden.dtype == torch.bfloat16 else _lib.EAS_FP32
    out = [torch.full((T,), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]
    st = lib.eas_lmhead_fwd_noalloc(
        hidden.data_ptr(), weight.data_ptr(), targets.data_ptr(), mask.data_ptr(),
        spans.data_ptr(), ns.data_ptr(), spans.shape[0], T, H, V, dt, 0,
        out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == _lib.EAS_OK, lib.eas_last_error()
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def test_noalloc_forward_matches_workspace_forward_twice(libeas):
    cases = [small_inputs(2048, 512, 5000, seed=11, mask_kind="sparse_short", w_std=2.0),
             W.make_inputs("tiny_fp32", w_std=2.0)]
    for inp in cases:                              # two calls in a row
        prob = _problem(inp)
        got = _noalloc(libeas, *prob)
        ref = [t.cpu().numpy() for t in eas.lmhead_fwd(*prob)]
        inactive = inp["mask"] == 0
        for g, r in zip(got, ref):
            assert np.all(np.isfinite(g))
            assert np.max(np.abs(g - r)) <= TOL
            assert np.all(g[inactive] == 0)


def test_noalloc_rejects_problems_beyond_the_static_scratch(libeas):
    T, H, V = 16384, 4096, 128256                  # needs ~230 MB of scratch
    p = torch.zeros(16, dtype=torch.uint8, device="cuda")
    st = libeas.eas_lmhead_fwd_noalloc(p.data_ptr(), p.data_ptr(), p.data_ptr(), p.data_ptr(),
                                       p.data_ptr(), p.data_ptr(), 1, T, H, V, _lib.EAS_BF16, 0,
                                       p.data_ptr(), p.data_ptr(), p.data_ptr(), None)
    assert st == _lib.EAS_ERR_WORKSPACE
    msg = libeas.eas_last_error().decode()
    assert "static scratch" in msg and str(_lib.EAS_STATIC_SCRATCH_BYTES) in msg
