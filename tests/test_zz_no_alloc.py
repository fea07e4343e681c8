"""The allocation-free forward (eas_lmhead_fwd_noalloc).

That entry point is for callers that cannot allocate device memory when they
run the forward: a host whose pool allocator owns the whole GPU and lends none
to libraries, a host that forbids allocation once it is running, or a plugin
interface that passes a library only its input and output buffers.  Its
scratch is a static 64 MiB device array shared by every call.

The tests call it through the C ABI twice in a row on different problems (so a
call that leaned on what the previous one left in the shared array would
show) and check each result against the fp64 oracle and against the
workspace forward (eas_lmhead_fwd), within the forward tolerance of the other
tests (2e-3 absolute; inactive rows exactly zero).  They also check what the
entry point exists for: once warm, a call changes neither the device's free
memory nor PyTorch's allocation counts.
"""
import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import _lib
from entropy_active_span_gb300 import workloads as W
from gpu_helpers import small_inputs, to_dev
import oracle

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _problem(inp):
    hidden, weight = to_dev(inp["hidden"]), to_dev(inp["weight"])
    targets, mask = to_dev(inp["targets"]), to_dev(inp["mask"].astype(np.uint8))
    spans, ns = eas.build_active_spans(mask, 128)
    return hidden, weight, targets, mask, spans, ns


def _outputs(T):
    return [torch.full((T,), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]


def _noalloc(lib, prob, out):
    hidden, weight, targets, mask, spans, ns = prob
    T, H = hidden.shape
    V = weight.shape[0]
    dt = _lib.EAS_BF16 if hidden.dtype == torch.bfloat16 else _lib.EAS_FP32
    st = lib.eas_lmhead_fwd_noalloc(
        hidden.data_ptr(), weight.data_ptr(), targets.data_ptr(), mask.data_ptr(),
        spans.data_ptr(), ns.data_ptr(), spans.shape[0], T, H, V, dt, 0,
        out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == _lib.EAS_OK, lib.eas_last_error()


def _cases():
    return [small_inputs(2048, 512, 5000, seed=11, mask_kind="sparse_short", w_std=2.0),
            W.make_inputs("tiny_fp32", w_std=2.0)]


def test_noalloc_forward_matches_oracle_and_workspace_forward_twice(libeas):
    for inp in _cases():                           # two calls in a row
        prob = _problem(inp)
        out = _outputs(prob[0].shape[0])
        _noalloc(libeas, prob, out)
        torch.cuda.synchronize()
        got = [o.cpu().numpy() for o in out]
        ws_fwd = [t.cpu().numpy() for t in eas.lmhead_fwd(*prob)]
        ref = oracle.lmhead_forward(W.to_f64(inp["hidden"]), W.to_f64(inp["weight"]),
                                    inp["targets"], inp["mask"])
        inactive = inp["mask"] == 0
        for g, r, o in zip(got, ws_fwd, ref):
            assert np.all(np.isfinite(g))
            assert np.max(np.abs(g - o)) <= TOL        # against the oracle
            assert np.max(np.abs(g - r)) <= TOL        # against the workspace forward
            assert np.all(g[inactive] == 0)


def test_noalloc_forward_allocates_nothing(libeas):
    inp = _cases()[0]
    prob = _problem(inp)
    out = _outputs(prob[0].shape[0])
    _noalloc(libeas, prob, out)                    # warm: set-up done in this context
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(2):
        _noalloc(libeas, prob, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0
    for k in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats1.get(k, 0) == stats0.get(k, 0), k


def test_noalloc_rejects_problems_beyond_the_static_scratch(libeas):
    T, H, V = 16384, 4096, 128256                  # needs ~230 MB of scratch
    p = torch.zeros(16, dtype=torch.uint8, device="cuda")
    st = libeas.eas_lmhead_fwd_noalloc(p.data_ptr(), p.data_ptr(), p.data_ptr(), p.data_ptr(),
                                       p.data_ptr(), p.data_ptr(), 1, T, H, V, _lib.EAS_BF16, 0,
                                       p.data_ptr(), p.data_ptr(), p.data_ptr(), None)
    assert st == _lib.EAS_ERR_WORKSPACE
    msg = libeas.eas_last_error().decode()
    assert "static scratch" in msg and str(_lib.EAS_STATIC_SCRATCH_BYTES) in msg
