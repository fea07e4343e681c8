"""Shared helpers of the GPU parity tests: move generated inputs to the device,
run the library through its binding, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import workloads as W

BF16_TOL = dict(lp=2e-3, ent=2e-3, fro=1e-2)
FP32_TOL = dict(lp=2e-3, ent=2e-3, fro=1e-5)


def to_dev(x: np.ndarray) -> torch.Tensor:
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(np.asarray(got, np.float64) - ref) / (den if den > 0 else 1.0))


def small_inputs(T, H, V, dtype="bf16", seed=7, mask=None, mask_kind="bernoulli0.6",
                 w_std=None, targets=None):
    w = W.Workload(f"small_{T}_{H}_{V}", T, H, V, dtype, seed, mask_kind)
    inp = W.make_inputs(w, w_std=w_std)
    if mask is not None:
        inp["mask"] = np.asarray(mask, np.uint8)
    if targets is not None:
        inp["targets"] = np.asarray(targets, np.int32)
    return inp


def run_gpu(inp, max_gap=128, flags=eas.EAS_ROWS_ACTIVE, vocab_chunk=0, g_lp=None, g_h=None,
            spans=None, num_spans=None, want_status=False):
    """fwd + bwd through the binding; returns host numpy results."""
    T, H = inp["hidden"].shape
    V = inp["weight"].shape[0]
    hidden = to_dev(inp["hidden"])
    weight = to_dev(inp["weight"])
    dt = hidden.dtype
    targets = to_dev(inp["targets"])
    mask = to_dev(inp["mask"].astype(np.uint8))
    glp = to_dev(inp["g_logprob"] if g_lp is None else np.asarray(g_lp, np.float32))
    gh = to_dev(inp["g_entropy"] if g_h is None else np.asarray(g_h, np.float32))
    if spans is None:
        spans, num_spans = eas.build_active_spans(mask, max_gap)
    ws = eas.workspace(eas.lmhead_workspace_size(T, H, V, dt, vocab_chunk), hidden.device)
    lp, ent, lse = eas.lmhead_fwd(hidden, weight, targets, mask, spans, num_spans, flags, ws=ws)
    st_fwd = eas.read_device_status(ws)
    dh, dw = eas.lmhead_bwd(glp, gh, hidden, weight, targets, mask, spans, num_spans, lse, ent,
                            flags, vocab_chunk, ws=ws)
    st_bwd = eas.read_device_status(ws)
    torch.cuda.synchronize()
    out = dict(logprob=lp.cpu().numpy(), entropy=ent.cpu().numpy(), lse=lse.cpu().numpy(),
               dhidden=dh.float().cpu().numpy(), dweight=dw.cpu().numpy())
    if want_status:
        out["status"] = (st_fwd, st_bwd)
    else:
        assert st_fwd == 0 and st_bwd == 0, (st_fwd, st_bwd)
    return out
