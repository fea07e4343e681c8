"""Context-parallel layouts on one GPU ("How it works": forward mask and
spans from a CP-aware packed layout; diagram: "CP-local ordered spans").

Each CP rank's local token order and mask must match the oracle bit for bit,
its spans must be the oracle's spans of its local mask, and running the
LM head on each rank's local rows must reproduce the global run: identical
forward outputs and dHidden rows for every token, and dW summed over the
ranks equal to the global dW."""
import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import _lib
from gpu_helpers import BF16_TOL, rel_fro, small_inputs, to_dev
import oracle

pytestmark = pytest.mark.gpu


def packed_offsets(rng, n_segs, cp):
    lens = rng.integers(1, 12, size=n_segs) * 2 * cp
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


@pytest.mark.parametrize("cp", [1, 2, 4])
def test_cp_local_layout_and_spans(cp):
    rng = np.random.default_rng(100 + cp)
    offs = packed_offsets(rng, 23, cp)
    T = int(offs[-1])
    mask = (rng.random(T) < 0.45).astype(np.uint8)
    m = to_dev(mask)
    o = to_dev(offs)
    for r in range(cp):
        lm, l2g = eas.cp_local_layout(m, o, cp, r)
        ref_l2g = oracle.cp_local_to_global(offs, cp, r)
        np.testing.assert_array_equal(l2g.cpu().numpy(), ref_l2g)
        ref_mask = oracle.cp_local_mask(mask, offs, cp, r)
        np.testing.assert_array_equal(lm.cpu().numpy(), ref_mask)
        spans, ns = eas.build_active_spans(lm, 128)
        n = int(ns.item())
        np.testing.assert_array_equal(spans[:n].cpu().numpy(), oracle.active_spans(ref_mask, 128))


def test_invalid_layout_is_reported():
    mask = torch.ones(64, dtype=torch.uint8, device="cuda")
    offs = torch.tensor([0, 10, 64], dtype=torch.int32, device="cuda")   # 10 % 4 != 0
    ws = eas.workspace(64, "cuda")
    eas.cp_local_layout(mask, offs, 2, 0, ws=ws)
    assert eas.read_device_status(ws) == _lib.EAS_ERR_INVALID_LAYOUT


def test_cp_ranks_reproduce_the_global_run():
    cp = 2
    rng = np.random.default_rng(7)
    offs = packed_offsets(rng, 9, cp)
    T = int(offs[-1])
    inp = small_inputs(T, 256, 1500, seed=21, mask_kind="bernoulli0.5", w_std=3.0)
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd(h, w, t, m, spans, ns)
    dh, dw = eas.lmhead_bwd(glp, gh, h, w, t, m, spans, ns, lse, ent, vocab_chunk=512)
    dw_sum = torch.zeros_like(dw)
    o = to_dev(offs)
    for r in range(cp):
        lm, l2g = eas.cp_local_layout(m, o, cp, r)
        idx = l2g.long()
        # what rank r holds in CP: its local rows of every per-token tensor
        hl, tl, gl, ghl = (x.index_select(0, idx).contiguous() for x in (h, t, glp, gh))
        sl, nsl = eas.build_active_spans(lm, 128)
        lpl, entl, lsel = eas.lmhead_fwd(hl, w, tl, lm, sl, nsl)
        dhl, dwl = eas.lmhead_bwd(gl, ghl, hl, w, tl, lm, sl, nsl, lsel, entl, vocab_chunk=512)
        # row-local arithmetic in the same vocabulary tiling: bit for bit
        assert torch.equal(lpl, lp[idx]) and torch.equal(entl, ent[idx])
        assert torch.equal(dhl, dh[idx])
        dw_sum += dwl
    assert rel_fro(dw_sum.cpu().numpy(), dw.cpu().numpy()) <= 1e-5
