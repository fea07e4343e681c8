"""e4m3 (FP8) operands: the device quantiser must give the oracle's codes and
scales bit for bit, and the FP8 forward must match the fp64 oracle run on the
dequantised operands (the quantisation itself is the oracle's, so the only
difference left is fp32 accumulation) within the forward tolerance."""
import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import workloads as W
from gpu_helpers import BF16_TOL, rel_fro, small_inputs, to_dev
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
    # the oracle quantises the host copies itself (its codes equal the
    # device's, test_quantizer_bit_exact)
    hq = oracle.dequantize_rows_e4m3(*oracle.quantize_rows_e4m3(W.to_f64(inp["hidden"]).astype(np.float32)))
    wq = oracle.dequantize_rows_e4m3(*oracle.quantize_rows_e4m3(W.to_f64(inp["weight"]).astype(np.float32)))
    rlp, rent, rlse = oracle.lmhead_forward(hq, wq, inp["targets"], inp["mask"])
    assert np.max(np.abs(lp.cpu().numpy() - rlp)) <= BF16_TOL["lp"]
    assert np.max(np.abs(ent.cpu().numpy() - rent)) <= BF16_TOL["ent"]
    assert np.max(np.abs(lse.cpu().numpy() - rlse)) <= BF16_TOL["lp"]
    inactive = inp["mask"] == 0
    assert np.all(lp.cpu().numpy()[inactive] == 0)


def test_misaligned_column_scales_give_identical_results():
    """Column scales that start 4 bytes past a 16-byte boundary take the
    epilogue's scalar loads; the outputs must equal the aligned call's."""
    inp = small_inputs(600, 256, 1024, seed=44, mask_kind="bernoulli0.7", w_std=3.0)
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    h8, hs = eas.quantize_rows_e4m3(h)
    w8, wsc = eas.quantize_rows_e4m3(w)
    spans, ns = eas.build_active_spans(m, 128)
    shifted = torch.empty(wsc.numel() + 1, dtype=wsc.dtype, device=wsc.device)
    shifted[1:] = wsc
    wsc_odd = shifted[1:]
    assert wsc_odd.data_ptr() % 16 != 0
    a = eas.lmhead_fwd_fp8(h8, hs, w8, wsc, t, m, spans, ns)
    b = eas.lmhead_fwd_fp8(h8, hs, w8, wsc_odd, t, m, spans, ns)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_fp8_forward_full_size_rl_16k():
    """The e4m3 forward at the rl_16k shape the forward-only bench line times
    (T=16384, H=4096, V=128256), with a large-std W so the softmax is peaked;
    sampled active rows are checked against the oracle run on operands it
    quantised itself (about a minute of host work for W)."""
    w = W.WORKLOADS["rl_16k"]
    inp = W.make_inputs(w, w_std=1.5)
    h, wt = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    h8, hs = eas.quantize_rows_e4m3(h)
    w8, wsc = eas.quantize_rows_e4m3(wt)
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd_fp8(h8, hs, w8, wsc, t, m, spans, ns)
    inactive = inp["mask"] == 0
    assert np.all(lp.cpu().numpy()[inactive] == 0)
    assert np.all(ent.cpu().numpy()[inactive] == 0)
    act = np.flatnonzero(inp["mask"])
    rng = np.random.default_rng(w.seed)
    rows = np.sort(np.concatenate([act[:2], act[-2:], rng.choice(act, 60, replace=False)]))
    rows = np.unique(rows)
    wq = oracle.dequantize_rows_e4m3(*oracle.quantize_rows_e4m3(W.to_f64(inp["weight"]).astype(np.float32)))
    hq = oracle.dequantize_rows_e4m3(
        *oracle.quantize_rows_e4m3(W.to_f64(inp["hidden"][rows]).astype(np.float32)))
    rlp, rent, rlse = oracle.lmhead_forward_rows(hq, wq, inp["targets"][rows])
    idx = torch.from_numpy(rows).cuda()
    assert np.max(np.abs(lp[idx].cpu().numpy() - rlp)) <= BF16_TOL["lp"]
    assert np.max(np.abs(ent[idx].cpu().numpy() - rent)) <= BF16_TOL["ent"]
    assert np.max(np.abs(lse[idx].cpu().numpy() - rlse)) <= BF16_TOL["lp"]


# ------------------------------------------------------------- backward
#
# eas_lmhead_bwd_fp8: d-logits of the e4m3 logits (recomputed from the same
# e4m3 operands the forward used), projected with the bf16 operands.  The
# oracle is oracle.lmhead_backward_e4m3 (it quantises its own operands; its
# codes equal the device's, test_quantizer_bit_exact), pinned on the CPU to
# the bf16 oracle by the special cases in test_oracle_fp8.py.

def _fp8_step(inp, chunk=0, flags=eas.EAS_ROWS_ACTIVE):
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    h8, hs = eas.quantize_rows_e4m3(h)
    w8, wsc = eas.quantize_rows_e4m3(w)
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd_fp8(h8, hs, w8, wsc, t, m, spans, ns, flags)
    ws = eas.workspace(eas.lmhead_bwd_fp8_workspace_size(*h.shape, w.shape[0], chunk), h.device)
    dh, dw = eas.lmhead_bwd_fp8(glp, gh, h, w, h8, hs, w8, wsc, t, m, spans, ns, lse, ent, flags,
                                chunk, ws=ws)
    assert eas.read_device_status(ws) == 0
    torch.cuda.synchronize()
    return dh.float().cpu().numpy(), dw.cpu().numpy()


@pytest.mark.parametrize("T,H,V,chunk,kind,w_std,flags", [
    (700, 256, 1000, 0, "bernoulli0.6", 3.0, eas.EAS_ROWS_ACTIVE),
    (700, 256, 1000, 384, "bernoulli0.6", 3.0, eas.EAS_ROWS_ACTIVE),
    (300, 128, 257, 0, "bernoulli0.9", 8.0, eas.EAS_ROWS_SPAN),
    (2048, 512, 5000, 1537, "sparse_short", 2.0, eas.EAS_ROWS_ACTIVE),
    (1000, 384, 3000, 1000, "bernoulli0.5", 1.0, eas.EAS_ROWS_SPAN),
])
def test_fp8_backward_matches_oracle(T, H, V, chunk, kind, w_std, flags):
    inp = small_inputs(T, H, V, seed=T + V + chunk, mask_kind=kind, w_std=w_std)
    dh, dw = _fp8_step(inp, chunk, flags)
    rdh, rdw = oracle.lmhead_backward_e4m3(W.to_f64(inp["hidden"]), W.to_f64(inp["weight"]),
                                           inp["targets"], inp["mask"], inp["g_logprob"],
                                           inp["g_entropy"])
    assert rel_fro(dh, rdh) <= BF16_TOL["fro"]
    assert rel_fro(dw, rdw) <= BF16_TOL["fro"]
    inactive = inp["mask"] == 0
    assert np.all(dh[inactive] == 0)


def test_fp8_backward_is_the_e4m3_gradient_not_the_bf16_one():
    """With logits of std ~5 the e4m3 and bf16 gradients differ by about 4 %
    (relative Frobenius), four times the tolerance: the result must match the
    e4m3 oracle and miss the bf16 one, so a recompute that silently ran on the
    bf16 operands would fail."""
    inp = small_inputs(512, 512, 2048, seed=77, mask_kind="bernoulli0.6", w_std=10.0)
    dh, dw = _fp8_step(inp, 1024)
    args = (W.to_f64(inp["hidden"]), W.to_f64(inp["weight"]), inp["targets"], inp["mask"],
            inp["g_logprob"], inp["g_entropy"])
    rdh, rdw = oracle.lmhead_backward_e4m3(*args)
    bdh, bdw = oracle.lmhead_backward(*args)
    assert rel_fro(rdh, bdh) > 3 * BF16_TOL["fro"]
    assert rel_fro(dh, rdh) <= BF16_TOL["fro"] and rel_fro(dw, rdw) <= BF16_TOL["fro"]
    assert rel_fro(dh, bdh) > 2 * BF16_TOL["fro"] and rel_fro(dw, bdw) > 2 * BF16_TOL["fro"]


def test_fp8_backward_is_deterministic():
    inp = small_inputs(1000, 256, 1000, seed=5, mask_kind="bernoulli0.6", w_std=4.0)
    a = _fp8_step(inp, 384)
    b = _fp8_step(inp, 384)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_fp8_backward_rejects_forward_row_reuse():
    inp = small_inputs(256, 128, 512, seed=6)
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    g = to_dev(inp["g_logprob"])
    h8, hs = eas.quantize_rows_e4m3(h)
    w8, wsc = eas.quantize_rows_e4m3(w)
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd_fp8(h8, hs, w8, wsc, t, m, spans, ns)
    with pytest.raises(eas.EasError):
        eas.lmhead_bwd_fp8(g, g, h, w, h8, hs, w8, wsc, t, m, spans, ns, lse, ent,
                           eas.EAS_REUSE_FWD_ROWS)


def test_fp8_backward_full_size_rl_16k():
    """The e4m3 backward at the rl_16k shape with a peaked W: dHidden on
    sampled rows, and the whole dW from a second backward whose upstream
    gradients vanish outside a row sample S."""
    w = W.WORKLOADS["rl_16k"]
    inp = W.make_inputs(w, w_std=1.5)
    h, wt = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    h8, hs = eas.quantize_rows_e4m3(h)
    w8, wsc = eas.quantize_rows_e4m3(wt)
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd_fp8(h8, hs, w8, wsc, t, m, spans, ns)
    ws = eas.workspace(eas.lmhead_bwd_fp8_workspace_size(w.T, w.H, w.V), h.device)
    act = np.flatnonzero(inp["mask"])
    rng = np.random.default_rng(w.seed)
    S = np.unique(np.concatenate([act[:2], act[-2:], rng.choice(act, 48, replace=False)]))
    g1 = np.zeros(w.T, np.float32)
    g2 = np.zeros(w.T, np.float32)
    g1[S] = inp["g_logprob"][S]
    g2[S] = inp["g_entropy"][S]
    dh, dw = eas.lmhead_bwd_fp8(to_dev(g1), to_dev(g2), h, wt, h8, hs, w8, wsc, t, m, spans, ns,
                                lse, ent, ws=ws)
    assert eas.read_device_status(ws) == 0
    W64 = W.to_f64(inp["weight"])
    Wq = oracle.dequantized_rows(W64)
    rdh, rdw = oracle.lmhead_backward_e4m3_rows_weighted(W.to_f64(inp["hidden"][S]), W64, Wq,
                                                         inp["targets"][S], g1[S], g2[S])
    idx = torch.from_numpy(S).cuda()
    assert rel_fro(dh[idx].float().cpu().numpy(), rdh) <= BF16_TOL["fro"]
    assert rel_fro(dw.cpu().numpy(), rdw) <= BF16_TOL["fro"]
    others = torch.ones(w.T, dtype=torch.bool, device="cuda")
    others[idx] = False
    assert torch.all(dh[others] == 0)
