"""GPU fused LM-head vs the fp64 oracle, element by element, on shapes the
oracle finishes in seconds that still span several tiles and ragged tails.

Tolerances (stated for the path): logprob and entropy within 2e-3 absolute;
dHidden and dW within 1e-2 relative Frobenius error for bf16 inputs and 1e-5
for fp32; inactive rows exactly zero.
"""
import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import _lib
from entropy_active_span_gb300 import workloads as W
from gpu_helpers import BF16_TOL, FP32_TOL, rel_fro, run_gpu, small_inputs, to_dev
import oracle

pytestmark = pytest.mark.gpu


def oracle_all(inp):
    h = W.to_f64(inp["hidden"])
    w = W.to_f64(inp["weight"])
    lp, ent, lse = oracle.lmhead_forward(h, w, inp["targets"], inp["mask"])
    dh, dw = oracle.lmhead_backward(h, w, inp["targets"], inp["mask"], inp["g_logprob"],
                                    inp["g_entropy"])
    return dict(logprob=lp, entropy=ent, lse=lse, dhidden=dh, dweight=dw)


def check(got, ref, mask, tol):
    act = np.asarray(mask) != 0
    assert np.max(np.abs(got["logprob"] - ref["logprob"]), initial=0) <= tol["lp"]
    assert np.max(np.abs(got["entropy"] - ref["entropy"]), initial=0) <= tol["ent"]
    assert np.max(np.abs(got["lse"] - ref["lse"]), initial=0) <= tol["lp"]
    assert rel_fro(got["dhidden"], ref["dhidden"]) <= tol["fro"]
    assert rel_fro(got["dweight"], ref["dweight"]) <= tol["fro"]
    # inactive rows are exactly zero
    assert np.all(got["logprob"][~act] == 0) and np.all(got["entropy"][~act] == 0)
    assert np.all(got["lse"][~act] == 0)
    assert np.all(got["dhidden"][~act] == 0)


def test_tiny_fp32_workload():
    inp = W.make_inputs("tiny_fp32")
    got = run_gpu(inp)
    check(got, oracle_all(inp), inp["mask"], FP32_TOL)


@pytest.mark.parametrize("max_gap", [0, 128])
def test_tiny_fp32_multi_chunk(max_gap):
    inp = W.make_inputs("tiny_fp32", w_std=2.0)
    got = run_gpu(inp, max_gap=max_gap, vocab_chunk=320)      # chunks 320, 320, 320, 64
    check(got, oracle_all(inp), inp["mask"], FP32_TOL)


CASES = [
    # T,    H,   V,    chunk, mask kind,        w_std
    (1000, 256, 1000, 0, "bernoulli0.6", None),
    (1000, 256, 1000, 384, "bernoulli0.6", 6.0),
    (300, 128, 257, 0, "bernoulli0.9", 8.0),
    (130, 64, 100, 0, "bernoulli0.5", 3.0),
    (2048, 512, 5000, 2048, "sparse_short", 2.0),
]


@pytest.mark.parametrize("T,H,V,chunk,kind,w_std", CASES)
@pytest.mark.parametrize("flags", [eas.EAS_ROWS_ACTIVE, eas.EAS_ROWS_SPAN])
def test_bf16_small(T, H, V, chunk, kind, w_std, flags):
    inp = small_inputs(T, H, V, seed=T + V, mask_kind=kind, w_std=w_std)
    got = run_gpu(inp, flags=flags, vocab_chunk=chunk)
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)


def test_bf16_targets_at_vocab_edges():
    T, H, V = 256, 128, 700
    t = np.where(np.arange(T) % 2 == 0, 0, V - 1).astype(np.int32)
    inp = small_inputs(T, H, V, seed=3, mask_kind="bernoulli0.7", w_std=4.0, targets=t)
    got = run_gpu(inp, vocab_chunk=256)                        # chunks 256, 256, 188
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)


def test_empty_mask_gives_zeros():
    inp = small_inputs(500, 128, 300, mask_kind="empty")
    got = run_gpu(inp)
    for k in ("logprob", "entropy", "lse", "dhidden", "dweight"):
        assert np.all(got[k] == 0), k


def test_all_active_mask():
    inp = small_inputs(384, 128, 512, mask_kind="dense", w_std=3.0)
    got = run_gpu(inp)
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)


def test_nan_upstream_on_inactive_rows_stays_out():
    inp = small_inputs(600, 128, 400, mask_kind="bernoulli0.5", w_std=2.0)
    g_lp = inp["g_logprob"].copy()
    g_h = inp["g_entropy"].copy()
    g_lp[inp["mask"] == 0] = np.nan
    g_h[inp["mask"] == 0] = np.inf
    got = run_gpu(inp, g_lp=g_lp, g_h=g_h)
    assert np.all(got["dhidden"][inp["mask"] == 0] == 0)
    assert np.all(np.isfinite(got["dweight"]))
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)


def test_spans_that_miss_active_rows_are_rejected():
    inp = small_inputs(400, 128, 300, mask_kind="bernoulli0.5")
    # spans covering only the first half of the tokens
    spans = torch.tensor([[0, 200]], dtype=torch.int32, device="cuda")
    ns = torch.tensor([1], dtype=torch.int32, device="cuda")
    got = run_gpu(inp, spans=spans, num_spans=ns, want_status=True)
    assert got["status"] == (_lib.EAS_ERR_INVALID_SPANS, _lib.EAS_ERR_INVALID_SPANS)
    for k in ("logprob", "entropy", "lse", "dhidden", "dweight"):
        assert np.all(got[k] == 0), k


def test_unsorted_spans_are_rejected():
    inp = small_inputs(400, 128, 300, mask_kind="dense")
    spans = torch.tensor([[200, 400], [0, 200]], dtype=torch.int32, device="cuda")
    ns = torch.tensor([2], dtype=torch.int32, device="cuda")
    got = run_gpu(inp, spans=spans, num_spans=ns, want_status=True)
    assert got["status"][0] == _lib.EAS_ERR_INVALID_SPANS


def test_bitwise_deterministic():
    inp = small_inputs(1000, 256, 1000, mask_kind="bernoulli0.6", w_std=4.0)
    a = run_gpu(inp, vocab_chunk=384)
    b = run_gpu(inp, vocab_chunk=384)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_active_rows_independent_of_row_policy():
    """Active rows give the same forward outputs whether gap rows are packed
    into the tiles or skipped (row-local arithmetic, same vocabulary tiling)."""
    inp = small_inputs(1000, 256, 1000, mask_kind="bernoulli0.4", w_std=4.0)
    a = run_gpu(inp, flags=eas.EAS_ROWS_ACTIVE)
    b = run_gpu(inp, flags=eas.EAS_ROWS_SPAN)
    for k in ("logprob", "entropy", "lse"):
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_active_rows_match_the_dense_mask_run(dtype):
    """A sparse mask's active rows get bit-identical forward outputs and
    dHidden rows to the same rows in a run where every token is active: each
    row's arithmetic depends only on that row and the vocabulary tiling, not
    on which other rows share its tile."""
    inp = small_inputs(900, 256 if dtype == "bf16" else 36, 1500, dtype=dtype, seed=31,
                       mask_kind="bernoulli0.4", w_std=3.0)
    sparse = run_gpu(inp, vocab_chunk=512)
    dense_inp = dict(inp, mask=np.ones_like(inp["mask"]))
    dense = run_gpu(dense_inp, vocab_chunk=512)
    act = inp["mask"] != 0
    for k in ("logprob", "entropy", "lse", "dhidden"):
        np.testing.assert_array_equal(sparse[k][act], dense[k][act])


@pytest.mark.parametrize("R", [1, 64, 127, 128, 129, 255, 256, 257, 300, 383, 384, 385, 511])
def test_last_row_tile_of_at_most_128_rows(R):
    """When the last 256-row tile holds at most 128 real rows it runs as a
    128 x 256 pair MMA (forward, d-logits, dHidden).  R active tokens, drawn
    from tokens 0..511: the results match the oracle, and every active row is
    bit-identical to the same token in the dense-mask run, where tokens
    0..511 all sit in full 256-row tiles."""
    T, H, V = 600, 256, 700
    rng = np.random.default_rng(4000 + R)
    mask = np.zeros(T, np.uint8)
    mask[rng.choice(512, size=R, replace=False)] = 1
    inp = small_inputs(T, H, V, seed=77, mask=mask, w_std=3.0)
    got = run_gpu(inp, vocab_chunk=512)                 # chunks 512 and 188
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)
    dense = run_gpu(dict(inp, mask=np.ones(T, np.uint8)), vocab_chunk=512)
    act = mask != 0
    for k in ("logprob", "entropy", "lse", "dhidden"):
        np.testing.assert_array_equal(got[k][act], dense[k][act])


@pytest.mark.parametrize("H,chunk", [(1024, 768), (1088, 1024), (1152, 1088), (960, 1280)])
def test_wide_tile_k_extents_and_half_tiles(H, chunk):
    """The backward's 256 x 512 tiles run half 0 alone for the first 16
    k-blocks, then both halves, then half 1 alone.  K extents of 15, 16, 17
    and 18 k-blocks (d-logits over H, dHidden over the chunk) cover an empty
    and a one-step two-half phase; chunk widths of 3 or 5 256-column blocks
    leave a last wide tile with half 0 only."""
    inp = small_inputs(300, H, 2100, seed=H + chunk, mask_kind="bernoulli0.7", w_std=3.0)
    got = run_gpu(inp, vocab_chunk=chunk)
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)


@pytest.mark.parametrize("T,H,V", [(300, 192, 300), (513, 320, 1000), (1, 64, 50), (257, 448, 2049)])
def test_bf16_hidden_width_not_a_tile_multiple(T, H, V):
    """H % 256 != 0 leaves a partial N tile in dHidden and dW; T = 1 is a
    single token; V just past a tile boundary leaves a one-column tail."""
    inp = small_inputs(T, H, V, seed=T * 7 + H, mask_kind="bernoulli0.8", w_std=3.0)
    if inp["mask"].sum() == 0:
        inp["mask"][0] = 1
    got = run_gpu(inp, vocab_chunk=512)
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)


def test_autograd_wrapper_matches_oracle():
    inp = small_inputs(700, 256, 900, seed=5, mask_kind="bernoulli0.6", w_std=3.0)
    h = to_dev(inp["hidden"]).requires_grad_(True)
    w = to_dev(inp["weight"]).requires_grad_(True)
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    lp, ent = eas.fused_logprob_entropy(h, w, t, m, vocab_chunk=256)
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    (lp * glp + ent * gh).sum().backward()
    ref = oracle_all(inp)
    assert np.max(np.abs(lp.detach().cpu().numpy() - ref["logprob"])) <= BF16_TOL["lp"]
    assert np.max(np.abs(ent.detach().cpu().numpy() - ref["entropy"])) <= BF16_TOL["ent"]
    # the products lp*glp on inactive rows are 0 * g, so their gradients vanish there too
    assert rel_fro(h.grad.float().cpu().numpy(), ref["dhidden"]) <= BF16_TOL["fro"]
    assert rel_fro(w.grad.float().cpu().numpy(), ref["dweight"]) <= BF16_TOL["fro"]


def test_forward_only_scoring_matches_full_forward():
    inp = small_inputs(900, 256, 1100, seed=9, mask_kind="bernoulli0.5", w_std=3.0)
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd(h, w, t, m, spans, ns)
    lp2, ent2, lse2 = eas.lmhead_fwd(h, w, t, m, spans, ns, want_lse=False)
    assert lse2 is None
    assert torch.equal(lp, lp2) and torch.equal(ent, ent2)
    with torch.no_grad():
        lp3, ent3 = eas.fused_logprob_entropy(h, w, t, m)
    assert torch.equal(lp, lp3) and torch.equal(ent, ent3)


def test_step_captured_in_a_cuda_graph_matches_eager():
    """spans + forward + backward enqueue only kernels and memsets on the
    stream (no allocation, no host sync), so the whole step replays from a
    CUDA graph with the same results."""
    inp = small_inputs(1500, 256, 3000, seed=13, mask_kind="sparse_short", w_std=3.0)
    T, H = inp["hidden"].shape
    V = inp["weight"].shape[0]
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    spans = torch.empty((T, 2), dtype=torch.int32, device="cuda")
    ns = torch.empty(1, dtype=torch.int32, device="cuda")
    sws = eas.workspace(eas.spans_workspace_size(T), "cuda")
    ws = eas.workspace(eas.lmhead_workspace_size(T, H, V, torch.bfloat16, 1024), "cuda")
    lp, ent, lse = (torch.empty(T, device="cuda") for _ in range(3))
    dh = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((V, H), dtype=torch.float32, device="cuda")

    def step():
        eas.build_active_spans(m, 128, spans=spans, num_spans=ns, ws=sws)
        eas.lmhead_fwd(h, w, t, m, spans, ns, ws=ws, out=(lp, ent, lse))
        eas.lmhead_bwd(glp, gh, h, w, t, m, spans, ns, lse, ent, vocab_chunk=1024, ws=ws,
                       dhidden=dh, dweight=dw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # eager, also warms up the launch paths
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [x.clone() for x in (lp, ent, lse, dh, dw)]
    for x in (lp, ent, lse, dh, dw):
        x.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert eas.read_device_status(ws) == 0
    for a, b in zip(eager, (lp, ent, lse, dh, dw)):
        assert torch.equal(a, b)


def test_out_of_range_target_is_reported():
    inp = small_inputs(300, 128, 400, mask_kind="dense", w_std=2.0)
    inp["targets"] = inp["targets"].copy()
    inp["targets"][17] = 400                       # == V
    got = run_gpu(inp, want_status=True)
    assert got["status"] == (_lib.EAS_ERR_INVALID_ARG, _lib.EAS_ERR_INVALID_ARG)


def test_very_large_logits_stay_finite_and_match():
    """W std 60 gives logits of magnitude ~100: the online max keeps every
    exponent in range and the forward and gradients still match the oracle
    at the usual tolerances."""
    inp = small_inputs(400, 256, 1500, seed=31, mask_kind="bernoulli0.7", w_std=60.0)
    got = run_gpu(inp, vocab_chunk=512)
    for k in got:
        assert np.all(np.isfinite(got[k])), k
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_single_word_vocabulary(dtype):
    """V = 1: every softmax is the point mass, so logprob = entropy = 0 and
    all gradients vanish; lse is the single logit."""
    inp = small_inputs(300, 128, 1, dtype=dtype, seed=2, mask_kind="bernoulli0.7", w_std=3.0)
    got = run_gpu(inp)
    ref = oracle_all(inp)
    assert np.max(np.abs(got["logprob"])) <= 1e-6 and np.max(np.abs(got["entropy"])) <= 1e-6
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= BF16_TOL["lp"]
    # p = 2^((z - lse) log2 e) is 1 only up to ex2 rounding (~1e-7), so the
    # d-logits are ~1e-7 g_lp and the gradients ~1e-7 |W|, not exact zeros
    assert np.max(np.abs(got["dhidden"])) <= 1e-4 and np.max(np.abs(got["dweight"])) <= 1e-4


def test_two_word_vocabulary():
    inp = small_inputs(500, 128, 2, seed=4, mask_kind="bernoulli0.7", w_std=6.0)
    got = run_gpu(inp)
    check(got, oracle_all(inp), inp["mask"], BF16_TOL)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_zero_tokens(dtype):
    H, V = 128, 300
    h = torch.empty((0, H), dtype=dtype, device="cuda")
    w = torch.randn((V, H), device="cuda").to(dtype)
    t = torch.empty(0, dtype=torch.int32, device="cuda")
    m = torch.empty(0, dtype=torch.uint8, device="cuda")
    spans, ns = eas.build_active_spans(m, 128)
    assert int(ns.item()) == 0
    lp, ent, lse = eas.lmhead_fwd(h, w, t, m, spans, ns)
    assert lp.numel() == 0
    g = torch.empty(0, device="cuda")
    dh, dw = eas.lmhead_bwd(g, g, h, w, t, m, spans, ns, lse, ent)
    torch.cuda.synchronize()
    assert dh.shape == (0, H) and torch.all(dw == 0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("rows", [eas.EAS_ROWS_ACTIVE, eas.EAS_ROWS_SPAN])
def test_backward_reusing_forward_rows_is_bitwise_equal(dtype, rows):
    inp = small_inputs(1100, 256, 1300, dtype=dtype, seed=8, mask_kind="bernoulli0.5", w_std=3.0)
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    spans, ns = eas.build_active_spans(m, 128)
    T, H = h.shape
    V = w.shape[0]
    ws = eas.workspace(eas.lmhead_workspace_size(T, H, V, h.dtype, 384), "cuda")
    lp, ent, lse = eas.lmhead_fwd(h, w, t, m, spans, ns, rows, ws=ws)
    ref = eas.lmhead_bwd(glp, gh, h, w, t, m, spans, ns, lse, ent, rows, 384, ws=ws)
    ref = [x.clone() for x in ref]
    eas.lmhead_fwd(h, w, t, m, spans, ns, rows, ws=ws, out=(lp, ent, lse))
    got = eas.lmhead_bwd(glp, gh, h, w, t, m, spans, ns, lse, ent,
                         rows | eas.EAS_REUSE_FWD_ROWS, 384, ws=ws)
    assert eas.read_device_status(ws) == 0
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


def test_trace_records_every_launch():
    inp = small_inputs(600, 256, 1200, seed=12, mask_kind="bernoulli0.6")
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    eas.trace_enable(True)
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd(h, w, t, m, spans, ns)
    eas.lmhead_bwd(glp, gh, h, w, t, m, spans, ns, lse, ent, vocab_chunk=512)
    eas.trace_enable(False)
    recs = eas.trace_read()
    names = [n for n, _ in recs]
    for k in ("spans_build", "rowmap", "gather_rows", "fwd_gemm_tc", "combine",
              "dlogits_gemm_tc", "bwd_chunk_gemm_tc", "dproj_gemm_tc", "zero_rows"):
        assert k in names, k
    # three vocabulary chunks: d-logits(0), two chunk launches, the last projections
    assert names.count("bwd_chunk_gemm_tc") == 2 and names.count("dproj_gemm_tc") == 1
    assert all(ms >= 0 for _, ms in recs)
