"""Seeded random sweeps of small problems against the oracle (the full
path, the e4m3 forward, vocabulary shards and context-parallel layouts).

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

import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import workloads as W
from gpu_helpers import BF16_TOL, FP32_TOL, rel_fro, run_gpu, small_inputs, to_dev
from test_gpu_2_lmhead import check, oracle_all
import oracle

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


@pytest.mark.parametrize("i", range(30))
def test_random_e4m3_forward_matches_oracle(i):
    """e4m3 forward on random shapes; the oracle quantises its own copies of
    the operands (its codes equal the device quantiser's)."""
    rng = np.random.default_rng(7000 + i)
    T, H, V = int(rng.integers(1, 600)), int(rng.choice([128, 256, 384, 512])), int(rng.integers(3, 3000))
    inp = small_inputs(T, H, V, seed=int(rng.integers(1, 1 << 30)), mask_kind=str(rng.choice(MASKS)),
                       w_std=[None, 2.0, 5.0][int(rng.integers(0, 3))])
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    h8, hs = eas.quantize_rows_e4m3(h)
    w8, wsc = eas.quantize_rows_e4m3(w)
    spans, ns = eas.build_active_spans(m, 128)
    lp, ent, lse = eas.lmhead_fwd_fp8(h8, hs, w8, wsc, t, m, spans, ns)
    hq = oracle.dequantize_rows_e4m3(*oracle.quantize_rows_e4m3(W.to_f64(inp["hidden"]).astype(np.float32)))
    wq = oracle.dequantize_rows_e4m3(*oracle.quantize_rows_e4m3(W.to_f64(inp["weight"]).astype(np.float32)))
    rlp, rent, rlse = oracle.lmhead_forward(hq, wq, inp["targets"], inp["mask"])
    assert np.max(np.abs(lp.cpu().numpy() - rlp), initial=0) <= BF16_TOL["lp"]
    assert np.max(np.abs(ent.cpu().numpy() - rent), initial=0) <= BF16_TOL["ent"]
    assert np.max(np.abs(lse.cpu().numpy() - rlse), initial=0) <= BF16_TOL["lp"]
    assert np.all(lp.cpu().numpy()[inp["mask"] == 0] == 0)


@pytest.mark.parametrize("i", range(30))
def test_random_vocab_shards_match_oracle(i):
    """W cut into 1-5 random row shards: merged shard statistics and the
    shards' dW rows and summed dHidden partials against the oracle."""
    rng = np.random.default_rng(8000 + i)
    fp32 = rng.random() < 0.25
    H = int(rng.choice([4, 36, 132])) if fp32 else int(rng.choice([64, 192, 320]))
    T, V = int(rng.integers(1, 500)), int(rng.integers(5, 2500))
    n = int(rng.integers(1, 6))
    inner = np.sort(rng.choice(np.arange(1, V), size=min(n - 1, V - 1), replace=False))
    cuts = [0] + [int(x) for x in inner] + [V]
    inp = small_inputs(T, H, V, dtype="fp32" if fp32 else "bf16", seed=int(rng.integers(1, 1 << 30)),
                       mask_kind=str(rng.choice(MASKS)), w_std=[None, 3.0][int(rng.integers(0, 2))])
    tol = FP32_TOL if fp32 else BF16_TOL
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    spans, ns = eas.build_active_spans(m, 128)
    k_n = len(cuts) - 1
    stats = torch.empty((k_n, T, 4), dtype=torch.float32, device="cuda")
    for k in range(k_n):
        eas.lmhead_fwd_shard(h, w[cuts[k]:cuts[k + 1]], cuts[k], t, m, spans, ns, stats=stats[k])
    lp, ent, lse = eas.lmhead_combine_shards(stats, m)
    h64, w64 = W.to_f64(inp["hidden"]), W.to_f64(inp["weight"])
    rlp, rent, rlse = oracle.lmhead_forward(h64, w64, inp["targets"], inp["mask"])
    assert np.max(np.abs(lp.cpu().numpy() - rlp), initial=0) <= tol["lp"]
    assert np.max(np.abs(ent.cpu().numpy() - rent), initial=0) <= tol["ent"]
    assert np.max(np.abs(lse.cpu().numpy() - rlse), initial=0) <= tol["lp"]
    rdh, rdw = oracle.lmhead_backward(h64, w64, inp["targets"], inp["mask"], inp["g_logprob"],
                                      inp["g_entropy"])
    dh_sum = torch.zeros(h.shape, dtype=torch.float32, device="cuda")
    dws = []
    for k in range(k_n):
        dh_k, dw_k = eas.lmhead_bwd_shard(glp, gh, h, w[cuts[k]:cuts[k + 1]], cuts[k], t, m,
                                          spans, ns, lse, ent, vocab_chunk=int(rng.choice([0, 300, 512])))
        dh_sum += dh_k.float()
        dws.append(dw_k)
    assert rel_fro(dh_sum.cpu().numpy(), rdh) <= tol["fro"]
    assert rel_fro(torch.cat(dws).cpu().numpy(), rdw) <= tol["fro"]
    assert torch.all(dh_sum[torch.from_numpy(inp["mask"] == 0).cuda()] == 0)


@pytest.mark.parametrize("i", range(20))
def test_random_cp_layouts_match_oracle(i):
    """Random packed layouts (1-40 segments, CP sizes 1-8, mask densities
    from 5 to 95 %): every rank's local order, local mask and CP-local spans
    bit for bit against the oracle."""
    rng = np.random.default_rng(6000 + i)
    cp = int(rng.choice([1, 2, 3, 4, 8]))
    n_segs = int(rng.integers(1, 41))
    lens = rng.integers(1, 20, size=n_segs) * 2 * cp
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(offs[-1])
    mask = (rng.random(T) < rng.uniform(0.05, 0.95)).astype(np.uint8)
    m, o = to_dev(mask), to_dev(offs)
    gap = int(rng.choice([0, 3, 128]))
    for r in range(cp):
        lm, l2g = eas.cp_local_layout(m, o, cp, r)
        np.testing.assert_array_equal(l2g.cpu().numpy(), oracle.cp_local_to_global(offs, cp, r))
        ref_mask = oracle.cp_local_mask(mask, offs, cp, r)
        np.testing.assert_array_equal(lm.cpu().numpy(), ref_mask)
        spans, ns = eas.build_active_spans(lm, gap)
        n = int(ns.item())
        np.testing.assert_array_equal(spans[:n].cpu().numpy(), oracle.active_spans(ref_mask, gap))
