"""Vocabulary-parallel use on one GPU (the page's TP layouts, "Performance":
every (TP, CP) with TP x CP <= 8): W split into uneven row shards; shard
statistics merged by eas_lmhead_combine_shards must match the unsharded
forward and the oracle, and the shards' dW rows and summed dHidden partials
must match the oracle's gradients."""
import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from gpu_helpers import BF16_TOL, FP32_TOL, rel_fro, small_inputs, to_dev
from entropy_active_span_gb300 import workloads as W
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,cuts", [("bf16", (0, 700, 1301, 2500)),
                                        ("bf16", (0, 2500)),
                                        ("fp32", (0, 333, 1000, 2048, 2500))])
def test_vocab_shards_match_unsharded_and_oracle(dtype, cuts):
    inp = small_inputs(900, 256, 2500, dtype=dtype, seed=17, mask_kind="bernoulli0.6",
                       w_std=3.0)
    tol = BF16_TOL if dtype == "bf16" else FP32_TOL
    h, w = to_dev(inp["hidden"]), to_dev(inp["weight"])
    t, m = to_dev(inp["targets"]), to_dev(inp["mask"])
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    spans, ns = eas.build_active_spans(m, 128)
    T = h.shape[0]
    n = len(cuts) - 1
    stats = torch.empty((n, T, 4), dtype=torch.float32, device="cuda")
    for k in range(n):
        eas.lmhead_fwd_shard(h, w[cuts[k]:cuts[k + 1]], cuts[k], t, m, spans, ns, stats=stats[k])
    lp, ent, lse = eas.lmhead_combine_shards(stats, m)
    lp0, ent0, lse0 = eas.lmhead_fwd(h, w, t, m, spans, ns)
    for a, b in ((lp, lp0), (ent, ent0), (lse, lse0)):
        assert torch.max(torch.abs(a - b)).item() <= 1e-4
    h64, w64 = W.to_f64(inp["hidden"]), W.to_f64(inp["weight"])
    rlp, rent, rlse = oracle.lmhead_forward(h64, w64, inp["targets"], inp["mask"])
    assert np.max(np.abs(lp.cpu().numpy() - rlp)) <= tol["lp"]
    assert np.max(np.abs(ent.cpu().numpy() - rent)) <= tol["ent"]
    rdh, rdw = oracle.lmhead_backward(h64, w64, inp["targets"], inp["mask"], inp["g_logprob"],
                                      inp["g_entropy"])
    dh_sum = torch.zeros(h.shape, dtype=torch.float32, device="cuda")
    dws = []
    for k in range(n):
        dh_k, dw_k = eas.lmhead_bwd_shard(glp, gh, h, w[cuts[k]:cuts[k + 1]], cuts[k], t, m,
                                          spans, ns, lse, ent, vocab_chunk=512)
        dh_sum += dh_k.float()
        dws.append(dw_k)
    assert rel_fro(dh_sum.cpu().numpy(), rdh) <= tol["fro"]
    assert rel_fro(torch.cat(dws).cpu().numpy(), rdw) <= tol["fro"]
    assert torch.all(dh_sum[torch.from_numpy(inp["mask"] == 0).cuda()] == 0)
