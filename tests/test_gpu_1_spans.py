"""GPU span builder vs the oracle: bit-exact ("perf(megatron): add
block-sparse fused LM-head backward", Bugbot "Overview": ordered spans
coalesced with gaps <= 128)."""
import itertools
import os

import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from entropy_active_span_gb300 import _lib
from entropy_active_span_gb300 import workloads as W
from oracle import active_spans

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def gpu_spans(mask_np, max_gap, cap=None, ws=None):
    m = torch.from_numpy(np.ascontiguousarray(mask_np, dtype=np.uint8)).cuda()
    spans, n = eas.build_active_spans(m, max_gap, cap=cap, ws=ws)
    n = int(n.item())
    return spans[:min(n, spans.shape[0])].cpu().numpy().astype(np.int64), n


def run_mask(T, rng, lo_on, hi_on, lo_off, hi_off, start_on=False):
    mask = np.zeros(T, np.uint8)
    pos, on = 0, start_on
    while pos < T:
        n = int(rng.integers(lo_on, hi_on + 1)) if on else int(rng.integers(lo_off, hi_off + 1))
        if on:
            mask[pos:pos + n] = 1
        pos += n
        on = not on
    return mask


def test_exhaustive_small_masks():
    for T in range(0, 10):
        for bits in itertools.product((0, 1), repeat=T):
            mask = np.array(bits, np.uint8)
            for g in (0, 1, 2, 3, 5, 128):
                got, n = gpu_spans(mask, g)
                ref = active_spans(mask, g)
                assert n == len(ref)
                np.testing.assert_array_equal(got, ref.reshape(-1, 2))


@pytest.mark.parametrize("T", [10, 12, 14, 16])
@pytest.mark.parametrize("g", [0, 1, 2, 3, 5, 128])
def test_exhaustive_masks_in_one_call(T, g):
    """Every mask of T tokens at once: the 2^T masks laid end to end, each
    followed by g + 1 inactive tokens so that no span can join two of them.
    The spans of the whole are then each mask's own spans, offset by the
    mask's position."""
    n_masks = 1 << T
    stride = T + g + 1
    bits = ((np.arange(n_masks)[:, None] >> np.arange(T)[None, :]) & 1).astype(np.uint8)
    whole = np.zeros((n_masks, stride), np.uint8)
    whole[:, :T] = bits
    got, n = gpu_spans(whole.reshape(-1), g)
    ref = [active_spans(bits[k], g).reshape(-1, 2) + k * stride for k in range(n_masks)]
    ref = np.concatenate([r for r in ref if len(r)] or [np.zeros((0, 2), np.int64)])
    assert n == len(ref)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
@pytest.mark.parametrize("g", [0, 128])
def test_workload_masks_match_golden(name, g):
    mask = W.make_mask(W.WORKLOADS[name])
    golden = np.loadtxt(os.path.join(GOLDEN, f"spans_{name}_g{g}.txt"), dtype=np.int64,
                        ndmin=2).reshape(-1, 2)
    got, n = gpu_spans(mask, g)
    assert n == len(golden)
    np.testing.assert_array_equal(got, golden)


@pytest.mark.parametrize("T", [1, 15, 16, 16383, 16384, 16385, 50001, 262144 + 77])
def test_random_large_masks(T):
    rng = np.random.default_rng(T)
    for args in ((1, 40, 1, 300), (1, 3, 1, 3), (100, 5000, 120, 140), (1, 1, 127, 130)):
        mask = run_mask(T, rng, *args, start_on=bool(rng.integers(0, 2)))
        for g in (0, 17, 128, 129):
            got, n = gpu_spans(mask, g)
            ref = active_spans(mask, g)
            assert n == len(ref)
            np.testing.assert_array_equal(got, ref.reshape(-1, 2))


def test_empty_full_and_zero_length():
    got, n = gpu_spans(np.zeros(1000, np.uint8), 128)
    assert n == 0
    got, n = gpu_spans(np.ones(70000, np.uint8), 0)
    assert n == 1 and got.tolist() == [[0, 70000]]
    got, n = gpu_spans(np.zeros(0, np.uint8), 128)
    assert n == 0


def test_capacity_overflow_reports_true_count():
    mask = np.zeros(200, np.uint8)
    mask[::20] = 1                       # 10 isolated tokens, gaps of 19
    ref = active_spans(mask, 5)
    assert len(ref) == 10
    ws = eas.workspace(eas.spans_workspace_size(200), "cuda")
    got, n = gpu_spans(mask, 5, cap=4, ws=ws)
    assert n == 10
    np.testing.assert_array_equal(got, ref[:4])
    assert eas.read_device_status(ws) == _lib.EAS_ERR_SPAN_CAPACITY
