"""Seeded synthetic workloads for the block-sparse fused LM-head.

This module only draws random inputs: loss masks with the structure of the
five workloads (RL prompt/response masks, packed bins with alignment padding,
sparse short spans, long responses), targets, hidden states, weights and the
upstream gradients.  It holds none of the method's arithmetic, so both the CPU
oracle's tests and the GPU path's tests and benchmark draw from it.

Every array is a pure function of (workload, seed): sub-streams come from
``numpy.random.SeedSequence(seed).spawn`` and large normal tensors are filled
in fixed-size chunks (each chunk its own Philox stream), so the values do not
depend on the number of threads used to fill them.

bf16 tensors are returned as ``uint16`` bit patterns (round-to-nearest-even
from float32); :func:`bf16_bits_to_f32` widens them exactly.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 24  # elements per independently seeded chunk of a normal tensor


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    V: int
    dtype: str          # "fp32" or "bf16"
    seed: int
    mask_kind: str
    targets: str = "uniform"   # or "zipf1.1"
    std: float = 0.02           # std of hidden and W entries
    description: str = ""

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the block-sparse LM-head is measured on.  Seeds 1001..1005.
WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", 256, 128, 1024, "fp32", 1001, "three_spans",
        description="T=256 H=128 V=1024 fp32; 3 active spans, ~50% active"),
    "rl_16k": Workload(
        "rl_16k", 16384, 4096, 128256, "bf16", 1002, "rl_prompts_1024",
        description="T=16384 H=4096 V=128256 bf16; 16 sequences x 1024, "
                    "prompt 256..512 inactive"),
    "packed_64k": Workload(
        "packed_64k", 65536, 5120, 152064, "bf16", 1003, "packed_bins",
        description="T=65536 H=5120 V=152064 bf16; 4 bins x 16384 of segments "
                    "128..8192 padded to 128, gaps 1..300"),
    "sparse_128k": Workload(
        "sparse_128k", 131072, 7168, 129280, "bf16", 1004, "sparse_short",
        targets="zipf1.1",
        description="T=131072 H=7168 V=129280 bf16; ~10% active in 8..64-token "
                    "spans; Zipf(1.1) targets"),
    "long_256k": Workload(
        "long_256k", 262144, 8192, 128256, "bf16", 1005, "rl_prompts_8192",
        description="T=262144 H=8192 V=128256 bf16; 32 sequences x 8192, "
                    "prompt 2458..4096 inactive"),
}

# A reduced shape of the RL workload for profiler captures (W still larger
# than L2, about 1 GB on the device in total).
PROFILE_WORKLOADS = {
    "rl_4k_v32k": Workload(
        "rl_4k_v32k", 4096, 4096, 32768, "bf16", 1102, "rl_prompts_1024",
        description="T=4096 H=4096 V=32768 bf16; 4 sequences x 1024, prompt 256..512 inactive"),
    "rl_16k_v32k": Workload(
        "rl_16k_v32k", 16384, 4096, 32768, "bf16", 1002, "rl_prompts_1024",
        description="rl_16k's rows and mask with V=32768: its backward launches have the "
                    "shapes of rl_16k's (about 2 GB on the device)"),
    "long_16k_v48k": Workload(
        "long_16k_v48k", 16384, 8192, 49152, "bf16", 1105, "rl_prompts_8192",
        description="long_256k's H, mask structure and vocabulary chunk on 2 sequences x 8192 "
                    "and V=49152 (3 chunks): tiles with long_256k's K extents, about 5 GB "
                    "on the device"),
}
ALL_WORKLOADS = {**WORKLOADS, **PROFILE_WORKLOADS}


def _streams(seed: int):
    names = ("mask", "targets", "hidden", "weight", "g_logprob", "g_entropy")
    children = np.random.SeedSequence(seed).spawn(len(names))
    return dict(zip(names, children))


def _rng(ss: np.random.SeedSequence) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(ss))


# --------------------------------------------------------------------------
# loss masks
# --------------------------------------------------------------------------

def _mask_three_spans(T: int, rng) -> np.ndarray:
    """3 active spans (each >= 8 tokens, 128 in total) and 4 gaps summing to
    T-128, interior gaps >= 1, so every interior gap is <= 128 for T=256."""
    n_active = T // 2
    lens = 8 + rng.multinomial(n_active - 24, [1 / 3] * 3)
    gaps = rng.multinomial(T - n_active - 2, [1 / 4] * 4)
    gaps[1] += 1
    gaps[2] += 1
    mask = np.zeros(T, np.uint8)
    pos = int(gaps[0])
    for k in range(3):
        mask[pos:pos + lens[k]] = 1
        pos += int(lens[k]) + int(gaps[k + 1])
    assert pos == T
    return mask


def _mask_rl_prompts(T: int, seq: int, p_lo: int, p_hi: int, rng) -> np.ndarray:
    mask = np.zeros(T, np.uint8)
    for s in range(T // seq):
        p = int(rng.integers(p_lo, p_hi + 1))
        mask[s * seq + p:(s + 1) * seq] = 1
    return mask


def _alternate(mask: np.ndarray, lo: int, hi: int, inact, act, rng) -> None:
    """Fill mask[lo:hi] with alternating inactive/active runs, inactive first."""
    pos = lo
    active = False
    while pos < hi:
        n = int(rng.integers(act[0], act[1] + 1)) if active else \
            int(rng.integers(inact[0], inact[1] + 1))
        end = min(hi, pos + n)
        if active:
            mask[pos:end] = 1
        pos = end
        active = not active


def _mask_packed_bins(T: int, rng, bin_len=16384, align=128) -> np.ndarray:
    mask = np.zeros(T, np.uint8)
    for b in range(T // bin_len):
        pos = b * bin_len
        end = (b + 1) * bin_len
        while pos < end:
            left = end - pos
            L = int(rng.integers(128, min(8192, left) + 1))
            _alternate(mask, pos, pos + L, (1, 300), (16, 160), rng)
            pos += -(-L // align) * align     # alignment padding stays inactive
    return mask


def _mask_sparse_short(T: int, rng) -> np.ndarray:
    mask = np.zeros(T, np.uint8)
    _alternate(mask, 0, T, (1, 647), (8, 64), rng)
    return mask


def make_mask(w: Workload) -> np.ndarray:
    rng = _rng(_streams(w.seed)["mask"])
    kind = w.mask_kind
    if kind == "three_spans":
        return _mask_three_spans(w.T, rng)
    if kind == "rl_prompts_1024":
        return _mask_rl_prompts(w.T, 1024, 256, 512, rng)
    if kind == "rl_prompts_8192":
        return _mask_rl_prompts(w.T, 8192, 2458, 4096, rng)
    if kind == "packed_bins":
        return _mask_packed_bins(w.T, rng)
    if kind == "sparse_short":
        return _mask_sparse_short(w.T, rng)
    if kind == "dense":
        return np.ones(w.T, np.uint8)
    if kind == "empty":
        return np.zeros(w.T, np.uint8)
    if kind.startswith("bernoulli"):
        p = float(kind[len("bernoulli"):])
        return (rng.random(w.T) < p).astype(np.uint8)
    raise ValueError(f"unknown mask kind {kind!r}")


# --------------------------------------------------------------------------
# targets, tensors, upstream gradients
# --------------------------------------------------------------------------

def make_targets(w: Workload) -> np.ndarray:
    rng = _rng(_streams(w.seed)["targets"])
    if w.targets == "uniform":
        return rng.integers(0, w.V, size=w.T, dtype=np.int64).astype(np.int32)
    if w.targets.startswith("zipf"):
        a = float(w.targets[4:])
        weights = (np.arange(1, w.V + 1, dtype=np.float64)) ** (-a)
        cdf = np.cumsum(weights)
        cdf /= cdf[-1]
        u = rng.random(w.T)
        t = np.searchsorted(cdf, u, side="right")
        return np.minimum(t, w.V - 1).astype(np.int32)
    raise ValueError(f"unknown target kind {w.targets!r}")


def _normal_f32(ss: np.random.SeedSequence, n: int, std: float,
                threads: int | None = None) -> np.ndarray:
    out = np.empty(n, np.float32)
    nchunks = -(-n // _CHUNK)
    children = ss.spawn(nchunks)

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        g = _rng(children[i])
        g.standard_normal(out=out[lo:hi], dtype=np.float32)
        out[lo:hi] *= np.float32(std)

    if nchunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(threads or os.cpu_count() or 4) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even) and return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, np.uint16)
    n = u.size
    step = 1 << 24
    uf, of = u.reshape(-1), out.reshape(-1)

    def conv(i):
        a = uf[i:i + step]
        r = ((a >> 16) & 1) + np.uint32(0x7FFF)
        of[i:i + step] = ((a + r) >> 16).astype(np.uint16)

    with ThreadPoolExecutor(os.cpu_count() or 4) as ex:
        list(ex.map(conv, range(0, n, step)))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_tensor(w: Workload, which: str, std: float | None = None) -> np.ndarray:
    """``which`` is "hidden" ([T,H]) or "weight" ([V,H]).

    Returns float32 for fp32 workloads, bf16 bits (uint16) for bf16 ones."""
    rows = w.T if which == "hidden" else w.V
    x = _normal_f32(_streams(w.seed)[which], rows * w.H, w.std if std is None else std)
    x = x.reshape(rows, w.H)
    if w.dtype == "bf16":
        return f32_to_bf16_bits(x)
    return x


def make_upstream(w: Workload):
    """g_logprob ~ N(0,1) and g_entropy ~ N(0, 0.1^2) on every row (active or not)."""
    s = _streams(w.seed)
    g_lp = _rng(s["g_logprob"]).standard_normal(w.T).astype(np.float32)
    g_h = (0.1 * _rng(s["g_entropy"]).standard_normal(w.T)).astype(np.float32)
    return g_lp, g_h


def make_inputs(w: Workload | str, *, mask_kind: str | None = None,
                w_std: float | None = None) -> dict:
    """All inputs of one workload as host numpy arrays.

    ``mask_kind`` swaps the mask (e.g. "dense" for the all-active ablation);
    ``w_std`` swaps the std of W (to give peaked, far-from-uniform softmaxes)."""
    if isinstance(w, str):
        w = ALL_WORKLOADS[w]
    if mask_kind is not None:
        w = w.replace(mask_kind=mask_kind)
    g_lp, g_h = make_upstream(w)
    return dict(
        workload=w,
        mask=make_mask(w),
        targets=make_targets(w),
        hidden=make_tensor(w, "hidden"),
        weight=make_tensor(w, "weight", std=w_std),
        g_logprob=g_lp,
        g_entropy=g_h,
    )


def to_f64(x: np.ndarray) -> np.ndarray:
    """Exact float64 view of a generated tensor (bf16 bits or float32)."""
    if x.dtype == np.uint16:
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)
