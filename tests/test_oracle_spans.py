"""Pins for the span oracle (CPU only).

The oracle walks the mask and merges runs; these tests check it against a
brute-force enumeration written from a different definition: a span is an
interval [s, e) whose end tokens are active, whose every interior inactive
run is at most max_gap long, and which cannot be extended to a neighbouring
active token without crossing a gap longer than max_gap.  ("perf(megatron):
add block-sparse fused LM-head backward", Bugbot "Overview": spans coalesced
with gaps <= 128; "How it works": ordered spans, tokens not reordered.)
"""
import itertools

import numpy as np
import pytest

from oracle import active_spans, span_rows

GAPS = (0, 1, 2, 3, 5, 128)


def brute_force_spans(mask, max_gap):
    m = [bool(x) for x in mask]
    T = len(m)
    act = [i for i in range(T) if m[i]]
    out = []
    for s in range(T):
        for e in range(s + 1, T + 1):
            if not (m[s] and m[e - 1]):
                continue
            # every inactive run inside [s, e) is <= max_gap long
            ok, run = True, 0
            for i in range(s, e):
                run = 0 if m[i] else run + 1
                if run > max_gap:
                    ok = False
                    break
            if not ok:
                continue
            prev = [i for i in act if i < s]
            nxt = [i for i in act if i >= e]
            if prev and s - prev[-1] - 1 <= max_gap:
                continue          # extendable to the left
            if nxt and nxt[0] - e <= max_gap:
                continue          # extendable to the right
            out.append((s, e))
    return out


@pytest.mark.parametrize("T", range(0, 11))
def test_exhaustive_small(T):
    for bits in itertools.product((0, 1), repeat=T):
        for g in GAPS:
            got = [tuple(map(int, x)) for x in active_spans(np.array(bits, np.uint8), g)]
            assert got == brute_force_spans(bits, g), (bits, g)


def test_random_medium():
    rng = np.random.default_rng(7)
    for _ in range(300):
        T = int(rng.integers(11, 40))
        p = rng.random()
        mask = (rng.random(T) < p).astype(np.uint8)
        for g in GAPS:
            got = [tuple(map(int, x)) for x in active_spans(mask, g)]
            assert got == brute_force_spans(mask, g)


def check_invariants(mask, spans, max_gap):
    mask = np.asarray(mask).astype(bool)
    T = len(mask)
    covered = np.zeros(T, bool)
    for k, (s, e) in enumerate(spans):
        assert 0 <= s < e <= T
        assert mask[s] and mask[e - 1]
        covered[s:e] = True
        if k:
            gap = s - spans[k - 1][1]
            assert gap > max_gap       # coalesced spans are separated by long gaps
    assert np.all(covered[mask])       # union covers every active token


@pytest.mark.parametrize("max_gap", [0, 1, 17, 128])
def test_invariants_random_long(max_gap):
    rng = np.random.default_rng(11 + max_gap)
    for _ in range(20):
        T = int(rng.integers(1, 5000))
        mask = np.zeros(T, np.uint8)
        pos, on = 0, False
        while pos < T:
            n = int(rng.integers(1, 300))
            if on:
                mask[pos:pos + n] = 1
            pos += n
            on = not on
        check_invariants(mask, active_spans(mask, max_gap), max_gap)


def test_special_cases():
    assert active_spans(np.zeros(100, np.uint8)).shape == (0, 2)
    assert active_spans(np.zeros(0, np.uint8)).shape == (0, 2)
    assert active_spans(np.ones(77, np.uint8)).tolist() == [[0, 77]]
    m = np.zeros(1000, np.uint8)
    m[[5, 500, 900]] = 1
    assert active_spans(m, 10_000).tolist() == [[5, 901]]
    assert active_spans(m, 0).tolist() == [[5, 6], [500, 501], [900, 901]]
    # a gap of exactly max_gap merges, one more does not
    m = np.zeros(400, np.uint8)
    m[10:20] = 1
    m[148:150] = 1          # gap 128
    m[279:280] = 1          # gap 129
    assert active_spans(m, 128).tolist() == [[10, 150], [279, 280]]


def test_span_rows():
    m = np.array([0, 1, 1, 0, 0, 1, 0, 0, 0, 0, 1], np.uint8)
    sp = active_spans(m, 2)
    assert sp.tolist() == [[1, 6], [10, 11]]
    assert span_rows(sp, m).tolist() == [1, 2, 5, 10]
    assert span_rows(sp, m, include_gaps=True).tolist() == [1, 2, 3, 4, 5, 10]
