"""Oracle for the active-span builder (test infrastructure only).

Source: "perf(megatron): add block-sparse fused LM-head backward" (SkyRL PR
#2376), "What does this PR do?" and "How it works": the backward works on
*ordered* active spans derived from the loss mask, tokens are never
reordered; Bugbot "Overview": spans are *coalesced* when the gap between them
is at most 128 tokens.

Readings where the page is silent (each listed in the design notes):
  * a run is a maximal block of consecutive active tokens;
  * the gap between two runs is the number of inactive tokens between them
    (next run's start minus the previous run's end);
  * two runs merge when gap <= max_gap (inclusive), max_gap = 128 by default;
  * spans are half-open [start, end) pairs of token indices, ascending;
    leading and trailing inactive tokens are never inside a span;
  * an empty mask has no spans.
"""
from __future__ import annotations

import numpy as np


def active_spans(mask, max_gap: int = 128) -> np.ndarray:
    """Ordered, coalesced active spans of a 0/1 loss mask.

    Walks the mask once, emitting maximal active runs, and folds each run into
    the previous span when the inactive gap between them is <= ``max_gap``.
    Returns an ``int64`` array of shape [S, 2] of half-open spans."""
    if max_gap < 0:
        raise ValueError("max_gap must be >= 0")
    m = [int(v) != 0 for v in np.asarray(mask).reshape(-1)]
    spans: list[list[int]] = []
    i, T = 0, len(m)
    while i < T:
        if not m[i]:
            i += 1
            continue
        start = i
        while i < T and m[i]:
            i += 1
        end = i                       # run is [start, end)
        if spans and start - spans[-1][1] <= max_gap:
            spans[-1][1] = end        # coalesce with the previous span
        else:
            spans.append([start, end])
    return np.asarray(spans, dtype=np.int64).reshape(-1, 2)


def span_rows(spans: np.ndarray, mask=None, include_gaps: bool = False) -> np.ndarray:
    """Token rows the spans cover, in span order.

    With ``include_gaps`` every row of every span is listed (the span-contiguous
    schedule); otherwise only rows whose mask bit is set (the active rows)."""
    rows = []
    for s, e in np.asarray(spans).reshape(-1, 2):
        r = np.arange(int(s), int(e))
        if not include_gaps:
            r = r[np.asarray(mask)[r] != 0]
        rows.append(r)
    if not rows:
        return np.zeros(0, np.int64)
    return np.concatenate(rows).astype(np.int64)
