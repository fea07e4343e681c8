"""Oracle for context-parallel (CP) token layouts (test infrastructure only).

Source: "perf(megatron): add block-sparse fused LM-head backward" (SkyRL PR
#2376), "How it works": the metadata builder derives the forward mask and the
backward spans from a TP/CP-aware token layout, and packed spans keep a
CP-aware path; diagram: "CP-local ordered spans".  The page does not spell
out the CP split.  Reading taken here (Megatron's load-balanced context
parallelism): every packed segment, whose length is a multiple of 2*cp_size,
is cut into 2*cp_size equal chunks and rank r holds chunk r followed by chunk
2*cp_size-1-r; a rank's local token stream is that pair of chunks for each
segment in order.
"""
from __future__ import annotations

import numpy as np


def cp_local_to_global(seg_offsets, cp_size: int, cp_rank: int) -> np.ndarray:
    """Global token index of each of rank cp_rank's local tokens."""
    seg_offsets = [int(x) for x in seg_offsets]
    out = []
    for k in range(len(seg_offsets) - 1):
        lo, hi = seg_offsets[k], seg_offsets[k + 1]
        L = hi - lo
        if L % (2 * cp_size):
            raise ValueError(f"segment {k} of length {L} is not a multiple of {2 * cp_size}")
        c = L // (2 * cp_size)
        for chunk in (cp_rank, 2 * cp_size - 1 - cp_rank):
            out.extend(range(lo + chunk * c, lo + (chunk + 1) * c))
    return np.asarray(out, dtype=np.int64)


def cp_local_mask(mask, seg_offsets, cp_size: int, cp_rank: int) -> np.ndarray:
    """The loss mask in rank cp_rank's local token order."""
    return np.asarray(mask)[cp_local_to_global(seg_offsets, cp_size, cp_rank)]
