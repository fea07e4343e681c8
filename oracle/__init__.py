"""CPU oracle for the block-sparse fused LM-head (test infrastructure only).

Plain, slow, obviously correct float64 NumPy restatements of what the path
computes, written from "perf(megatron): add block-sparse fused LM-head
backward" (SkyRL PR #2376; sections "What does this PR do?", "How it works",
Bugbot "Overview") and the textbook definitions of log-softmax, softmax
entropy and their gradients that the page names.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never calls it.
"""
from .spans import active_spans, span_rows
from .cp import cp_local_mask, cp_local_to_global
from .fp8 import (dequantize_rows_e4m3, dequantized_rows, e4m3_decode, e4m3_encode_rne,
                  lmhead_backward_e4m3, lmhead_backward_e4m3_rows_weighted,
                  quantize_rows_e4m3)
from .lmhead import (lmhead_forward, lmhead_forward_rows, lmhead_dlogits_rows,
                     lmhead_backward, lmhead_backward_rows_weighted, loss_value)

__all__ = [
    "active_spans", "span_rows", "cp_local_mask", "cp_local_to_global", "lmhead_forward", "lmhead_forward_rows",
    "lmhead_dlogits_rows", "lmhead_backward", "lmhead_backward_rows_weighted",
    "loss_value", "e4m3_decode", "e4m3_encode_rne", "quantize_rows_e4m3",
    "dequantize_rows_e4m3", "dequantized_rows", "lmhead_backward_e4m3",
    "lmhead_backward_e4m3_rows_weighted",
]
