"""GB300 (sm_103a) block-sparse fused LM-head.

Python binding of the C ABI in include/eas.h.  Every function here only
checks and marshals arguments (device pointers, sizes, the current CUDA
stream) and calls the library; all arithmetic runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.

    spans, num_spans = build_active_spans(mask, max_gap=128)
    logprob, entropy, lse = lmhead_fwd(hidden, weight, targets, mask, spans, num_spans)
    dhidden, dweight = lmhead_bwd(g_logprob, g_entropy, hidden, weight, targets, mask,
                                  spans, num_spans, lse, entropy)
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import (EAS_BF16, EAS_DEFAULT_VOCAB_CHUNK, EAS_E4M3, EAS_FP32, EAS_REUSE_FWD_ROWS,
                   EAS_ROWS_ACTIVE, EAS_ROWS_SPAN, EasError)

__all__ = [
    "build_active_spans", "lmhead_fwd", "lmhead_bwd", "lmhead_workspace_size",
    "spans_workspace_size", "read_device_status", "workspace", "EasError",
    "EAS_ROWS_ACTIVE", "EAS_ROWS_SPAN", "EAS_REUSE_FWD_ROWS", "EAS_DEFAULT_VOCAB_CHUNK",
    "FusedLMHeadLogprob",
    "fused_logprob_entropy", "trace_enable", "trace_read", "lmhead_fwd_shard",
    "lmhead_combine_shards", "lmhead_bwd_shard", "cp_local_layout", "quantize_rows_e4m3",
    "lmhead_fwd_fp8", "lmhead_bwd_fp8", "lmhead_bwd_fp8_workspace_size",
]


def _ptr(t):
    return None if t is None else ctypes_ptr(t)


def ctypes_ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return EAS_BF16
    if dt == torch.float32:
        return EAS_FP32
    if dt in (torch.uint8, torch.float8_e4m3fn):
        return EAS_E4M3
    raise TypeError(f"hidden/weight must be bfloat16, float32 or e4m3, got {dt}")


def _as_codes(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def spans_workspace_size(T: int) -> int:
    return int(_lib.load().eas_spans_workspace_size(T))


def lmhead_workspace_size(T: int, H: int, V: int, dtype: torch.dtype,
                          vocab_chunk: int = 0) -> int:
    return int(_lib.load().eas_lmhead_workspace_size(T, H, V, _dtype_code(dtype), vocab_chunk))


def workspace(nbytes: int, device) -> torch.Tensor:
    """A device buffer usable as workspace (torch's allocator aligns to 512 B)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def build_active_spans(mask: torch.Tensor, max_gap: int = 128, cap: int | None = None,
                       spans: torch.Tensor | None = None, num_spans: torch.Tensor | None = None,
                       ws: torch.Tensor | None = None):
    """Ordered active spans of a uint8 loss mask, built on the device.

    Returns (spans int32 [cap, 2], num_spans int32 [1]); only the first
    num_spans rows are meaningful.  cap defaults to the worst case (T+1)//2."""
    dev = mask.device
    _need(mask, "mask", torch.uint8, dev)
    T = mask.numel()
    if cap is None:
        cap = max(1, (T + 1) // 2)
    if spans is None:
        spans = torch.empty((cap, 2), dtype=torch.int32, device=dev)
    if num_spans is None:
        num_spans = torch.empty(1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(spans_workspace_size(T), dev)
    _need(spans, "spans", torch.int32, dev)
    _need(num_spans, "num_spans", torch.int32, dev)
    _lib.check(_lib.load().eas_build_active_spans(
        _ptr(mask), T, int(max_gap), _ptr(spans), int(spans.shape[0]), _ptr(num_spans),
        _ptr(ws), ws.numel(), _stream(dev)))
    return spans, num_spans


def cp_local_layout(mask, seg_offsets, cp_size: int, cp_rank: int, ws=None):
    """(local_mask uint8 [T/cp], local_to_global int32 [T/cp]) of one CP rank
    under the load-balanced split of every packed segment into 2*cp chunks."""
    dev = mask.device
    _need(mask, "mask", torch.uint8, dev)
    _need(seg_offsets, "seg_offsets", torch.int32, dev)
    T = mask.numel()
    n_local = T // cp_size
    local_mask = torch.empty(n_local, dtype=torch.uint8, device=dev)
    l2g = torch.empty(n_local, dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(64, dev)
    _lib.check(_lib.load().eas_cp_local_layout(
        _ptr(mask), _ptr(seg_offsets), int(seg_offsets.numel() - 1), T, int(cp_size),
        int(cp_rank), _ptr(local_mask), _ptr(l2g), _ptr(ws), ws.numel(), _stream(dev)))
    return local_mask, l2g


def lmhead_fwd(hidden, weight, targets, mask, spans, num_spans, flags: int = EAS_ROWS_ACTIVE,
               ws=None, out=None, want_lse: bool = True):
    """Target logprob, entropy and lse of the active rows.  Returns (logprob, entropy, lse).

    With want_lse=False (forward-only scoring) lse is neither computed into
    memory nor returned (None)."""
    dev = hidden.device
    dt = hidden.dtype
    code = _dtype_code(dt)
    T, H = hidden.shape
    V = weight.shape[0]
    _need(hidden, "hidden", dt, dev)
    _need(weight, "weight", dt, dev)
    if weight.shape[1] != H:
        raise ValueError("weight must be [V, H]")
    _need(targets, "targets", torch.int32, dev)
    _need(mask, "mask", torch.uint8, dev)
    _need(spans, "spans", torch.int32, dev)
    _need(num_spans, "num_spans", torch.int32, dev)
    if targets.numel() != T or mask.numel() != T:
        raise ValueError("targets and mask must have T entries")
    if out is None:
        out = tuple(torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
    if ws is None:
        ws = workspace(lmhead_workspace_size(T, H, V, dt), dev)
    logprob, entropy, lse = out
    if not want_lse:
        lse = None
    _lib.check(_lib.load().eas_lmhead_fwd(
        _ptr(hidden), _ptr(weight), _ptr(targets), _ptr(mask), _ptr(spans), _ptr(num_spans),
        int(spans.shape[0]), T, H, V, code, int(flags), _ptr(logprob), _ptr(entropy), _ptr(lse),
        _ptr(ws), ws.numel(), _stream(dev)))
    return logprob, entropy, lse


def lmhead_bwd(g_logprob, g_entropy, hidden, weight, targets, mask, spans, num_spans, lse,
               entropy, flags: int = EAS_ROWS_ACTIVE, vocab_chunk: int = 0, ws=None,
               dhidden=None, dweight=None):
    """dHidden (hidden's dtype) and dW (fp32) of sum_active g_lp logp + g_H H."""
    dev = hidden.device
    dt = hidden.dtype
    code = _dtype_code(dt)
    T, H = hidden.shape
    V = weight.shape[0]
    for t, n in ((g_logprob, "g_logprob"), (g_entropy, "g_entropy"), (lse, "lse"),
                 (entropy, "entropy")):
        _need(t, n, torch.float32, dev)
        if t.numel() != T:
            raise ValueError(f"{n} must have T entries")
    _need(hidden, "hidden", dt, dev)
    _need(weight, "weight", dt, dev)
    _need(targets, "targets", torch.int32, dev)
    _need(mask, "mask", torch.uint8, dev)
    _need(spans, "spans", torch.int32, dev)
    _need(num_spans, "num_spans", torch.int32, dev)
    if dhidden is None:
        dhidden = torch.empty((T, H), dtype=dt, device=dev)
    if dweight is None:
        dweight = torch.empty((V, H), dtype=torch.float32, device=dev)
    _need(dhidden, "dhidden", dt, dev)
    _need(dweight, "dweight", torch.float32, dev)
    if ws is None:
        ws = workspace(lmhead_workspace_size(T, H, V, dt, vocab_chunk), dev)
    _lib.check(_lib.load().eas_lmhead_bwd(
        _ptr(g_logprob), _ptr(g_entropy), _ptr(hidden), _ptr(weight), _ptr(targets), _ptr(mask),
        _ptr(spans), _ptr(num_spans), int(spans.shape[0]), _ptr(lse), _ptr(entropy),
        T, H, V, code, int(flags), int(vocab_chunk), _ptr(dhidden), _ptr(dweight),
        _ptr(ws), ws.numel(), _stream(dev)))
    return dhidden, dweight


def quantize_rows_e4m3(x: torch.Tensor, out=None, scale=None):
    """Per-row e4m3 quantisation of a bf16/fp32 [R, H] tensor on the device.
    Returns (codes uint8 [R, H], scale fp32 [R])."""
    dev = x.device
    code = _dtype_code(x.dtype)
    if code == EAS_E4M3:
        raise TypeError("x must be bfloat16 or float32")
    _need(x, "x", x.dtype, dev)
    R, H = x.shape
    if out is None:
        out = torch.empty((R, H), dtype=torch.uint8, device=dev)
    if scale is None:
        scale = torch.empty(R, dtype=torch.float32, device=dev)
    _lib.check(_lib.load().eas_quantize_rows_e4m3(_ptr(x), code, R, H, _ptr(out), _ptr(scale),
                                                  _stream(dev)))
    return out, scale


def lmhead_fwd_fp8(hidden_e4m3, hidden_scale, weight_e4m3, weight_scale, targets, mask, spans,
                   num_spans, flags: int = EAS_ROWS_ACTIVE, ws=None, out=None,
                   want_lse: bool = True):
    """Forward with e4m3 operands and per-row scales (forward-only scoring)."""
    h8, w8 = _as_codes(hidden_e4m3), _as_codes(weight_e4m3)
    dev = h8.device
    T, H = h8.shape
    V = w8.shape[0]
    for t, n, d in ((h8, "hidden_e4m3", torch.uint8), (w8, "weight_e4m3", torch.uint8),
                    (hidden_scale, "hidden_scale", torch.float32),
                    (weight_scale, "weight_scale", torch.float32),
                    (targets, "targets", torch.int32), (mask, "mask", torch.uint8),
                    (spans, "spans", torch.int32), (num_spans, "num_spans", torch.int32)):
        _need(t, n, d, dev)
    if out is None:
        out = tuple(torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
    lp, ent, lse = out
    if not want_lse:
        lse = None
    if ws is None:
        ws = workspace(lmhead_workspace_size(T, H, V, torch.uint8), dev)
    _lib.check(_lib.load().eas_lmhead_fwd_fp8(
        _ptr(h8), _ptr(hidden_scale), _ptr(w8), _ptr(weight_scale), _ptr(targets), _ptr(mask),
        _ptr(spans), _ptr(num_spans), int(spans.shape[0]), T, H, V, int(flags), _ptr(lp),
        _ptr(ent), _ptr(lse), _ptr(ws), ws.numel(), _stream(dev)))
    return lp, ent, lse


def lmhead_bwd_fp8_workspace_size(T: int, H: int, V: int, vocab_chunk: int = 0) -> int:
    return int(_lib.load().eas_lmhead_bwd_fp8_workspace_size(T, H, V, vocab_chunk))


def lmhead_bwd_fp8(g_logprob, g_entropy, hidden, weight, hidden_e4m3, hidden_scale, weight_e4m3,
                   weight_scale, targets, mask, spans, num_spans, lse, entropy,
                   flags: int = EAS_ROWS_ACTIVE, vocab_chunk: int = 0, ws=None, dhidden=None,
                   dweight=None):
    """Backward of the e4m3 forward: d-logits of the e4m3 logits, projected
    with the bf16 operands.  Returns (dHidden bf16, dW fp32)."""
    dev = hidden.device
    T, H = hidden.shape
    V = weight.shape[0]
    h8, w8 = _as_codes(hidden_e4m3), _as_codes(weight_e4m3)
    for t, n, d in ((g_logprob, "g_logprob", torch.float32), (g_entropy, "g_entropy", torch.float32),
                    (lse, "lse", torch.float32), (entropy, "entropy", torch.float32),
                    (hidden, "hidden", torch.bfloat16), (weight, "weight", torch.bfloat16),
                    (h8, "hidden_e4m3", torch.uint8), (w8, "weight_e4m3", torch.uint8),
                    (hidden_scale, "hidden_scale", torch.float32),
                    (weight_scale, "weight_scale", torch.float32),
                    (targets, "targets", torch.int32), (mask, "mask", torch.uint8),
                    (spans, "spans", torch.int32), (num_spans, "num_spans", torch.int32)):
        _need(t, n, d, dev)
    if h8.shape != (T, H) or w8.shape != (V, H):
        raise ValueError("the e4m3 operands must have the shapes of hidden and weight")
    if dhidden is None:
        dhidden = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if dweight is None:
        dweight = torch.empty((V, H), dtype=torch.float32, device=dev)
    _need(dhidden, "dhidden", torch.bfloat16, dev)
    _need(dweight, "dweight", torch.float32, dev)
    if ws is None:
        ws = workspace(lmhead_bwd_fp8_workspace_size(T, H, V, vocab_chunk), dev)
    _lib.check(_lib.load().eas_lmhead_bwd_fp8(
        _ptr(g_logprob), _ptr(g_entropy), _ptr(hidden), _ptr(weight), _ptr(h8), _ptr(hidden_scale),
        _ptr(w8), _ptr(weight_scale), _ptr(targets), _ptr(mask), _ptr(spans), _ptr(num_spans),
        int(spans.shape[0]), _ptr(lse), _ptr(entropy), T, H, V, int(flags), int(vocab_chunk),
        _ptr(dhidden), _ptr(dweight), _ptr(ws), ws.numel(), _stream(dev)))
    return dhidden, dweight


def lmhead_fwd_shard(hidden, weight_shard, v_lo: int, targets, mask, spans, num_spans,
                     flags: int = EAS_ROWS_ACTIVE, ws=None, stats=None):
    """Per-token (M, S, U, z) statistics of one vocabulary shard ([T, 4] fp32)."""
    dev = hidden.device
    dt = hidden.dtype
    T, H = hidden.shape
    Vs = weight_shard.shape[0]
    for t, n, d in ((hidden, "hidden", dt), (weight_shard, "weight_shard", dt),
                    (targets, "targets", torch.int32), (mask, "mask", torch.uint8),
                    (spans, "spans", torch.int32), (num_spans, "num_spans", torch.int32)):
        _need(t, n, d, dev)
    if stats is None:
        stats = torch.empty((T, 4), dtype=torch.float32, device=dev)
    _need(stats, "stats", torch.float32, dev)
    if ws is None:
        ws = workspace(lmhead_workspace_size(T, H, Vs, dt), dev)
    _lib.check(_lib.load().eas_lmhead_fwd_shard(
        _ptr(hidden), _ptr(weight_shard), int(v_lo), _ptr(targets), _ptr(mask), _ptr(spans),
        _ptr(num_spans), int(spans.shape[0]), T, H, Vs, _dtype_code(dt), int(flags),
        _ptr(stats), _ptr(ws), ws.numel(), _stream(dev)))
    return stats


def lmhead_combine_shards(stats, mask, out=None, want_lse: bool = True):
    """Merges [n_shards, T, 4] shard statistics into (logprob, entropy, lse)."""
    dev = stats.device
    n, T = int(stats.shape[0]), int(stats.shape[1])
    _need(stats, "stats", torch.float32, dev)
    _need(mask, "mask", torch.uint8, dev)
    if out is None:
        out = tuple(torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
    lp, ent, lse = out
    if not want_lse:
        lse = None
    _lib.check(_lib.load().eas_lmhead_combine_shards(_ptr(stats), n, T, _ptr(mask), _ptr(lp),
                                                     _ptr(ent), _ptr(lse), _stream(dev)))
    return lp, ent, lse


def lmhead_bwd_shard(g_logprob, g_entropy, hidden, weight_shard, v_lo: int, targets, mask, spans,
                     num_spans, lse, entropy, flags: int = EAS_ROWS_ACTIVE, vocab_chunk: int = 0,
                     ws=None, dhidden_partial=None, dweight_shard=None):
    """This shard's dW rows and partial dHidden (the partials sum to dHidden)."""
    dev = hidden.device
    dt = hidden.dtype
    T, H = hidden.shape
    Vs = weight_shard.shape[0]
    for t, n in ((g_logprob, "g_logprob"), (g_entropy, "g_entropy"), (lse, "lse"),
                 (entropy, "entropy")):
        _need(t, n, torch.float32, dev)
    for t, n, d in ((hidden, "hidden", dt), (weight_shard, "weight_shard", dt),
                    (targets, "targets", torch.int32), (mask, "mask", torch.uint8),
                    (spans, "spans", torch.int32), (num_spans, "num_spans", torch.int32)):
        _need(t, n, d, dev)
    if dhidden_partial is None:
        dhidden_partial = torch.empty((T, H), dtype=dt, device=dev)
    if dweight_shard is None:
        dweight_shard = torch.empty((Vs, H), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(lmhead_workspace_size(T, H, Vs, dt, vocab_chunk), dev)
    _lib.check(_lib.load().eas_lmhead_bwd_shard(
        _ptr(g_logprob), _ptr(g_entropy), _ptr(hidden), _ptr(weight_shard), int(v_lo),
        _ptr(targets), _ptr(mask), _ptr(spans), _ptr(num_spans), int(spans.shape[0]), _ptr(lse),
        _ptr(entropy), T, H, Vs, _dtype_code(dt), int(flags), int(vocab_chunk),
        _ptr(dhidden_partial), _ptr(dweight_shard), _ptr(ws), ws.numel(), _stream(dev)))
    return dhidden_partial, dweight_shard


def read_device_status(ws: torch.Tensor) -> int:
    """Waits for the current stream and returns the status word in `ws` (0 = OK)."""
    st = _lib.load().eas_read_device_status(_ptr(ws), _stream(ws.device))
    return int(st)


def trace_enable(on: bool = True) -> None:
    """Start (clearing old records) or stop per-kernel event timing in the library."""
    _lib.load().eas_trace_enable(1 if on else 0)


def trace_read() -> list[tuple[str, float]]:
    """(kernel name, milliseconds) of every launch recorded since trace_enable(True)."""
    import ctypes
    lib = _lib.load()
    n = lib.eas_trace_read(None, None, 0)
    kinds = (ctypes.c_int32 * max(n, 1))()
    ms = (ctypes.c_float * max(n, 1))()
    n = lib.eas_trace_read(kinds, ms, n)
    return [(lib.eas_kernel_name(kinds[i]).decode(), float(ms[i])) for i in range(n)]


class FusedLMHeadLogprob(torch.autograd.Function):
    """Autograd wrapper: (hidden, weight) -> (logprob, entropy) of the active rows.

    The backward feeds the upstream gradients of logprob and entropy to
    lmhead_bwd; weight's gradient is returned in weight's dtype."""

    @staticmethod
    def forward(ctx, hidden, weight, targets, mask, spans, num_spans, flags, vocab_chunk):
        logprob, entropy, lse = lmhead_fwd(hidden, weight, targets, mask, spans, num_spans, flags)
        ctx.save_for_backward(hidden, weight, targets, mask, spans, num_spans, lse, entropy)
        ctx.flags, ctx.vocab_chunk = flags, vocab_chunk
        return logprob, entropy

    @staticmethod
    def backward(ctx, g_logprob, g_entropy):
        hidden, weight, targets, mask, spans, num_spans, lse, entropy = ctx.saved_tensors
        if g_logprob is None:
            g_logprob = torch.zeros_like(lse)
        if g_entropy is None:
            g_entropy = torch.zeros_like(lse)
        dh, dw = lmhead_bwd(g_logprob.contiguous().float(), g_entropy.contiguous().float(),
                            hidden, weight, targets, mask, spans, num_spans, lse, entropy,
                            ctx.flags, ctx.vocab_chunk)
        return dh, dw.to(weight.dtype), None, None, None, None, None, None


def fused_logprob_entropy(hidden, weight, targets, mask, spans=None, num_spans=None,
                          max_gap: int = 128, flags: int = EAS_ROWS_ACTIVE, vocab_chunk: int = 0):
    """Differentiable (logprob, entropy) of the active rows; builds the spans
    from the mask on the device when they are not given.  Under
    torch.no_grad() (or when neither input needs a gradient) it runs the
    forward alone and keeps no lse."""
    if spans is None or num_spans is None:
        spans, num_spans = build_active_spans(mask, max_gap)
    if not (torch.is_grad_enabled() and (hidden.requires_grad or weight.requires_grad)):
        lp, ent, _ = lmhead_fwd(hidden, weight, targets, mask, spans, num_spans, flags,
                                want_lse=False)
        return lp, ent
    return FusedLMHeadLogprob.apply(hidden, weight, targets, mask, spans, num_spans, flags,
                                    vocab_chunk)
