"""Guard bands.  Every buffer the library writes (spans, workspaces, logprob,
entropy, lse, dHidden, dW, e4m3 codes and scales) is handed to it as the middle
of a larger allocation whose margins hold a canary byte.  After the spans,
the forward and the backward, every margin must still hold it, so no kernel
writes outside the bytes it was given.  The oracle comparisons of the other
tests look only inside the outputs; these look around them."""
import numpy as np
import pytest
import torch

import entropy_active_span_gb300 as eas
from gpu_helpers import small_inputs, to_dev

pytestmark = pytest.mark.gpu

PAD = 4096        # canary bytes on each side; keeps every view 512-byte aligned
CANARY = 0xA5


class Guarded:
    """Allocations with canary margins; views of their middles."""

    def __init__(self, dev):
        self.dev = dev
        self.bufs = []

    def view(self, shape, dtype):
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((nbytes + 2 * PAD,), CANARY, dtype=torch.uint8, device=self.dev)
        self.bufs.append((buf, nbytes))
        return buf[PAD:PAD + nbytes].view(dtype).view(shape)

    def bytes(self, nbytes):
        return self.view((max(int(nbytes), 1),), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        for i, (buf, nbytes) in enumerate(self.bufs):
            b = buf.cpu().numpy()
            assert (b[:PAD] == CANARY).all(), f"buffer {i}: bytes written before its start"
            assert (b[PAD + nbytes:] == CANARY).all(), f"buffer {i}: bytes written past its end"


def run_guarded(inp, dtype, vocab_chunk, flags):
    g = Guarded(torch.device("cuda", 0))
    T, H = inp["hidden"].shape
    V = inp["weight"].shape[0]
    hidden, weight = to_dev(inp["hidden"]), to_dev(inp["weight"])
    targets, mask = to_dev(inp["targets"]), to_dev(inp["mask"].astype(np.uint8))
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    cap = (T + 1) // 2
    spans = g.view((cap, 2), torch.int32)
    ns = g.view((1,), torch.int32)
    sws = g.bytes(eas.spans_workspace_size(T))
    eas.build_active_spans(mask, 128, spans=spans, num_spans=ns, ws=sws)
    ws = g.bytes(eas.lmhead_workspace_size(T, H, V, hidden.dtype, vocab_chunk))
    out = tuple(g.view((T,), torch.float32) for _ in range(3))
    lp, ent, lse = eas.lmhead_fwd(hidden, weight, targets, mask, spans, ns, flags, ws=ws, out=out)
    dh = g.view((T, H), hidden.dtype)
    dw = g.view((V, H), torch.float32)
    eas.lmhead_bwd(glp, gh, hidden, weight, targets, mask, spans, ns, lse, ent,
                   flags | eas.EAS_REUSE_FWD_ROWS, vocab_chunk, ws=ws, dhidden=dh, dweight=dw)
    assert eas.read_device_status(ws) == 0
    g.check()
    # the outputs themselves are written where they should be: finite, and
    # inactive rows are zero
    act = torch.from_numpy(inp["mask"] != 0)
    assert torch.isfinite(dw.cpu()).all() and torch.isfinite(dh.float().cpu()).all()
    assert (lp.cpu()[~act] == 0).all() and (dh.float().cpu()[~act] == 0).all()


@pytest.mark.parametrize("T,H,V,chunk,mask_kind,flags", [
    (777, 320, 1537, 512, "bernoulli0.6", eas.EAS_ROWS_ACTIVE),     # ragged everything
    (777, 320, 1537, 512, "bernoulli0.6", eas.EAS_ROWS_SPAN),
    (300, 1088, 2100, 1088, "bernoulli0.3", eas.EAS_ROWS_ACTIVE),   # a last row tile of 128 rows or fewer
    (1024, 512, 4096, 0, "bernoulli1.0", eas.EAS_ROWS_ACTIVE),      # every tile full
])
def test_bf16_writes_stay_inside_their_buffers(T, H, V, chunk, mask_kind, flags):
    inp = small_inputs(T, H, V, seed=T + H, mask_kind=mask_kind, w_std=3.0)
    run_guarded(inp, "bf16", chunk, flags)


def test_fp32_writes_stay_inside_their_buffers():
    inp = small_inputs(333, 96, 700, dtype="fp32", seed=5, mask_kind="bernoulli0.5", w_std=3.0)
    run_guarded(inp, "fp32", 256, eas.EAS_ROWS_ACTIVE)


def test_e4m3_writes_stay_inside_their_buffers():
    T, H, V, chunk = 600, 384, 1800, 768
    inp = small_inputs(T, H, V, seed=17, mask_kind="bernoulli0.6", w_std=3.0)
    g = Guarded(torch.device("cuda", 0))
    hidden, weight = to_dev(inp["hidden"]), to_dev(inp["weight"])
    targets, mask = to_dev(inp["targets"]), to_dev(inp["mask"].astype(np.uint8))
    glp, gh = to_dev(inp["g_logprob"]), to_dev(inp["g_entropy"])
    h8 = g.view((T, H), torch.uint8)
    hs = g.view((T,), torch.float32)
    w8 = g.view((V, H), torch.uint8)
    wsc = g.view((V,), torch.float32)
    eas.quantize_rows_e4m3(hidden, out=h8, scale=hs)
    eas.quantize_rows_e4m3(weight, out=w8, scale=wsc)
    spans, ns = eas.build_active_spans(mask, 128)
    ws = g.bytes(max(eas.lmhead_workspace_size(T, H, V, torch.uint8),
                     eas.lmhead_bwd_fp8_workspace_size(T, H, V, chunk)))
    out = tuple(g.view((T,), torch.float32) for _ in range(3))
    lp, ent, lse = eas.lmhead_fwd_fp8(h8, hs, w8, wsc, targets, mask, spans, ns, ws=ws, out=out)
    dh = g.view((T, H), torch.bfloat16)
    dw = g.view((V, H), torch.float32)
    eas.lmhead_bwd_fp8(glp, gh, hidden, weight, h8, hs, w8, wsc, targets, mask, spans, ns, lse,
                       ent, vocab_chunk=chunk, ws=ws, dhidden=dh, dweight=dw)
    assert eas.read_device_status(ws) == 0
    g.check()
    assert torch.isfinite(dw.cpu()).all() and torch.isfinite(dh.float().cpu()).all()
