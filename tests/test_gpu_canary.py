"""Guard bytes around every buffer the library writes (the library's bounds check in
place of a memory checker).

Each output and workspace is carved out of a larger device allocation with 4 KiB
before it and at least 4 KiB after it filled with a byte pattern; the call goes
through the C ABI on ragged shapes (rows 1, 63, 64, 65, 127, 129, K and N tails,
experts without rows, single-row experts, the two-CTA kernels' phantom and half-pair
m-tiles, the one-launch FFN) and afterwards every guard byte must still hold the
pattern: no kernel stores outside the extent the header gives for its output.  The
problem page's requirements ask that inputs are not modified; the inputs are
checked unchanged too."""

import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import _native
from situ_glu_activation_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5
BF16 = 0  # SITU_BF16


class Guarded:
    """nbytes of device (or pinned host) memory between two guard regions."""

    def __init__(self, nbytes: int, dev, fill: int = 0, host: bool = False):
        self.n = int(nbytes)
        total = GUARD + ((self.n + 255) // 256) * 256 + GUARD
        if host:
            self.raw = torch.full((total,), PATTERN, dtype=torch.uint8).pin_memory()
        else:
            self.raw = torch.full((total,), PATTERN, dtype=torch.uint8, device=dev)
        self.raw[GUARD:GUARD + self.n].fill_(fill)

    @property
    def ptr(self) -> int:
        return self.raw.data_ptr() + GUARD

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self) -> bool:
        return bool((self.raw[:GUARD] == PATTERN).all()) and \
            bool((self.raw[GUARD + self.n:] == PATTERN).all())


def guarded_copy(t: torch.Tensor, dev) -> Guarded:
    """A guarded device copy of tensor t (an input whose neighbours are checked too)."""
    g = Guarded(t.numel() * t.element_size(), dev)
    g.view(t.dtype, t.shape).copy_(t)
    return g


def stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def lib():
    return _native.lib()


def ok(status: int, what: str):
    assert status == 0, f"{what}: status {status}"


def finish(bufs, inputs=()):
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    for name, g in bufs.items():
        assert g.intact(), f"{name}: a guard byte changed"
    for name, g, ref in inputs:
        assert g.intact() and torch.equal(g.raw, ref), f"input {name} changed"


def inputs_of(**tensors):
    """Guarded device copies of the inputs, plus their bytes to compare afterwards."""
    out = {}
    for name, t in tensors.items():
        g = guarded_copy(t, "cuda")
        out[name] = (g, g.raw.clone())
    return out


def unchanged(ins):
    return [(name, g, ref) for name, (g, ref) in ins.items()]


# ---------------------------------------------------------------------------
# standalone activation
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rows,I", [(1, 8), (63, 3072), (129, 100), (65, 4)])
def test_act(cuda_dev, rows, I):
    g = wl.normal((rows, 2 * I), 3.0, seed=rows).bfloat16()
    ins = inputs_of(g=g)
    out = Guarded(rows * I * 2, cuda_dev)
    ok(lib().situ_glu_act(ins["g"][0].ptr, out.ptr, rows, I, 4.0, 25.0, BF16, stream()), "act")
    finish({"out": out}, unchanged(ins))


# ---------------------------------------------------------------------------
# dense FFN: one launch, two launches, the halves, training step
# ---------------------------------------------------------------------------
SHAPES = [(1, 128, 256), (63, 136, 200), (64, 256, 128), (65, 128, 384), (127, 192, 264),
          (129, 136, 200), (333, 256, 384)]


@pytest.mark.parametrize("single", [True, False])
@pytest.mark.parametrize("R,M,I", SHAPES)
def test_ffn_forward(cuda_dev, R, M, I, single):
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=R)
    ins = inputs_of(x=x, wgu=wgu, wd=wd)
    y = Guarded(R * M * 2, cuda_dev)
    wsb = lib().situ_ffn_workspace_size(R, M, I, BF16)
    ws = Guarded(wsb, cuda_dev)
    prev = situ.ffn_set_single_launch(single)
    try:
        ok(lib().situ_ffn_forward(ins["x"][0].ptr, ins["wgu"][0].ptr, ins["wd"][0].ptr, y.ptr,
                                  ws.ptr, wsb, R, M, I, 4.0, 25.0, BF16, stream()), "ffn")
    finally:
        situ.ffn_set_single_launch(prev)
    finish({"y": y, "workspace": ws}, unchanged(ins))


@pytest.mark.parametrize("R,M,I", SHAPES[:4])
def test_ffn_halves(cuda_dev, R, M, I):
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=R + 1)
    ins = inputs_of(x=x, wgu=wgu, wd=wd)
    h = Guarded(R * I * 2, cuda_dev)
    y = Guarded(R * M * 2, cuda_dev)
    ok(lib().situ_ffn_gate_up(ins["x"][0].ptr, ins["wgu"][0].ptr, h.ptr, R, M, I, 4.0, 25.0,
                              BF16, stream()), "gate_up")
    ok(lib().situ_ffn_down(h.ptr, ins["wd"][0].ptr, y.ptr, R, M, I, BF16, stream()), "down")
    finish({"h": h, "y": y}, unchanged(ins))


@pytest.mark.parametrize("R,M,I", [(1, 128, 256), (65, 136, 200), (129, 256, 384)])
def test_ffn_training_step(cuda_dev, R, M, I):
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=R + 2)
    dy = wl.normal((R, M), 1.0, seed=R + 3).bfloat16()
    ins = inputs_of(x=x, wgu=wgu, wd=wd, dy=dy)
    y, gu, h = (Guarded(R * c * 2, cuda_dev) for c in (M, 2 * I, I))
    ok(lib().situ_ffn_forward_train(ins["x"][0].ptr, ins["wgu"][0].ptr, ins["wd"][0].ptr, y.ptr,
                                    gu.ptr, h.ptr, R, M, I, 4.0, 25.0, BF16, stream()), "train")
    dx = Guarded(R * M * 2, cuda_dev)
    dwg = Guarded(2 * I * M * 2, cuda_dev)
    dwd = Guarded(M * I * 2, cuda_dev)
    wsb = lib().situ_ffn_backward_workspace_size(R, M, I, BF16)
    ws = Guarded(wsb, cuda_dev)
    ok(lib().situ_ffn_backward(ins["x"][0].ptr, ins["wgu"][0].ptr, ins["wd"][0].ptr, gu.ptr,
                               h.ptr, ins["dy"][0].ptr, dx.ptr, dwg.ptr, dwd.ptr, ws.ptr, wsb, R,
                               M, I, 4.0, 25.0, BF16, stream()), "backward")
    finish({"y": y, "gu": gu, "h": h, "dx": dx, "dW_gate_up": dwg, "dW_down": dwd,
            "workspace": ws}, unchanged(ins))


def test_ffn_host_buffers(cuda_dev):
    R, M, I = 333, 136, 200
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=4)
    xh = Guarded(R * M * 2, cuda_dev, host=True)
    xh.view(torch.bfloat16, (R, M)).copy_(x)
    xh_ref = xh.raw.clone()
    ins = inputs_of(wgu=wgu, wd=wd)
    yh = Guarded(R * M * 2, cuda_dev, host=True)
    wsb = lib().situ_ffn_host_workspace_size(R, M, I, BF16, 128)
    ws = Guarded(wsb, cuda_dev)
    ok(lib().situ_ffn_forward_host(xh.ptr, ins["wgu"][0].ptr, ins["wd"][0].ptr, yh.ptr, ws.ptr,
                                   wsb, R, M, I, 128, 4.0, 25.0, BF16, stream()), "host")
    finish({"y_host": yh, "workspace": ws}, unchanged(ins))
    assert torch.equal(xh.raw, xh_ref)


# ---------------------------------------------------------------------------
# routed experts
# ---------------------------------------------------------------------------
def _routes(sizes, k, seed):
    """ids [T, k] whose expert e gets about sizes[e] routes (exactly, for k = 1)."""
    ids = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
    ids = ids[torch.randperm(ids.numel(), generator=torch.Generator().manual_seed(seed))]
    T = ids.numel() // k
    return ids[:T * k].view(T, k).contiguous()


def _index(ids, E, dev):
    n = ids.numel()
    ins = inputs_of(ids=ids)
    off = Guarded((E + 1) * 4, dev)
    tix = Guarded(n * 4, dev)
    wsb = lib().situ_moe_index_workspace_size(n, E)
    ws = Guarded(wsb, dev)
    ok(lib().situ_moe_build_index(ins["ids"][0].ptr, off.ptr, tix.ptr, ws.ptr, wsb, n, E,
                                  stream()), "index")
    finish({"offsets": off, "token_index": tix, "index workspace": ws}, unchanged(ins))
    return off, tix


GROUPED = [
    ((20, 0, 7, 33, 1, 12), 1),          # one-CTA: empty and single-row experts
    ((300, 290, 0, 140, 77), 1),         # two-CTA: half-pair tails, an empty expert
    ((129, 192, 64, 385, 1), 1),         # phantom m-tiles, a 64-row and a 1-row expert
    ((60, 44, 90, 30, 12, 70), 2),       # two slots per token
]


@pytest.mark.parametrize("sizes,k", GROUPED)
def test_grouped_forward_and_combine(cuda_dev, sizes, k):
    E, M, I = len(sizes), 136, 200
    ids = _routes(sizes, k, seed=len(sizes))
    T = ids.shape[0]
    off, tix = _index(ids, E, cuda_dev)
    x = wl.normal((T, M), 1.0, seed=5).bfloat16()
    wgu, wd = wl.expert_weights(E, M, I, seed=6)
    w = torch.rand(T, k, generator=torch.Generator().manual_seed(7))
    ins = inputs_of(x=x, wgu=wgu, wd=wd, w=w)
    y = Guarded(T * k * M * 2, cuda_dev)
    R = T * k
    wsb = lib().situ_moe_workspace_size(R, E, M, I, BF16)
    ws = Guarded(wsb, cuda_dev)
    ok(lib().situ_moe_grouped_forward(ins["x"][0].ptr, off.ptr, tix.ptr, ins["wgu"][0].ptr,
                                      ins["wd"][0].ptr, y.ptr, ws.ptr, wsb, T, k, E, M, I, 4.0,
                                      25.0, BF16, stream()), "grouped")
    out = Guarded(T * M * 2, cuda_dev)
    ok(lib().situ_moe_combine(y.ptr, ins["w"][0].ptr, out.ptr, T, k, M, BF16, stream()),
       "combine")
    out2 = Guarded(T * M * 2, cuda_dev)
    wsb2 = lib().situ_moe_combined_workspace_size(T, k, E, M, I, BF16)
    ws2 = Guarded(wsb2, cuda_dev)
    ok(lib().situ_moe_grouped_forward_combined(
        ins["x"][0].ptr, off.ptr, tix.ptr, ins["wgu"][0].ptr, ins["wd"][0].ptr, ins["w"][0].ptr,
        out2.ptr, ws2.ptr, wsb2, T, k, E, M, I, 4.0, 25.0, BF16, stream()), "combined")
    finish({"y": y, "workspace": ws, "out": out, "fused out": out2, "fused workspace": ws2,
            "offsets": off, "token_index": tix}, unchanged(ins))


@pytest.mark.parametrize("sizes,k", GROUPED)
def test_grouped_training_step(cuda_dev, sizes, k):
    E, M, I = len(sizes), 136, 200
    ids = _routes(sizes, k, seed=len(sizes) + 1)
    T = ids.shape[0]
    R = T * k
    off, tix = _index(ids, E, cuda_dev)
    x = wl.normal((T, M), 1.0, seed=8).bfloat16()
    dy = wl.normal((T, k, M), 1.0, seed=9).bfloat16()
    wgu, wd = wl.expert_weights(E, M, I, seed=10)
    ins = inputs_of(x=x, wgu=wgu, wd=wd, dy=dy)
    y = Guarded(R * M * 2, cuda_dev)
    gu = Guarded(R * 2 * I * 2, cuda_dev)
    h = Guarded(R * I * 2, cuda_dev)
    wsb = lib().situ_moe_workspace_size(R, E, M, I, BF16)
    ws = Guarded(wsb, cuda_dev)
    ok(lib().situ_moe_grouped_forward_train(ins["x"][0].ptr, off.ptr, tix.ptr, ins["wgu"][0].ptr,
                                            ins["wd"][0].ptr, y.ptr, gu.ptr, h.ptr, ws.ptr, wsb,
                                            T, k, E, M, I, 4.0, 25.0, BF16, stream()), "train fwd")
    dx = Guarded(T * M * 2, cuda_dev)
    dwg = Guarded(E * 2 * I * M * 2, cuda_dev)
    dwd = Guarded(E * M * I * 2, cuda_dev)
    wsb2 = lib().situ_moe_backward_workspace_size(R, E, M, I, BF16)
    ws2 = Guarded(wsb2, cuda_dev)
    ok(lib().situ_moe_grouped_backward(ins["x"][0].ptr, off.ptr, tix.ptr, ins["wgu"][0].ptr,
                                       ins["wd"][0].ptr, gu.ptr, h.ptr, ins["dy"][0].ptr, dx.ptr,
                                       dwg.ptr, dwd.ptr, ws2.ptr, wsb2, T, k, E, M, I, 4.0, 25.0,
                                       BF16, stream()), "backward")
    finish({"y": y, "gu": gu, "h": h, "workspace": ws, "dx": dx, "dW_gate_up": dwg,
            "dW_down": dwd, "backward workspace": ws2}, unchanged(ins))


# ---------------------------------------------------------------------------
# MX experts
# ---------------------------------------------------------------------------
def _mx_weights(W, E, M, I, kind, fmt, dev):
    rows, K = (2 * I, M) if kind == situ.MX_GATE_UP else (M, I)
    codes = Guarded(E * rows * (K // 2 if fmt == situ.MX_E2M1 else K), dev)
    scales = Guarded(lib().situ_mx_weight_scales_size(E, M, I, kind), dev)
    ok(lib().situ_mx_quantize_weights(W.ptr, codes.ptr, scales.ptr, E, M, I, kind, fmt,
                                      stream()), "quantize weights")
    return codes, scales


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("R", [1, 129, 333])
def test_mx_dense(cuda_dev, R, fmt):
    M, I = 256, 384
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=R + 11)
    ins = inputs_of(x=x, wgu=wgu, wd=wd)
    gc, gs = _mx_weights(ins["wgu"][0], 1, M, I, situ.MX_GATE_UP, fmt, cuda_dev)
    dc, ds = _mx_weights(ins["wd"][0], 1, M, I, situ.MX_DOWN, fmt, cuda_dev)
    xc = Guarded(R * M, cuda_dev)
    xs = Guarded(lib().situ_mx_act_scales_size(R, M), cuda_dev)
    ok(lib().situ_mx_quantize_act(ins["x"][0].ptr, xc.ptr, xs.ptr, R, M, stream()), "quantize x")
    h = Guarded(R * I * 2, cuda_dev)
    ok(lib().situ_ffn_gate_up_mxfp8(xc.ptr, xs.ptr, gc.ptr, gs.ptr, fmt, h.ptr, R, M, I, 4.0,
                                    25.0, stream()), "mx gate_up")
    y = Guarded(R * M * 2, cuda_dev)
    wsb = lib().situ_ffn_mxfp8_workspace_size(R, M, I)
    ws = Guarded(wsb, cuda_dev)
    ok(lib().situ_ffn_forward_mxfp8(ins["x"][0].ptr, gc.ptr, gs.ptr, dc.ptr, ds.ptr, fmt, y.ptr,
                                    ws.ptr, wsb, R, M, I, 4.0, 25.0, stream()), "mx ffn")
    finish({"wgu codes": gc, "wgu scales": gs, "wd codes": dc, "wd scales": ds, "x codes": xc,
            "x scales": xs, "h": h, "y": y, "workspace": ws}, unchanged(ins))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("sizes", [(20, 0, 7, 33, 1, 12),   # one-CTA block-scaled kernels
                                   (700, 600, 0, 900)])    # two-CTA, a phantom m-tile
def test_mx_grouped(cuda_dev, sizes, fmt):
    E, M, I = len(sizes), 256, 384
    ids = _routes(sizes, 1, seed=12)
    T = ids.shape[0]
    off, tix = _index(ids, E, cuda_dev)
    x = wl.normal((T, M), 1.0, seed=13).bfloat16()
    wgu, wd = wl.expert_weights(E, M, I, seed=14)
    ins = inputs_of(x=x, wgu=wgu, wd=wd)
    gc, gs = _mx_weights(ins["wgu"][0], E, M, I, situ.MX_GATE_UP, fmt, cuda_dev)
    dc, ds = _mx_weights(ins["wd"][0], E, M, I, situ.MX_DOWN, fmt, cuda_dev)
    y = Guarded(T * M * 2, cuda_dev)
    wsb = lib().situ_moe_mxfp8_workspace_size(T, E, M, I)
    ws = Guarded(wsb, cuda_dev)
    ok(lib().situ_moe_grouped_forward_mxfp8(ins["x"][0].ptr, off.ptr, tix.ptr, gc.ptr, gs.ptr,
                                            dc.ptr, ds.ptr, fmt, y.ptr, ws.ptr, wsb, T, 1, E, M,
                                            I, 4.0, 25.0, stream()), "mx grouped")
    finish({"wgu codes": gc, "wgu scales": gs, "wd codes": dc, "wd scales": ds, "y": y,
            "workspace": ws}, unchanged(ins))
