"""Python front end of libsitu over PyTorch tensors.

Argument marshalling only: shapes are checked, leading dimensions flattened,
outputs and workspaces allocated with PyTorch on the input's device, and the
matching C entry point (include/situ.h) launched on PyTorch's current stream.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback, and a missing library raises.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _native
from ._native import SITU_BF16, SITU_F32, SituError, check

_DTYPES = {torch.bfloat16: SITU_BF16, torch.float32: SITU_F32}


def _dt(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}: bfloat16 or float32 expected") from None


def _cuda_contig(name: str, t: torch.Tensor) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def caps(beta, linear_beta):
    """The caps as the C ABI takes them.

    Follows the activation module of "Kimi K3 - Bound the up branch": a gate cap
    of None (or 0) becomes 1.0 (its ``beta or 1.0``), an up cap of None leaves the
    up branch uncapped, passed as +infinity (the limit beta -> infinity of
    beta tanh(x/beta) is x).  +infinity for both caps is SwiGLU.
    """
    b1 = 1.0 if not beta else float(beta)
    b2 = float("inf") if linear_beta is None else float(linear_beta)
    return b1, b2


def situ_glu_act(gate_up: torch.Tensor, beta: float = 4.0, linear_beta: float = 25.0,
                 out: torch.Tensor | None = None) -> torch.Tensor:
    """SiTU-GLU of a packed [..., 2I] tensor -> [..., I], same dtype.

    The first half of the last dimension is the gate projection g, the second
    half the up projection u; out = beta*tanh(g/beta)*sigmoid(g) *
    linear_beta*tanh(u/linear_beta), computed in FP32 and rounded once.
    """
    _cuda_contig("gate_up", gate_up)
    if gate_up.shape[-1] % 2:
        raise ValueError("the last dimension of gate_up must be even")
    I = gate_up.shape[-1] // 2
    rows = gate_up.numel() // max(gate_up.shape[-1], 1)
    if out is None:
        out = torch.empty(*gate_up.shape[:-1], I, dtype=gate_up.dtype, device=gate_up.device)
    else:
        _cuda_contig("out", out)
        if out.shape != (*gate_up.shape[:-1], I) or out.dtype != gate_up.dtype:
            raise ValueError("out has the wrong shape or dtype")
    if rows == 0 or I == 0:
        return out
    lib = _native.lib()
    check("situ_glu_act", lib.situ_glu_act(gate_up.data_ptr(), out.data_ptr(), rows, I,
                                           *caps(beta, linear_beta), _dt(gate_up),
                                           _stream(gate_up.device)))
    return out


def ffn_workspace_bytes(R: int, M: int, I: int, dtype=torch.bfloat16) -> int:
    return int(_native.lib().situ_ffn_workspace_size(R, M, I, _DTYPES[dtype]))


def situ_ffn_forward(x: torch.Tensor, W_gate_up: torch.Tensor, W_down: torch.Tensor,
                     beta: float = 4.0, linear_beta: float = 25.0,
                     y: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Dense SiTU-GLU feed-forward: y = (SiTU-GLU(x W_gate_up^T)) W_down^T.

    x [..., M]; W_gate_up [2I, M] (gate rows then up rows); W_down [M, I].
    """
    for n, t in (("x", x), ("W_gate_up", W_gate_up), ("W_down", W_down)):
        _cuda_contig(n, t)
        if t.dtype != x.dtype:
            raise TypeError("x and the weights must share a dtype")
    M = x.shape[-1]
    I = W_gate_up.shape[0] // 2
    if W_gate_up.shape != (2 * I, M) or W_down.shape != (M, I):
        raise ValueError(f"weights {tuple(W_gate_up.shape)}, {tuple(W_down.shape)} do not "
                         f"match M={M}")
    R = x.numel() // M if M else 0
    if y is None:
        y = torch.empty_like(x)
    else:
        _cuda_contig("y", y)
        if y.shape != x.shape or y.dtype != x.dtype:
            raise ValueError("y has the wrong shape or dtype")
    if R == 0:
        return y
    lib = _native.lib()
    need = int(lib.situ_ffn_workspace_size(R, M, I, _dt(x)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    check("situ_ffn_forward",
          lib.situ_ffn_forward(x.data_ptr(), W_gate_up.data_ptr(), W_down.data_ptr(),
                               y.data_ptr(), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), R, M, I,
                               *caps(beta, linear_beta), _dt(x), _stream(x.device)))
    return y


def situ_ffn_forward_host(x_host: torch.Tensor, W_gate_up: torch.Tensor, W_down: torch.Tensor,
                          beta: float = 4.0, linear_beta: float = 25.0,
                          y_host: torch.Tensor | None = None, chunk_rows: int = 0,
                          workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Dense SiTU-GLU FFN with x and y in (pinned) host memory.

    Row chunks are pipelined so host->device copies, the GEMMs and device->host
    copies overlap; returns y_host, complete once the current stream is synchronised.
    """
    if x_host.is_cuda or not x_host.is_contiguous():
        raise ValueError("x_host must be a contiguous host tensor")
    for n, t in (("W_gate_up", W_gate_up), ("W_down", W_down)):
        _cuda_contig(n, t)
        if t.dtype != x_host.dtype:
            raise TypeError("x_host and the weights must share a dtype")
    M = x_host.shape[-1]
    I = W_gate_up.shape[0] // 2
    if W_gate_up.shape != (2 * I, M) or W_down.shape != (M, I):
        raise ValueError("weight shapes do not match x_host")
    R = x_host.numel() // M if M else 0
    if y_host is None:
        y_host = torch.empty(x_host.shape, dtype=x_host.dtype, pin_memory=True)
    elif y_host.is_cuda or y_host.shape != x_host.shape or not y_host.is_contiguous():
        raise ValueError("y_host must be a contiguous host tensor shaped like x_host")
    if R == 0:
        return y_host
    lib = _native.lib()
    need = int(lib.situ_ffn_host_workspace_size(R, M, I, _dt(x_host), chunk_rows))
    dev = W_gate_up.device
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    check("situ_ffn_forward_host",
          lib.situ_ffn_forward_host(x_host.data_ptr(), W_gate_up.data_ptr(), W_down.data_ptr(),
                                    y_host.data_ptr(), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(), R, M, I,
                                    chunk_rows, *caps(beta, linear_beta), _dt(x_host),
                                    _stream(dev)))
    return y_host


def ffn_host_workspace_bytes(R: int, M: int, I: int, chunk_rows: int = 0,
                             dtype=torch.bfloat16) -> int:
    return int(_native.lib().situ_ffn_host_workspace_size(R, M, I, _DTYPES[dtype], chunk_rows))


def situ_ffn_gate_up(x: torch.Tensor, W_gate_up: torch.Tensor, beta: float = 4.0,
                     linear_beta: float = 25.0, h: torch.Tensor | None = None) -> torch.Tensor:
    """h = SiTU-GLU(x W_gate_up^T) [..., I], bf16: one tcgen05 GEMM, activation fused."""
    _cuda_contig("x", x)
    _cuda_contig("W_gate_up", W_gate_up)
    M = x.shape[-1]
    I = W_gate_up.shape[0] // 2
    if W_gate_up.shape != (2 * I, M) or W_gate_up.dtype != x.dtype:
        raise ValueError("W_gate_up must be [2I, M] of x's dtype")
    R = x.numel() // M if M else 0
    if h is None:
        h = torch.empty(*x.shape[:-1], I, dtype=x.dtype, device=x.device)
    if R == 0:
        return h
    check("situ_ffn_gate_up",
          _native.lib().situ_ffn_gate_up(x.data_ptr(), W_gate_up.data_ptr(), h.data_ptr(), R, M,
                                         I, *caps(beta, linear_beta), _dt(x),
                                         _stream(x.device)))
    return h


def situ_ffn_down(h: torch.Tensor, W_down: torch.Tensor,
                  y: torch.Tensor | None = None) -> torch.Tensor:
    """y = h W_down^T [..., M], bf16 tcgen05 GEMM."""
    _cuda_contig("h", h)
    _cuda_contig("W_down", W_down)
    I = h.shape[-1]
    M = W_down.shape[0]
    if W_down.shape != (M, I) or W_down.dtype != h.dtype:
        raise ValueError("W_down must be [M, I] of h's dtype")
    R = h.numel() // I if I else 0
    if y is None:
        y = torch.empty(*h.shape[:-1], M, dtype=h.dtype, device=h.device)
    if R == 0:
        return y
    check("situ_ffn_down",
          _native.lib().situ_ffn_down(h.data_ptr(), W_down.data_ptr(), y.data_ptr(), R, M, I,
                                      _dt(h), _stream(h.device)))
    return y


def situ_ffn_forward_train(x: torch.Tensor, W_gate_up: torch.Tensor, W_down: torch.Tensor,
                           beta: float = 4.0, linear_beta: float = 25.0):
    """Training forward of the dense FFN (bf16): returns (y, gu, h) where gu [R, 2I]
    is the pre-activation (gate then up columns) and h [R, I] the activation, both
    kept for situ_ffn_backward."""
    for n, t in (("x", x), ("W_gate_up", W_gate_up), ("W_down", W_down)):
        _cuda_contig(n, t)
    M = x.shape[-1]
    I = W_gate_up.shape[0] // 2
    if W_gate_up.shape != (2 * I, M) or W_down.shape != (M, I):
        raise ValueError("weight shapes do not match x")
    R = x.numel() // M
    y = torch.empty_like(x)
    gu = torch.empty(R, 2 * I, dtype=x.dtype, device=x.device)
    h = torch.empty(R, I, dtype=x.dtype, device=x.device)
    if R:
        check("situ_ffn_forward_train",
              _native.lib().situ_ffn_forward_train(x.data_ptr(), W_gate_up.data_ptr(),
                                                   W_down.data_ptr(), y.data_ptr(), gu.data_ptr(),
                                                   h.data_ptr(), R, M, I,
                                                   *caps(beta, linear_beta), _dt(x),
                                                   _stream(x.device)))
    return y, gu, h


def situ_ffn_backward(x: torch.Tensor, W_gate_up: torch.Tensor, W_down: torch.Tensor,
                      gu: torch.Tensor, h: torch.Tensor, dy: torch.Tensor, beta: float = 4.0,
                      linear_beta: float = 25.0, workspace: torch.Tensor | None = None):
    """Backward of the dense FFN for upstream dy [R, M] (bf16): returns
    (dx [R, M], dW_gate_up [2I, M], dW_down [M, I])."""
    for n, t in (("x", x), ("W_gate_up", W_gate_up), ("W_down", W_down), ("gu", gu), ("h", h),
                 ("dy", dy)):
        _cuda_contig(n, t)
    M = x.shape[-1]
    I = W_gate_up.shape[0] // 2
    R = x.numel() // M
    if gu.shape != (R, 2 * I) or h.shape != (R, I) or dy.numel() != R * M:
        raise ValueError("gu, h or dy do not match x and the weights")
    dx = torch.empty_like(x)
    dwg = torch.empty_like(W_gate_up)
    dwd = torch.empty_like(W_down)
    lib = _native.lib()
    need = int(lib.situ_ffn_backward_workspace_size(R, M, I, _dt(x)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    check("situ_ffn_backward",
          lib.situ_ffn_backward(x.data_ptr(), W_gate_up.data_ptr(), W_down.data_ptr(),
                                gu.data_ptr(), h.data_ptr(), dy.data_ptr(), dx.data_ptr(),
                                dwg.data_ptr(), dwd.data_ptr(), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), R, M, I,
                                *caps(beta, linear_beta), _dt(x), _stream(x.device)))
    return dx, dwg, dwd


def ffn_backward_workspace_bytes(R: int, M: int, I: int) -> int:
    return int(_native.lib().situ_ffn_backward_workspace_size(R, M, I, SITU_BF16))


def situ_moe_build_index(expert_ids: torch.Tensor, num_experts: int,
                         expert_offsets: torch.Tensor | None = None,
                         token_index: torch.Tensor | None = None):
    """Stable counting sort of flat routes by expert.

    expert_ids [T, k_eff] (or flat) int32 on the GPU ->
    (expert_offsets [E+1] int32, token_index [T*k_eff] int32).
    """
    _cuda_contig("expert_ids", expert_ids)
    if expert_ids.dtype != torch.int32:
        raise TypeError("expert_ids must be int32")
    n = expert_ids.numel()
    dev = expert_ids.device
    if expert_offsets is None:
        expert_offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    if token_index is None:
        token_index = torch.empty(n, dtype=torch.int32, device=dev)
    lib = _native.lib()
    need = int(lib.situ_moe_index_workspace_size(n, num_experts))
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    check("situ_moe_build_index",
          lib.situ_moe_build_index(expert_ids.data_ptr(), expert_offsets.data_ptr(),
                                   token_index.data_ptr(), ws.data_ptr(), ws.numel(), n,
                                   num_experts, _stream(dev)))
    return expert_offsets, token_index


def moe_workspace_bytes(R: int, E: int, M: int, I: int) -> int:
    return int(_native.lib().situ_moe_workspace_size(R, E, M, I, SITU_BF16))


def situ_moe_grouped_forward(x: torch.Tensor, expert_offsets: torch.Tensor,
                             token_index: torch.Tensor, W_gate_up: torch.Tensor,
                             W_down: torch.Tensor, k_eff: int, beta: float = 4.0,
                             linear_beta: float = 25.0, y: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Grouped SiTU-GLU experts: y[t, s] = FFN_{expert of (t, s)}(x[t]).

    x [T, M] bf16; expert_offsets [E+1], token_index [T*k_eff] int32 (from
    situ_moe_build_index); W_gate_up [E, 2I, M], W_down [E, M, I] bf16, stacked.
    Returns y [T, k_eff, M].
    """
    for n, t in (("x", x), ("expert_offsets", expert_offsets), ("token_index", token_index),
                 ("W_gate_up", W_gate_up), ("W_down", W_down)):
        _cuda_contig(n, t)
    T, M = x.shape
    E, twoI, _ = W_gate_up.shape
    I = twoI // 2
    if W_gate_up.shape != (E, 2 * I, M) or W_down.shape != (E, M, I):
        raise ValueError("stacked weight shapes do not match x")
    if expert_offsets.numel() != E + 1 or token_index.numel() != T * k_eff:
        raise ValueError("index arrays do not match E and T*k_eff")
    if y is None:
        y = torch.empty(T, k_eff, M, dtype=x.dtype, device=x.device)
    R = T * k_eff
    if R == 0:
        return y
    lib = _native.lib()
    need = int(lib.situ_moe_workspace_size(R, E, M, I, _dt(x)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    check("situ_moe_grouped_forward",
          lib.situ_moe_grouped_forward(x.data_ptr(), expert_offsets.data_ptr(),
                                       token_index.data_ptr(), W_gate_up.data_ptr(),
                                       W_down.data_ptr(), y.data_ptr(), workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(), T,
                                       k_eff, E, M, I, *caps(beta, linear_beta),
                                       _dt(x), _stream(x.device)))
    return y


def _moe_shapes(x, expert_offsets, token_index, W_gate_up, W_down, k_eff):
    for n, t in (("x", x), ("expert_offsets", expert_offsets), ("token_index", token_index),
                 ("W_gate_up", W_gate_up), ("W_down", W_down)):
        _cuda_contig(n, t)
    T, M = x.shape
    E, twoI, _ = W_gate_up.shape
    I = twoI // 2
    if W_gate_up.shape != (E, 2 * I, M) or W_down.shape != (E, M, I):
        raise ValueError("stacked weight shapes do not match x")
    if expert_offsets.numel() != E + 1 or token_index.numel() != T * k_eff:
        raise ValueError("index arrays do not match E and T*k_eff")
    return T, M, E, I


def situ_moe_grouped_forward_train(x: torch.Tensor, expert_offsets: torch.Tensor,
                                   token_index: torch.Tensor, W_gate_up: torch.Tensor,
                                   W_down: torch.Tensor, k_eff: int, beta: float = 4.0,
                                   linear_beta: float = 25.0,
                                   workspace: torch.Tensor | None = None):
    """Training forward of the grouped experts: returns (y [T, k_eff, M], gu [R, 2I],
    h [R, I]) with gu and h in expert order (row r is route token_index[r]), kept
    for situ_moe_grouped_backward."""
    T, M, E, I = _moe_shapes(x, expert_offsets, token_index, W_gate_up, W_down, k_eff)
    R = T * k_eff
    y = torch.empty(T, k_eff, M, dtype=x.dtype, device=x.device)
    gu = torch.empty(R, 2 * I, dtype=x.dtype, device=x.device)
    h = torch.empty(R, I, dtype=x.dtype, device=x.device)
    if R == 0:
        return y, gu, h
    lib = _native.lib()
    need = int(lib.situ_moe_workspace_size(R, E, M, I, _dt(x)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    check("situ_moe_grouped_forward_train",
          lib.situ_moe_grouped_forward_train(
              x.data_ptr(), expert_offsets.data_ptr(), token_index.data_ptr(),
              W_gate_up.data_ptr(), W_down.data_ptr(), y.data_ptr(), gu.data_ptr(), h.data_ptr(),
              workspace.data_ptr(), workspace.numel() * workspace.element_size(), T, k_eff, E, M,
              I, *caps(beta, linear_beta), _dt(x), _stream(x.device)))
    return y, gu, h


def moe_backward_workspace_bytes(R: int, E: int, M: int, I: int) -> int:
    return int(_native.lib().situ_moe_backward_workspace_size(R, E, M, I, SITU_BF16))


def situ_moe_grouped_backward(x: torch.Tensor, expert_offsets: torch.Tensor,
                              token_index: torch.Tensor, W_gate_up: torch.Tensor,
                              W_down: torch.Tensor, gu: torch.Tensor, h: torch.Tensor,
                              dy: torch.Tensor, beta: float = 4.0, linear_beta: float = 25.0,
                              workspace: torch.Tensor | None = None):
    """Backward of the grouped experts for dy [T, k_eff, M] (the gradient of the
    per-route outputs): returns (dx [T, M], dW_gate_up [E, 2I, M], dW_down [E, M, I])."""
    k_eff = dy.shape[1] if dy.dim() == 3 else token_index.numel() // max(x.shape[0], 1)
    T, M, E, I = _moe_shapes(x, expert_offsets, token_index, W_gate_up, W_down, k_eff)
    R = T * k_eff
    for n, t in (("gu", gu), ("h", h), ("dy", dy)):
        _cuda_contig(n, t)
    if gu.shape != (R, 2 * I) or h.shape != (R, I) or dy.numel() != R * M:
        raise ValueError("gu, h or dy do not match the routes")
    dx = torch.empty_like(x)
    dwg = torch.empty_like(W_gate_up)
    dwd = torch.empty_like(W_down)
    lib = _native.lib()
    need = int(lib.situ_moe_backward_workspace_size(R, E, M, I, _dt(x)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    check("situ_moe_grouped_backward",
          lib.situ_moe_grouped_backward(
              x.data_ptr(), expert_offsets.data_ptr(), token_index.data_ptr(),
              W_gate_up.data_ptr(), W_down.data_ptr(), gu.data_ptr(), h.data_ptr(),
              dy.data_ptr(), dx.data_ptr(), dwg.data_ptr(), dwd.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(), T, k_eff, E, M, I,
              *caps(beta, linear_beta), _dt(x), _stream(x.device)))
    return dx, dwg, dwd


# ---------------------------------------------------------------------------
# MXFP8 experts
# ---------------------------------------------------------------------------
MX_GATE_UP, MX_DOWN = 0, 1
MX_E4M3, MX_E2M1 = 0, 1  # weight formats: MXFP8, MXFP4


class MxWeights(tuple):
    """Quantized expert weights: (codes, scales, fmt) -- fmt MX_E4M3 (MXFP8, one code
    a byte) or MX_E2M1 (MXFP4, two codes a byte)."""

    def __new__(cls, codes, scales, fmt=MX_E4M3):
        return super().__new__(cls, (codes, scales, fmt))

    codes = property(lambda self: self[0])
    scales = property(lambda self: self[1])
    fmt = property(lambda self: self[2])


def _wfmt(w) -> int:
    return int(w[2]) if len(w) > 2 else MX_E4M3


def mx_act_scales_bytes(R: int, K: int) -> int:
    return int(_native.lib().situ_mx_act_scales_size(R, K))


def mx_weight_scales_bytes(E: int, M: int, I: int, kind: int) -> int:
    return int(_native.lib().situ_mx_weight_scales_size(E, M, I, kind))


def mx_quantize_act(x: torch.Tensor):
    """MXFP8 quantization of bf16 rows x [R, K]: (codes uint8 [R, K], scales uint8 in
    the activation tile layout)."""
    _cuda_contig("x", x)
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bf16")
    K = x.shape[-1]
    R = x.numel() // K
    codes = torch.empty(R, K, dtype=torch.uint8, device=x.device)
    scales = torch.empty(max(mx_act_scales_bytes(R, K), 1), dtype=torch.uint8, device=x.device)
    check("situ_mx_quantize_act",
          _native.lib().situ_mx_quantize_act(x.data_ptr(), codes.data_ptr(), scales.data_ptr(),
                                             R, K, _stream(x.device)))
    return codes, scales


def mx_quantize_weights(W: torch.Tensor, kind: int, fmt: int = MX_E4M3) -> MxWeights:
    """MX quantization of stacked expert weights: kind MX_GATE_UP takes W_gate_up
    [E, 2I, M] (or [2I, M]), MX_DOWN takes W_down [E, M, I] (or [M, I]); fmt MX_E4M3
    (MXFP8) or MX_E2M1 (MXFP4).  Returns MxWeights(codes uint8 of W's shape -- the last
    dimension halved for MXFP4 --, scales uint8 in the weight tile layout, fmt)."""
    _cuda_contig("W", W)
    if W.dtype != torch.bfloat16:
        raise TypeError("W must be bf16")
    w3 = W.view(1, *W.shape) if W.dim() == 2 else W
    E, rows, K = w3.shape
    if kind == MX_GATE_UP:
        M, I = K, rows // 2
    elif kind == MX_DOWN:
        M, I = rows, K
    else:
        raise ValueError("kind must be MX_GATE_UP or MX_DOWN")
    cshape = tuple(W.shape[:-1]) + (K // 2 if fmt == MX_E2M1 else K,)
    codes = torch.empty(cshape, dtype=torch.uint8, device=W.device)
    scales = torch.empty(max(mx_weight_scales_bytes(E, M, I, kind), 1), dtype=torch.uint8,
                         device=W.device)
    check("situ_mx_quantize_weights",
          _native.lib().situ_mx_quantize_weights(W.data_ptr(), codes.data_ptr(),
                                                 scales.data_ptr(), E, M, I, kind, fmt,
                                                 _stream(W.device)))
    return MxWeights(codes, scales, fmt)


def situ_ffn_gate_up_mxfp8(xq, wguq, beta: float = 4.0, linear_beta: float = 25.0):
    """MXFP8 gate_up GEMM + SiTU-GLU: xq = (codes [R, M], scales), wguq = one expert's
    (codes [2I, M], scales) -> h [R, I] bf16."""
    xc, xs = xq[0], xq[1]
    wc, ws = wguq[0], wguq[1]
    for n, t in (("x codes", xc), ("x scales", xs), ("W codes", wc), ("W scales", ws)):
        _cuda_contig(n, t)
    R, M = xc.shape
    I = wc.shape[-2] // 2
    h = torch.empty(R, I, dtype=torch.bfloat16, device=xc.device)
    check("situ_ffn_gate_up_mxfp8",
          _native.lib().situ_ffn_gate_up_mxfp8(xc.data_ptr(), xs.data_ptr(), wc.data_ptr(),
                                               ws.data_ptr(), _wfmt(wguq), h.data_ptr(), R, M, I,
                                               *caps(beta, linear_beta), _stream(xc.device)))
    return h


def ffn_mxfp8_workspace_bytes(R: int, M: int, I: int) -> int:
    return int(_native.lib().situ_ffn_mxfp8_workspace_size(R, M, I))


def situ_ffn_forward_mxfp8(x: torch.Tensor, wguq, wdq, beta: float = 4.0,
                           linear_beta: float = 25.0, y: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Dense SiTU-GLU FFN with MX experts: x [R, M] bf16 (quantized to MXFP8), wguq /
    wdq one expert's quantized weights (MXFP8 or MXFP4, from mx_quantize_weights) ->
    y [R, M] bf16."""
    _cuda_contig("x", x)
    M = x.shape[-1]
    R = x.numel() // M
    I = wguq[0].shape[-2] // 2
    if y is None:
        y = torch.empty_like(x)
    if R == 0:
        return y
    lib = _native.lib()
    need = int(lib.situ_ffn_mxfp8_workspace_size(R, M, I))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    check("situ_ffn_forward_mxfp8",
          lib.situ_ffn_forward_mxfp8(x.data_ptr(), wguq[0].data_ptr(), wguq[1].data_ptr(),
                                     wdq[0].data_ptr(), wdq[1].data_ptr(), _wfmt(wguq),
                                     y.data_ptr(),
                                     workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), R, M, I,
                                     *caps(beta, linear_beta), _stream(x.device)))
    return y


def moe_mxfp8_workspace_bytes(R: int, E: int, M: int, I: int) -> int:
    return int(_native.lib().situ_moe_mxfp8_workspace_size(R, E, M, I))


def situ_moe_grouped_forward_mxfp8(x: torch.Tensor, expert_offsets: torch.Tensor,
                                   token_index: torch.Tensor, wguq, wdq, k_eff: int,
                                   beta: float = 4.0, linear_beta: float = 25.0,
                                   y: torch.Tensor | None = None,
                                   workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Grouped SiTU-GLU experts with MXFP8 weights (stacked, from
    mx_quantize_weights): y[t, s] = FFN_{expert of (t, s)}(x[t]), [T, k_eff, M] bf16."""
    for n, t in (("x", x), ("expert_offsets", expert_offsets), ("token_index", token_index)):
        _cuda_contig(n, t)
    T, M = x.shape
    E, twoI, _ = wguq[0].shape
    I = twoI // 2
    if wguq[0].shape[-1] * (2 if _wfmt(wguq) == MX_E2M1 else 1) != M:
        raise ValueError("gate_up codes do not match x")
    if y is None:
        y = torch.empty(T, k_eff, M, dtype=x.dtype, device=x.device)
    R = T * k_eff
    if R == 0:
        return y
    lib = _native.lib()
    need = int(lib.situ_moe_mxfp8_workspace_size(R, E, M, I))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    check("situ_moe_grouped_forward_mxfp8",
          lib.situ_moe_grouped_forward_mxfp8(
              x.data_ptr(), expert_offsets.data_ptr(), token_index.data_ptr(),
              wguq[0].data_ptr(), wguq[1].data_ptr(), wdq[0].data_ptr(), wdq[1].data_ptr(),
              _wfmt(wguq), y.data_ptr(), workspace.data_ptr(),
              workspace.numel() * workspace.element_size(),
              T, k_eff, E, M, I, *caps(beta, linear_beta), _stream(x.device)))
    return y


def situ_moe_grouped_forward_combined(x: torch.Tensor, expert_offsets: torch.Tensor,
                                      token_index: torch.Tensor, W_gate_up: torch.Tensor,
                                      W_down: torch.Tensor, weights: torch.Tensor,
                                      beta: float = 4.0, linear_beta: float = 25.0,
                                      out: torch.Tensor | None = None,
                                      workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Routed layer output with the combine fused into the down projection (FP32
    scatter-add): out[t] = sum_s weights[t, s] * FFN_{expert of (t, s)}(x[t]), [T, M].
    Not bitwise reproducible (atomic order); situ_moe_combine is the deterministic path."""
    T, M, E, I = _moe_shapes(x, expert_offsets, token_index, W_gate_up, W_down,
                             weights.shape[1] if weights.dim() == 2 else 1)
    _cuda_contig("weights", weights)
    k_eff = weights.shape[1]
    if weights.dtype != torch.float32 or weights.shape != (T, k_eff):
        raise ValueError("weights must be float32 [T, k_eff]")
    if out is None:
        out = torch.empty(T, M, dtype=x.dtype, device=x.device)
    if T == 0:
        return out
    lib = _native.lib()
    need = int(lib.situ_moe_combined_workspace_size(T, k_eff, E, M, I, _dt(x)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    check("situ_moe_grouped_forward_combined",
          lib.situ_moe_grouped_forward_combined(
              x.data_ptr(), expert_offsets.data_ptr(), token_index.data_ptr(),
              W_gate_up.data_ptr(), W_down.data_ptr(), weights.data_ptr(), out.data_ptr(),
              workspace.data_ptr(), workspace.numel() * workspace.element_size(), T, k_eff, E, M,
              I, *caps(beta, linear_beta), _dt(x), _stream(x.device)))
    return out


def moe_combined_workspace_bytes(T: int, k_eff: int, E: int, M: int, I: int) -> int:
    return int(_native.lib().situ_moe_combined_workspace_size(T, k_eff, E, M, I, SITU_BF16))


def situ_moe_combine(y: torch.Tensor, weights: torch.Tensor,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """Layer output of a routed batch: out[t] = sum_s weights[t, s] * y[t, s] (FP32,
    slot order).  y [T, k_eff, M]; weights [T, k_eff] float32 -> out [T, M]."""
    _cuda_contig("y", y)
    _cuda_contig("weights", weights)
    T, k_eff, M = y.shape
    if weights.shape != (T, k_eff) or weights.dtype != torch.float32:
        raise ValueError("weights must be float32 [T, k_eff]")
    if out is None:
        out = torch.empty(T, M, dtype=y.dtype, device=y.device)
    if T == 0:
        return out
    check("situ_moe_combine",
          _native.lib().situ_moe_combine(y.data_ptr(), weights.data_ptr(), out.data_ptr(), T,
                                         k_eff, M, _dt(y), _stream(y.device)))
    return out


FFN_PATH_FUSED, FFN_PATH_TWO_LAUNCHES = 1, 2


def ffn_last_path() -> int:
    """The path of this thread's last bf16 situ_ffn_forward: FFN_PATH_FUSED (one
    persistent launch), FFN_PATH_TWO_LAUNCHES, or 0 before the first call."""
    return int(_native.lib().situ_ffn_last_path())


def ffn_set_single_launch(enable: bool) -> bool:
    """Turn the one-launch bf16 dense forward on or off for the process (on by
    default; off runs the two launches, e.g. under a kernel profiler that cannot
    replay a cooperative cluster launch).  Returns the previous setting."""
    return bool(_native.lib().situ_ffn_set_single_launch(1 if enable else 0))


def moe_set_kgrouped_two_cta(enable: bool) -> bool:
    """Two-CTA form (per-expert tensor maps) of the grouped backward's weight gradients on
    or off for the process (on by default; off: one CTA per tile, the form used where
    two-CTA clusters cannot launch; same bits).  Returns the previous setting."""
    return bool(_native.lib().situ_moe_set_kgrouped_two_cta(1 if enable else 0))


def device_status(clear: bool = True) -> int:
    """First device-side failure recorded since the last clear (0 = SITU_OK)."""
    return int(_native.lib().situ_device_status(1 if clear else 0))


def set_wait_limit_ns(ns: int) -> int:
    """Bound (ns of wall time) of every pipeline wait in the GEMM kernels launched from
    now on; 0 restores the default of 10 s.  Returns the previous bound."""
    return int(_native.lib().situ_set_wait_limit_ns(int(ns)))


def selftest_group_maps(k_offsets, rows: int, cols: int) -> int:
    """Per-group tensor maps written on the device against the driver's encoding:
    returns [groups, 2] int32 flags, 1 where group g's A or B map differs (see
    situ_selftest_group_maps)."""
    off = np.ascontiguousarray(np.asarray(k_offsets, dtype=np.int32))
    out = np.zeros(2 * (len(off) - 1), dtype=np.int32)
    check("situ_selftest_group_maps",
          _native.lib().situ_selftest_group_maps(off.ctypes.data, len(off) - 1, int(rows),
                                                 int(cols), out.ctypes.data,
                                                 _stream(torch.device("cuda"))))
    return out.reshape(-1, 2)


def selftest_bounded_wait(limit_us: int = 2000) -> None:
    """Launch the bounded-wait self test on the current stream."""
    check("situ_selftest_bounded_wait",
          _native.lib().situ_selftest_bounded_wait(int(limit_us),
                                                   _stream(torch.device("cuda"))))


__all__ = [
    "SituError", "situ_glu_act", "situ_ffn_forward", "situ_ffn_forward_host", "situ_ffn_gate_up",
    "situ_ffn_down",
    "situ_moe_build_index",
    "situ_moe_grouped_forward", "ffn_workspace_bytes", "moe_workspace_bytes",
    "device_status", "selftest_bounded_wait", "selftest_group_maps", "set_wait_limit_ns", "ffn_host_workspace_bytes", "situ_moe_combine",
    "ffn_last_path", "FFN_PATH_FUSED", "FFN_PATH_TWO_LAUNCHES", "ffn_set_single_launch",
    "moe_set_kgrouped_two_cta",
    "situ_ffn_forward_train", "situ_ffn_backward", "ffn_backward_workspace_bytes",
    "situ_moe_grouped_forward_train", "situ_moe_grouped_backward", "moe_backward_workspace_bytes",
    "situ_moe_grouped_forward_combined", "moe_combined_workspace_bytes",
    "MX_GATE_UP", "MX_DOWN", "MX_E4M3", "MX_E2M1", "MxWeights", "mx_act_scales_bytes", "mx_weight_scales_bytes", "mx_quantize_act",
    "mx_quantize_weights", "situ_ffn_gate_up_mxfp8", "situ_ffn_forward_mxfp8",
    "ffn_mxfp8_workspace_bytes", "situ_moe_grouped_forward_mxfp8", "moe_mxfp8_workspace_bytes",
]
