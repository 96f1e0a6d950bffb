"""FP64 CPU oracle for the SiTU-GLU expert feed-forward -- TEST INFRASTRUCTURE.

Only the test suite, the package's smoke check and the benchmark's CPU-baseline
leg (and its ``--impl reference`` arm) may import this module.  The GPU library
neither imports nor links it, and the two share no code: the arithmetic lives in
``situ_oracle.c`` (plain C, IEEE double), this file only compiles it with gcc and
marshals numpy arrays through ctypes.

What each C function follows is cited in ``situ_oracle.c``; the CPU test suite
pins every one of them against values printed on the SiTU-GLU pages and against
closed forms.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "situ_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsitu_oracle.so")

# The oracle's own input-type codes (see the enum in situ_oracle.c).
F64, BF16, F32 = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle into a shared object with gcc and return its path.

    ``-ffp-contract=off`` keeps every multiply and add separately rounded on
    both x86-64 and aarch64, so the oracle gives the same bits on either host.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    d, i64, i32, vp, dp = (ctypes.c_double, ctypes.c_int64, ctypes.c_int32,
                           ctypes.c_void_p, ctypes.c_void_p)
    ci = ctypes.c_int
    for name, args, res in [
        ("oracle_softcap", [d, d], d),
        ("oracle_sigmoid", [d], d),
        ("oracle_gate_branch", [d, d], d),
        ("oracle_up_branch", [d, d], d),
        ("oracle_situ_pair", [d, d, d, d], d),
        ("oracle_situ_glu_act", [vp, ci, dp, i64, i64, d, d], ci),
        ("oracle_ffn_forward", [vp, ci, vp, vp, ci, dp, dp, i64, i64, i64, d, d], ci),
        ("oracle_moe_build_index", [vp, i64, i32, vp, vp], ci),
        ("oracle_moe_grouped_forward",
         [vp, ci, vp, vp, vp, ci, dp, i64, i32, i32, i64, i64, d, d], ci),
        ("oracle_moe_combine", [dp, vp, ci, dp, i64, i32, i64], ci),
        ("oracle_situ_pair_grad", [d, d, d, d, dp, dp], None),
        ("oracle_moe_grouped_backward", [vp, ci, vp, vp, vp, ci, vp, ci, dp, dp, dp, i64, i32,
                                         i32, i64, i64, d, d], ci),
        ("oracle_ffn_backward", [vp, ci, vp, vp, ci, vp, ci, dp, dp, dp, dp, i64, i64, i64, d, d],
         ci),
        ("oracle_num_threads", [], ci),
        ("oracle_e4m3_decode", [ctypes.c_uint32], d),
        ("oracle_e4m3_encode", [d], ctypes.c_uint32),
        ("oracle_e8m0_decode", [ctypes.c_uint32], d),
        ("oracle_mx_scale_code", [d], ctypes.c_uint32),
        ("oracle_mx_quantize", [vp, ci, i64, i64, vp, vp], ci),
        ("oracle_mx_dequantize", [vp, vp, i64, i64, dp], ci),
        ("oracle_e4m3_encode_array", [dp, i64, vp], ci),
        ("oracle_e4m3_decode_array", [vp, i64, dp], ci),
        ("oracle_round_bf16_array", [dp, i64, vp], ci),
        ("oracle_e2m1_decode", [ctypes.c_uint32], d),
        ("oracle_e2m1_encode", [d], ctypes.c_uint32),
        ("oracle_e2m1_encode_array", [dp, i64, vp], ci),
        ("oracle_mxfp4_quantize", [vp, ci, i64, i64, vp, vp], ci),
        ("oracle_mxfp4_dequantize", [vp, vp, i64, i64, dp], ci),
    ]:
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared object.

    With ``path`` given, load that build (used by the tests that compile
    deliberately broken copies of the oracle); otherwise the cached default.
    """
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _as_input(a: np.ndarray):
    """Return (contiguous array, oracle dtype code) for a float64, float32 or
    bfloat16-bit-pattern (uint16) array."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"oracle input must be float64, float32 or uint16 (bf16 bits), got {a.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(status: int, what: str):
    if status != 0:
        raise ValueError(f"{what}: oracle status {status}")


class Oracle:
    """numpy front end to the C oracle.  All outputs are float64."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    # -- scalars --------------------------------------------------------------
    def softcap(self, x, beta):
        return self.lib.oracle_softcap(float(x), float(beta))

    def sigmoid(self, g):
        return self.lib.oracle_sigmoid(float(g))

    def gate(self, g, beta=4.0):
        return self.lib.oracle_gate_branch(float(g), float(beta))

    def up(self, u, linear_beta=25.0):
        return self.lib.oracle_up_branch(float(u), float(linear_beta))

    def pair(self, g, u, beta=4.0, linear_beta=25.0):
        return self.lib.oracle_situ_pair(float(g), float(u), float(beta), float(linear_beta))

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    # -- tensors --------------------------------------------------------------
    def situ_glu_act(self, gate_up: np.ndarray, beta=4.0, linear_beta=25.0) -> np.ndarray:
        """gate_up [..., 2I] -> [..., I] in float64."""
        g, dt = _as_input(gate_up)
        if g.shape[-1] % 2:
            raise ValueError("last dimension must be even (gate half, up half)")
        I = g.shape[-1] // 2
        rows = int(np.prod(g.shape[:-1], dtype=np.int64))
        out = np.empty(g.shape[:-1] + (I,), dtype=np.float64)
        _check(self.lib.oracle_situ_glu_act(_ptr(g), dt, _ptr(out), rows, I,
                                            float(beta), float(linear_beta)), "situ_glu_act")
        return out

    def ffn_forward(self, x: np.ndarray, w_gate_up: np.ndarray, w_down: np.ndarray,
                    beta=4.0, linear_beta=25.0, want_h=False):
        """x [..., M], w_gate_up [2I, M], w_down [M, I] -> y [..., M] (and h)."""
        xa, xdt = _as_input(x)
        wg, wdt = _as_input(w_gate_up)
        wd, wdt2 = _as_input(w_down)
        if wdt != wdt2:
            raise TypeError("w_gate_up and w_down must share a dtype")
        M = xa.shape[-1]
        I = wg.shape[0] // 2
        if wg.shape != (2 * I, M) or wd.shape != (M, I):
            raise ValueError(f"bad weight shapes {wg.shape}, {wd.shape} for M={M}")
        R = int(np.prod(xa.shape[:-1], dtype=np.int64))
        y = np.empty(xa.shape[:-1] + (M,), dtype=np.float64)
        h = np.empty(xa.shape[:-1] + (I,), dtype=np.float64) if want_h else None
        _check(self.lib.oracle_ffn_forward(_ptr(xa), xdt, _ptr(wg), _ptr(wd), wdt,
                                           _ptr(h) if want_h else None, _ptr(y),
                                           R, M, I, float(beta), float(linear_beta)),
               "ffn_forward")
        return (y, h) if want_h else y

    def moe_build_index(self, expert_ids: np.ndarray, E: int):
        """Flat routes [T*k_eff] (int32) -> (offsets [E+1], token_index [T*k_eff])."""
        ids = np.ascontiguousarray(expert_ids, dtype=np.int32).reshape(-1)
        offsets = np.empty(E + 1, dtype=np.int32)
        token_index = np.empty(ids.size, dtype=np.int32)
        _check(self.lib.oracle_moe_build_index(_ptr(ids), ids.size, E, _ptr(offsets),
                                               _ptr(token_index)), "moe_build_index")
        return offsets, token_index

    def pair_grad(self, g, u, beta=4.0, linear_beta=25.0):
        """(dh/dg, dh/du) of one SiTU-GLU coordinate."""
        dg, du = ctypes.c_double(), ctypes.c_double()
        self.lib.oracle_situ_pair_grad(float(g), float(u), float(beta), float(linear_beta),
                                       ctypes.byref(dg), ctypes.byref(du))
        return dg.value, du.value

    def ffn_backward(self, x, w_gate_up, w_down, dy, beta=4.0, linear_beta=25.0,
                     want_dgu=False):
        """Gradients of the dense FFN for upstream dy [R, M]:
        (dx [R, M], dW_gate_up [2I, M], dW_down [M, I]) and optionally dgu [R, 2I]."""
        xa, xdt = _as_input(x)
        wg, wdt = _as_input(w_gate_up)
        wd, wdt2 = _as_input(w_down)
        dya, dydt = _as_input(dy)
        if wdt != wdt2:
            raise TypeError("w_gate_up and w_down must share a dtype")
        M = xa.shape[-1]
        I = wg.shape[0] // 2
        R = int(np.prod(xa.shape[:-1], dtype=np.int64))
        if wg.shape != (2 * I, M) or wd.shape != (M, I) or dya.size != R * M:
            raise ValueError("bad shapes")
        dx = np.empty((R, M))
        dwg = np.empty((2 * I, M))
        dwd = np.empty((M, I))
        dgu = np.empty((R, 2 * I)) if want_dgu else None
        _check(self.lib.oracle_ffn_backward(_ptr(xa), xdt, _ptr(wg), _ptr(wd), wdt, _ptr(dya),
                                            dydt, _ptr(dx), _ptr(dwg), _ptr(dwd),
                                            _ptr(dgu) if want_dgu else None, R, M, I,
                                            float(beta), float(linear_beta)), "ffn_backward")
        out = (dx.reshape(xa.shape), dwg, dwd)
        return out + (dgu,) if want_dgu else out

    def moe_grouped_backward(self, x, expert_ids, w_gate_up, w_down, dy, beta=4.0,
                             linear_beta=25.0):
        """Gradients of the grouped experts for dy [T, k_eff, M]:
        (dx [T, M], dW_gate_up [E, 2I, M], dW_down [E, M, I])."""
        xa, xdt = _as_input(x)
        ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
        wg, wdt = _as_input(w_gate_up)
        wd, _ = _as_input(w_down)
        dya, dydt = _as_input(dy)
        T, M = xa.shape
        k_eff = ids.shape[1]
        E, twoI, _ = wg.shape
        I = twoI // 2
        dx = np.empty((T, M))
        dwg = np.empty((E, 2 * I, M))
        dwd = np.empty((E, M, I))
        _check(self.lib.oracle_moe_grouped_backward(_ptr(xa), xdt, _ptr(ids), _ptr(wg), _ptr(wd),
                                                    wdt, _ptr(dya), dydt, _ptr(dx), _ptr(dwg),
                                                    _ptr(dwd), T, k_eff, E, M, I, float(beta),
                                                    float(linear_beta)), "moe_grouped_backward")
        return dx, dwg, dwd

    # ----- MXFP8 (OCP MX v1.0: E4M3 elements, E8M0 scales per 32) -----------
    def e4m3_decode(self, codes) -> np.ndarray:
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape)
        _check(self.lib.oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out)), "e4m3_decode")
        return out

    def e4m3_encode(self, v) -> np.ndarray:
        a = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint8)
        _check(self.lib.oracle_e4m3_encode_array(_ptr(a), a.size, _ptr(out)), "e4m3_encode")
        return out

    def e8m0_decode(self, c) -> float:
        return self.lib.oracle_e8m0_decode(int(c))

    def mx_scale_code(self, amax) -> int:
        return int(self.lib.oracle_mx_scale_code(float(amax)))

    def round_bf16(self, v) -> np.ndarray:
        """Round doubles to bfloat16 (RNE); returns the bit patterns (uint16)."""
        a = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        _check(self.lib.oracle_round_bf16_array(_ptr(a), a.size, _ptr(out)), "round_bf16")
        return out

    def mx_quantize(self, a):
        """MX quantization of a [R, K] tensor: (codes uint8 [R, K], scales uint8
        [R, K/32])."""
        src, dt = _as_input(a)
        R, K = src.shape
        codes = np.empty((R, K), dtype=np.uint8)
        scales = np.empty((R, K // 32), dtype=np.uint8)
        _check(self.lib.oracle_mx_quantize(_ptr(src), dt, R, K, _ptr(codes), _ptr(scales)),
               "mx_quantize")
        return codes, scales

    def mx_dequantize(self, codes, scales) -> np.ndarray:
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        sc = np.ascontiguousarray(scales, dtype=np.uint8)
        R, K = c.shape
        out = np.empty((R, K))
        _check(self.lib.oracle_mx_dequantize(_ptr(c), _ptr(sc), R, K, _ptr(out)), "mx_dequantize")
        return out

    def e2m1_decode(self, c) -> float:
        return self.lib.oracle_e2m1_decode(int(c))

    def e2m1_encode(self, v) -> np.ndarray:
        a = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint8)
        _check(self.lib.oracle_e2m1_encode_array(_ptr(a), a.size, _ptr(out)), "e2m1_encode")
        return out

    def mxfp4_quantize(self, a):
        """MXFP4 quantization of a [R, K] tensor: (codes uint8 [R, K/2], two E2M1 per
        byte with the even element in the low nibble; scales uint8 [R, K/32])."""
        src, dt = _as_input(a)
        R, K = src.shape
        codes = np.empty((R, K // 2), dtype=np.uint8)
        scales = np.empty((R, K // 32), dtype=np.uint8)
        _check(self.lib.oracle_mxfp4_quantize(_ptr(src), dt, R, K, _ptr(codes), _ptr(scales)),
               "mxfp4_quantize")
        return codes, scales

    def mxfp4_dequantize(self, codes, scales) -> np.ndarray:
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        sc = np.ascontiguousarray(scales, dtype=np.uint8)
        R, K = c.shape[0], c.shape[1] * 2
        out = np.empty((R, K))
        _check(self.lib.oracle_mxfp4_dequantize(_ptr(c), _ptr(sc), R, K, _ptr(out)),
               "mxfp4_dequantize")
        return out

    def mx_ffn_forward(self, xq, wguq, wdq, beta=4.0, linear_beta=25.0, weights_fp4=False):
        """The SiTU-GLU FFN with MXFP8 operands (weights MXFP4 with weights_fp4): each
        argument is a (codes, scales) pair.  gu and h in FP64 on the decoded x and W_gate_up; h cast to bf16 (the
        pages' cast back to the input dtype), MX-quantized as the down projection's
        input, and y = dequant(h) dequant(W_down)^T in FP64.  Returns
        (y [R, M], h_bf16 bits [R, I], (h codes, h scales))."""
        x = self.mx_dequantize(*xq)
        wdeq = self.mxfp4_dequantize if weights_fp4 else self.mx_dequantize
        wgu = wdeq(*wguq)
        wd = wdeq(*wdq)
        _, h = self.ffn_forward(x, wgu, wd, beta, linear_beta, want_h=True)
        hb = self.round_bf16(h)
        hq = self.mx_quantize(hb)
        y = self.mx_dequantize(*hq) @ wd.T  # library matmul of the decoded values
        return y, hb, hq

    def moe_combine(self, y: np.ndarray, w: np.ndarray) -> np.ndarray:
        """y [T, k_eff, M] (float64), w [T, k_eff] -> out [T, M] = sum_s w[t,s] y[t,s]."""
        ya = np.ascontiguousarray(y, dtype=np.float64)
        wa, wdt = _as_input(w)
        T, k_eff, M = ya.shape
        if wa.shape != (T, k_eff):
            raise ValueError("weights must be [T, k_eff]")
        out = np.empty((T, M), dtype=np.float64)
        _check(self.lib.oracle_moe_combine(_ptr(ya), _ptr(wa), wdt, _ptr(out), T, k_eff, M),
               "moe_combine")
        return out

    def moe_grouped_forward(self, x: np.ndarray, expert_ids: np.ndarray,
                            w_gate_up: np.ndarray, w_down: np.ndarray,
                            beta=4.0, linear_beta=25.0) -> np.ndarray:
        """x [T, M], expert_ids [T, k_eff], w_gate_up [E, 2I, M], w_down [E, M, I]
        -> y [T, k_eff, M] (one FFN output per (token, slot))."""
        xa, xdt = _as_input(x)
        ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
        wg, wdt = _as_input(w_gate_up)
        wd, wdt2 = _as_input(w_down)
        if wdt != wdt2:
            raise TypeError("w_gate_up and w_down must share a dtype")
        T, M = xa.shape
        k_eff = ids.shape[1]
        E, twoI, _ = wg.shape
        I = twoI // 2
        if wd.shape != (E, M, I) or wg.shape != (E, 2 * I, M):
            raise ValueError("bad stacked weight shapes")
        y = np.zeros((T, k_eff, M), dtype=np.float64)
        _check(self.lib.oracle_moe_grouped_forward(_ptr(xa), xdt, _ptr(ids), _ptr(wg), _ptr(wd),
                                                   wdt, _ptr(y), T, k_eff, E, M, I,
                                                   float(beta), float(linear_beta)),
               "moe_grouped_forward")
        return y
