"""ctypes loader for libsitu.so (the C ABI declared in include/situ.h).

There is no fallback: if the library is missing or fails to load, every call
raises.  Build it with ``__graft_entry__.build()`` or
``python -m situ_glu_activation_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

# Mirrors of the C enums in include/situ.h.
SITU_BF16, SITU_F32 = 0, 1
STATUS_NAMES = {
    0: "SITU_OK", 1: "SITU_ERR_ARG", 2: "SITU_ERR_ALIGN", 3: "SITU_ERR_ALIAS",
    4: "SITU_ERR_CUDA", 5: "SITU_ERR_TIMEOUT", 6: "SITU_ERR_UNSUPPORTED",
    7: "SITU_ERR_INDEX", 8: "SITU_ERR_WORKSPACE",
}

# Every symbol the header declares, with (argtypes, restype).
_vp, _i64, _i32, _u32, _f32, _ci, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                          ctypes.c_uint32, ctypes.c_float, ctypes.c_int,
                                          ctypes.c_size_t)
_u64 = ctypes.c_uint64
SIGNATURES = {
    "situ_abi_version": ([], _ci),
    "situ_status_string": ([_ci], ctypes.c_char_p),
    "situ_last_cuda_error": ([], ctypes.c_char_p),
    "situ_ffn_last_path": ([], _ci),
    "situ_ffn_set_single_launch": ([_ci], _ci),
    "situ_moe_set_kgrouped_two_cta": ([_ci], _ci),
    "situ_device_status": ([_ci], _ci),
    "situ_glu_act": ([_vp, _vp, _i64, _i64, _f32, _f32, _ci, _vp], _ci),
    "situ_ffn_workspace_size": ([_i64, _i64, _i64, _ci], _sz),
    "situ_ffn_forward": ([_vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _i64, _f32, _f32, _ci, _vp],
                         _ci),
    "situ_ffn_gate_up": ([_vp, _vp, _vp, _i64, _i64, _i64, _f32, _f32, _ci, _vp], _ci),
    "situ_ffn_down": ([_vp, _vp, _vp, _i64, _i64, _i64, _ci, _vp], _ci),
    "situ_ffn_forward_train": ([_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _f32, _f32, _ci,
                                _vp], _ci),
    "situ_ffn_backward_workspace_size": ([_i64, _i64, _i64, _ci], _sz),
    "situ_ffn_backward": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64,
                           _i64, _f32, _f32, _ci, _vp], _ci),
    "situ_ffn_host_workspace_size": ([_i64, _i64, _i64, _ci, _i64], _sz),
    "situ_ffn_forward_host": ([_vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _i64, _i64, _f32, _f32,
                               _ci, _vp], _ci),
    "situ_ffn_forward_noalloc": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _f32, _f32, _ci, _vp],
                                 _ci),
    "situ_moe_index_workspace_size": ([_i64, _i32], _sz),
    "situ_moe_build_index": ([_vp, _vp, _vp, _vp, _sz, _i64, _i32, _vp], _ci),
    "situ_moe_workspace_size": ([_i64, _i32, _i64, _i64, _ci], _sz),
    "situ_moe_grouped_forward": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i32, _i32,
                                  _i64, _i64, _f32, _f32, _ci, _vp], _ci),
    "situ_moe_grouped_forward_train": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64,
                                        _i32, _i32, _i64, _i64, _f32, _f32, _ci, _vp], _ci),
    "situ_moe_backward_workspace_size": ([_i64, _i32, _i64, _i64, _ci], _sz),
    "situ_moe_grouped_backward": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                   _sz, _i64, _i32, _i32, _i64, _i64, _f32, _f32, _ci, _vp], _ci),
    "situ_moe_combine": ([_vp, _vp, _vp, _i64, _i32, _i64, _ci, _vp], _ci),
    "situ_moe_combined_workspace_size": ([_i64, _i32, _i32, _i64, _i64, _ci], _sz),
    "situ_moe_grouped_forward_combined": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64,
                                           _i32, _i32, _i64, _i64, _f32, _f32, _ci, _vp], _ci),
    "situ_mx_act_scales_size": ([_i64, _i64], _sz),
    "situ_mx_weight_scales_size": ([_i32, _i64, _i64, _ci], _sz),
    "situ_mx_quantize_act": ([_vp, _vp, _vp, _i64, _i64, _vp], _ci),
    "situ_mx_quantize_weights": ([_vp, _vp, _vp, _i32, _i64, _i64, _ci, _ci, _vp], _ci),
    "situ_ffn_gate_up_mxfp8": ([_vp, _vp, _vp, _vp, _ci, _vp, _i64, _i64, _i64, _f32, _f32, _vp],
                               _ci),
    "situ_ffn_mxfp8_workspace_size": ([_i64, _i64, _i64], _sz),
    "situ_ffn_forward_mxfp8": ([_vp, _vp, _vp, _vp, _vp, _ci, _vp, _vp, _sz, _i64, _i64, _i64,
                                _f32, _f32, _vp], _ci),
    "situ_moe_mxfp8_workspace_size": ([_i64, _i32, _i64, _i64], _sz),
    "situ_moe_grouped_forward_mxfp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _vp, _vp, _sz,
                                        _i64, _i32, _i32, _i64, _i64, _f32, _f32, _vp], _ci),
    "situ_selftest_bounded_wait": ([_u32, _vp], _ci),
    "situ_selftest_group_maps": ([_vp, _i32, _i64, _i64, _vp, _vp], _ci),
    "situ_set_wait_limit_ns": ([_u64], _u64),
}

_lock = threading.Lock()
_lib = None


class SituError(RuntimeError):
    """A libsitu call returned a status other than SITU_OK."""

    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, f"status {status}")
        super().__init__(f"{fn}: {name}" + (f" ({detail})" if detail else ""))


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load libsitu.so (once) and declare its prototypes."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"libsitu.so not found at {p}: build it first "
                    "(python -m situ_glu_activation_gb300.build)")
            handle = ctypes.CDLL(p)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            if path is not None:
                return handle
            _lib = handle
    return _lib


def check(fn: str, status: int) -> None:
    if status != 0:
        detail = ""
        if status == 4:  # SITU_ERR_CUDA
            detail = (lib().situ_last_cuda_error() or b"").decode()
        raise SituError(fn, status, detail)
