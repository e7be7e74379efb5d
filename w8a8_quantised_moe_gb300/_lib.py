"""ctypes binding of ``libmoe_w8a8.so`` (declarations in include/moe_w8a8.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
There is no fallback; if the library is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_w8a8.so")

STATUS = {
    0: "MOE_OK",
    -1: "MOE_ERR_INVALID_ARG",
    -2: "MOE_ERR_UNSUPPORTED_SHAPE",
    -3: "MOE_ERR_WORKSPACE_TOO_SMALL",
    -4: "MOE_ERR_CUDA",
    -5: "MOE_ERR_DEVICE_TIMEOUT",
    -6: "MOE_ERR_NOT_IMPLEMENTED",
    -7: "MOE_ERR_DEVICE",
}

# every symbol include/moe_w8a8.h declares
EXPORTS = (
    "moe_w8a8_status_string",
    "moe_w8a8_version",
    "moe_w8a8_quantize_weights",
    "moe_w8a8_workspace_size",
    "moe_w8a8_forward",
    "moe_w8a8_forward_debug",
    "moe_w8a8_linear_workspace_size",
    "moe_w8a8_linear",
    "moe_w8a8_device_error",
    "moe_w8a8_set_wait_timeout_ns",
    "moe_w8a8_set_gemm_path",
    "moe_w8a8_set_profile_events",
    "moe_w8a8_launch_count",
    "moe_w8a8_linear_static",
    "moe_w8a8_linear_static_error",
    "moe_w8a8_fp8_quantize_weights",
    "moe_w8a8_fp8_forward",
    "moe_w8a8_fp8_forward_debug",
    "moe_w8a8_forward_host",
    "moe_w8a8_fp8_forward_host",
    "moe_w8a8_host_chunks",
    "moe_w8a8_quantize_weights_smoothed",
    "moe_w8a8_forward_smooth",
    "moe_w8a8_forward_fused",
    "moe_w8a8_fused_supported",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class DebugBuffers(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "topk_ids", "topk_w", "offsets", "slot_of", "slot_token", "s_x", "q_x", "acc1", "h",
        "s_h", "q_h", "acc2", "o", "s_slot", "q_slot")]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = open_library(path)
        return _lib


def open_library(path: str):
    """A separately loaded copy of a build of the library (e.g. the checked
    build), its C signatures declared; load() is not affected."""
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    _declare(lib)
    return lib


def _declare(lib) -> None:
    i64, vp, sz, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    decl = {
        "moe_w8a8_status_string": ([i32], ctypes.c_char_p),
        "moe_w8a8_version": ([], i32),
        "moe_w8a8_quantize_weights": ([vp, i64, i64, vp, vp, vp], i32),
        "moe_w8a8_workspace_size": ([i64, i64, i64, i64, i64], sz),
        "moe_w8a8_forward": ([vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, sz, vp], i32),
        "moe_w8a8_forward_debug": ([vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, sz, vp,
                                    ctypes.POINTER(DebugBuffers)], i32),
        "moe_w8a8_linear_workspace_size": ([i64, i64, i64], sz),
        "moe_w8a8_linear": ([vp, vp, vp, i64, i64, i64, vp, vp, sz, vp], i32),
        "moe_w8a8_device_error": ([vp, vp], i32),
        "moe_w8a8_set_wait_timeout_ns": ([ctypes.c_uint64], ctypes.c_uint64),
        "moe_w8a8_set_gemm_path": ([i32], i32),
        "moe_w8a8_set_profile_events": ([ctypes.c_void_p, i32], i32),
        "moe_w8a8_launch_count": ([], ctypes.c_uint64),
        "moe_w8a8_linear_static": ([vp, vp, vp, i64, i64, i64, vp, vp], i32),
        "moe_w8a8_linear_static_error": ([vp], i32),
        "moe_w8a8_fp8_quantize_weights": ([vp, i64, i64, vp, vp, vp], i32),
        "moe_w8a8_fp8_forward": ([vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, sz, vp], i32),
        "moe_w8a8_fp8_forward_debug": ([vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, sz, vp,
                                        ctypes.POINTER(DebugBuffers)], i32),
        "moe_w8a8_forward_host": ([vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, sz, vp,
                                   vp, i32], i32),
        "moe_w8a8_fp8_forward_host": ([vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, sz,
                                       vp, vp, i32], i32),
        "moe_w8a8_host_chunks": ([i64, i64, i64, i64], i32),
        "moe_w8a8_quantize_weights_smoothed": ([vp, i64, i64, vp, vp, vp, vp], i32),
        "moe_w8a8_forward_smooth": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, sz, vp,
                                     ctypes.POINTER(DebugBuffers)], i32),
        "moe_w8a8_forward_fused": ([vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, sz, vp,
                                    ctypes.POINTER(DebugBuffers)], i32),
        "moe_w8a8_fused_supported": ([i64, i64, i64, i64, i64], i32),
    }
    for name, (args, res) in decl.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res


def check(status: int, what: str) -> None:
    if status != 0:
        raise MoeError(status, what)
