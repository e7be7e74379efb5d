"""ctypes front end of the C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the tests, the smoke check and
the benchmark's CPU-baseline leg import this module.  It marshals numpy
arrays into the C functions and does no arithmetic of the method itself;
every formula lives in ``oracle.c`` with its citation.

bf16 arrays travel as ``numpy.uint16`` bit patterns (numpy has no bf16).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# The flags matter: no FMA contraction (aarch64 gcc contracts by default) and
# no fast-math, so every binary32 multiply and add rounds on its own.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-fopenmp"]


def compile_source(src: str, out: str) -> str:
    """Compile one oracle source file into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``oracle/_build/liboracle.so`` (gcc)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class _Dump(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in (
        "topk_ids", "topk_w", "offsets", "slot_of", "slot_token", "s_x", "q_x", "acc1",
        "h", "s_h", "q_h", "acc2", "o")]


def open_library(path: str):
    """Load an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    sig = {
        "oracle_quantize_rows": [vp, i64, i64, vp, vp],
        "oracle_quantize_rows_bf16": [vp, i64, i64, vp, vp],
        "oracle_router": [vp, vp, vp, i64, i64, i64, i64, vp, vp, vp],
        "oracle_permute": [vp, i64, i64, i64, vp, vp, vp, vp],
        "oracle_gemm_s8": [vp, vp, i64, i64, i64, vp],
        "oracle_epilogue_gate_up": [vp, vp, vp, i64, i64, vp],
        "oracle_epilogue_scale": [vp, vp, vp, i64, i64, vp],
        "oracle_combine": [vp, vp, vp, i64, i64, i64, vp],
        "oracle_moe_forward": [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp,
                               ctypes.POINTER(_Dump)],
        "oracle_moe_forward_dense": [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp],
        "oracle_linear": [vp, vp, vp, i64, i64, i64, vp, vp, vp, vp],
        "oracle_bf16_to_f32": [vp, i64, vp],
        "oracle_f32_to_bf16": [vp, i64, vp],
        "oracle_e4m3_encode": [vp, i64, vp],
        "oracle_e4m3_decode": [vp, i64, vp],
        "oracle_quantize_rows_fp8": [vp, i64, i64, vp, vp],
        "oracle_quantize_rows_bf16_fp8": [vp, i64, i64, vp, vp],
        "oracle_gemm_fp8": [vp, vp, i64, i64, i64, vp],
        "oracle_epilogue_gate_up_f32": [vp, vp, vp, i64, i64, vp],
        "oracle_epilogue_scale_f32": [vp, vp, vp, i64, i64, vp],
        "oracle_moe_forward_fp8": [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp,
                                   ctypes.POINTER(_Dump)],
        "oracle_smooth_factors": [vp, vp, i64, ctypes.c_double, vp],
        "oracle_quantize_rows_smoothed": [vp, vp, i64, i64, vp, vp],
        "oracle_moe_forward_smooth": [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp,
                                      ctypes.POINTER(_Dump), vp, vp],
        "oracle_num_threads": [],
        "oracle_set_num_threads": [ctypes.c_int],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int if name != "oracle_set_num_threads" else None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily route every function of this module to another build of
    the oracle (the tests use it to run the pins against planted mistakes)."""
    global _lib
    _load()
    with _lock:
        saved, _lib = _lib, open_library(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        names = {-1: "invalid argument", -2: "int32 overflow", -3: "out of memory"}
        raise OracleError(f"{what}: {names.get(rc, rc)}")


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def bf16_to_f32(x_bits: np.ndarray) -> np.ndarray:
    x_bits = _c(x_bits, np.uint16)
    out = np.empty(x_bits.shape, np.float32)
    _check(_load().oracle_bf16_to_f32(_p(x_bits), x_bits.size, _p(out)), "bf16_to_f32")
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _check(_load().oracle_f32_to_bf16(_p(x), x.size, _p(out)), "f32_to_bf16")
    return out


def quantize_rows(x: np.ndarray):
    """Per-row symmetric INT8 quantisation of a 2-D fp32 array -> (q int8, s fp32)."""
    x = _c(x, np.float32)
    rows, K = x.shape
    q = np.empty((rows, K), np.int8)
    s = np.empty(rows, np.float32)
    _check(_load().oracle_quantize_rows(_p(x), rows, K, _p(q), _p(s)), "quantize_rows")
    return q, s


def quantize_rows_bf16(x_bits: np.ndarray):
    """Per-row quantisation of a 2-D bf16 (uint16 bits) array -> (q, s)."""
    x_bits = _c(x_bits, np.uint16)
    rows, K = x_bits.shape
    q = np.empty((rows, K), np.int8)
    s = np.empty(rows, np.float32)
    _check(_load().oracle_quantize_rows_bf16(_p(x_bits), rows, K, _p(q), _p(s)), "quantize_rows_bf16")
    return q, s


def router(x_bits, Wr, bias, k):
    """-> (topk_ids int32 [T,k], topk_w fp32 [T,k], logits fp32 [T,E])."""
    x_bits = _c(x_bits, np.uint16)
    Wr = _c(Wr, np.float32)
    T, H = x_bits.shape
    E = Wr.shape[1]
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    logits = np.empty((T, E), np.float32)
    _check(_load().oracle_router(_p(x_bits), _p(Wr), _p(b), T, H, E, k, _p(ids), _p(w), _p(logits)),
           "router")
    return ids, w, logits


def permute(topk_ids, E):
    """-> (counts [E], offsets [E+1], slot_of [T,k], slot_token [T*k]), all int32."""
    topk_ids = _c(topk_ids, np.int32)
    T, k = topk_ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot_of = np.empty((T, k), np.int32)
    slot_token = np.empty(T * k, np.int32)
    _check(_load().oracle_permute(_p(topk_ids), T, E, k, _p(counts), _p(offsets), _p(slot_of),
                                  _p(slot_token)), "permute")
    return counts, offsets, slot_of, slot_token


def gemm_s8(a, b):
    """acc[m][n] = sum_k a[m][k] * b[n][k] exactly (int32 result)."""
    a = _c(a, np.int8)
    b = _c(b, np.int8)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == K
    acc = np.empty((M, N), np.int32)
    _check(_load().oracle_gemm_s8(_p(a), _p(b), M, N, K, _p(acc)), "gemm_s8")
    return acc


def epilogue_gate_up(acc1, s_act, s_w13):
    acc1 = _c(acc1, np.int32)
    S, two_i = acc1.shape
    I = two_i // 2
    s_act = _c(s_act, np.float32)
    s_w13 = _c(s_w13, np.float32)
    h = np.empty((S, I), np.float32)
    _check(_load().oracle_epilogue_gate_up(_p(acc1), _p(s_act), _p(s_w13), S, I, _p(h)),
           "epilogue_gate_up")
    return h


def epilogue_scale(acc, s_act, s_w):
    acc = _c(acc, np.int32)
    S, N = acc.shape
    s_act = _c(s_act, np.float32)
    s_w = _c(s_w, np.float32)
    out = np.empty((S, N), np.float32)
    _check(_load().oracle_epilogue_scale(_p(acc), _p(s_act), _p(s_w), S, N, _p(out)), "epilogue_scale")
    return out


def combine(o, slot_of, topk_w):
    o = _c(o, np.float32)
    slot_of = _c(slot_of, np.int32)
    topk_w = _c(topk_w, np.float32)
    T, k = slot_of.shape
    H = o.shape[1]
    y = np.empty((T, H), np.uint16)
    _check(_load().oracle_combine(_p(o), _p(slot_of), _p(topk_w), T, k, H, _p(y)), "combine")
    return y


_DUMP_SPEC = {
    "topk_ids": (np.int32, lambda T, H, I, E, k: (T, k)),
    "topk_w": (np.float32, lambda T, H, I, E, k: (T, k)),
    "offsets": (np.int32, lambda T, H, I, E, k: (E + 1,)),
    "slot_of": (np.int32, lambda T, H, I, E, k: (T, k)),
    "slot_token": (np.int32, lambda T, H, I, E, k: (T * k,)),
    "s_x": (np.float32, lambda T, H, I, E, k: (T,)),
    "q_x": (np.int8, lambda T, H, I, E, k: (T, H)),
    "acc1": (np.int32, lambda T, H, I, E, k: (T * k, 2 * I)),
    "h": (np.float32, lambda T, H, I, E, k: (T * k, I)),
    "s_h": (np.float32, lambda T, H, I, E, k: (T * k,)),
    "q_h": (np.int8, lambda T, H, I, E, k: (T * k, I)),
    "acc2": (np.int32, lambda T, H, I, E, k: (T * k, H)),
    "o": (np.float32, lambda T, H, I, E, k: (T * k, H)),
}


def moe_forward(x_bits, Wr, bias, w13_q, s_w13, w2_q, s_w2, k, dump=()):
    """Sparse-path layer forward.  Returns y (bf16 bits [T,H]) and, if
    ``dump`` names intermediates, a dict of them."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    w13_q = _c(w13_q, np.int8)
    E, two_i, _ = w13_q.shape
    I = two_i // 2
    Wr = _c(Wr, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    s_w13 = _c(s_w13, np.float32)
    w2_q = _c(w2_q, np.int8)
    s_w2 = _c(s_w2, np.float32)
    y = np.empty((T, H), np.uint16)
    out = {}
    d = _Dump()
    for name in dump:
        dt, shape = _DUMP_SPEC[name]
        arr = np.empty(shape(T, H, I, E, k), dt)
        out[name] = arr
        setattr(d, name, arr.ctypes.data)
    _check(_load().oracle_moe_forward(_p(x_bits), _p(Wr), _p(b), _p(w13_q), _p(s_w13), _p(w2_q),
                                      _p(s_w2), T, H, I, E, k, _p(y), ctypes.byref(d)), "moe_forward")
    return (y, out) if dump else y


def moe_forward_dense(x_bits, Wr, bias, w13_q, s_w13, w2_q, s_w2, k):
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    w13_q = _c(w13_q, np.int8)
    E, two_i, _ = w13_q.shape
    I = two_i // 2
    Wr = _c(Wr, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    y = np.empty((T, H), np.uint16)
    _check(_load().oracle_moe_forward_dense(_p(x_bits), _p(Wr), _p(b), _p(w13_q),
                                            _p(_c(s_w13, np.float32)), _p(_c(w2_q, np.int8)),
                                            _p(_c(s_w2, np.float32)), T, H, I, E, k, _p(y)),
           "moe_forward_dense")
    return y


def linear(x_bits, w_q, s_w, want_intermediates=False):
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    w_q = _c(w_q, np.int8)
    N = w_q.shape[0]
    s_w = _c(s_w, np.float32)
    y = np.empty((M, N), np.uint16)
    q_x = np.empty((M, K), np.int8) if want_intermediates else None
    s_x = np.empty(M, np.float32) if want_intermediates else None
    acc = np.empty((M, N), np.int32) if want_intermediates else None
    _check(_load().oracle_linear(_p(x_bits), _p(w_q), _p(s_w), M, N, K, _p(y), _p(q_x), _p(s_x),
                                 _p(acc)), "linear")
    if want_intermediates:
        return y, {"q_x": q_x, "s_x": s_x, "acc": acc}
    return y


# ---- FP8 (E4M3) variant (oracle.c, "FP8 (E4M3) variant of the layer") ----

def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code of each binary32 value (ties to even, saturating)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _check(_load().oracle_e4m3_encode(_p(x), x.size, _p(out)), "e4m3_encode")
    return out


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float32)
    _check(_load().oracle_e4m3_decode(_p(codes), codes.size, _p(out)), "e4m3_decode")
    return out


def quantize_rows_fp8(x: np.ndarray):
    """Per-row E4M3 quantisation of a 2-D fp32 array -> (codes uint8, s fp32)."""
    x = _c(x, np.float32)
    rows, K = x.shape
    q = np.empty((rows, K), np.uint8)
    s = np.empty(rows, np.float32)
    _check(_load().oracle_quantize_rows_fp8(_p(x), rows, K, _p(q), _p(s)), "quantize_rows_fp8")
    return q, s


def quantize_rows_bf16_fp8(x_bits: np.ndarray):
    x_bits = _c(x_bits, np.uint16)
    rows, K = x_bits.shape
    q = np.empty((rows, K), np.uint8)
    s = np.empty(rows, np.float32)
    _check(_load().oracle_quantize_rows_bf16_fp8(_p(x_bits), rows, K, _p(q), _p(s)), "quantize_rows_bf16_fp8")
    return q, s


def gemm_fp8(a, b):
    """acc[m][n] = binary32(exact sum_k value(a[m][k]) * value(b[n][k]))."""
    a = _c(a, np.uint8)
    b = _c(b, np.uint8)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == K
    acc = np.empty((M, N), np.float32)
    _check(_load().oracle_gemm_fp8(_p(a), _p(b), M, N, K, _p(acc)), "gemm_fp8")
    return acc


def epilogue_gate_up_f32(acc1, s_act, s_w13):
    acc1 = _c(acc1, np.float32)
    S, two_i = acc1.shape
    I = two_i // 2
    h = np.empty((S, I), np.float32)
    _check(_load().oracle_epilogue_gate_up_f32(_p(acc1), _p(_c(s_act, np.float32)), _p(_c(s_w13, np.float32)),
                                               S, I, _p(h)), "epilogue_gate_up_f32")
    return h


def epilogue_scale_f32(acc, s_act, s_w):
    acc = _c(acc, np.float32)
    S, N = acc.shape
    out = np.empty((S, N), np.float32)
    _check(_load().oracle_epilogue_scale_f32(_p(acc), _p(_c(s_act, np.float32)), _p(_c(s_w, np.float32)),
                                             S, N, _p(out)), "epilogue_scale_f32")
    return out


_DUMP_SPEC_FP8 = dict(_DUMP_SPEC, q_x=(np.uint8, _DUMP_SPEC["q_x"][1]), q_h=(np.uint8, _DUMP_SPEC["q_h"][1]),
                      acc1=(np.float32, _DUMP_SPEC["acc1"][1]), acc2=(np.float32, _DUMP_SPEC["acc2"][1]))


def moe_forward_fp8(x_bits, Wr, bias, w13_q, s_w13, w2_q, s_w2, k, dump=()):
    """FP8 layer forward (E4M3 codes as uint8).  Returns y (bf16 bits) and,
    if ``dump`` names intermediates, a dict of them (q_x, q_h: E4M3 codes;
    acc1, acc2: binary32)."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    w13_q = _c(w13_q, np.uint8)
    E, two_i, _ = w13_q.shape
    I = two_i // 2
    Wr = _c(Wr, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    y = np.empty((T, H), np.uint16)
    out = {}
    d = _Dump()
    for name in dump:
        dt, shape = _DUMP_SPEC_FP8[name]
        arr = np.empty(shape(T, H, I, E, k), dt)
        out[name] = arr
        setattr(d, name, arr.ctypes.data)
    _check(_load().oracle_moe_forward_fp8(_p(x_bits), _p(Wr), _p(b), _p(w13_q), _p(_c(s_w13, np.float32)),
                                          _p(_c(w2_q, np.uint8)), _p(_c(s_w2, np.float32)), T, H, I, E, k,
                                          _p(y), ctypes.byref(d)), "moe_forward_fp8")
    return (y, out) if dump else y


# ---- SmoothQuant-folded activations, calibrated per expert -------------------

def smooth_factors(x_absmax, w_absmax, alpha=0.5):
    """Per-channel factors max|X|^alpha / max|W|^(1 - alpha) (1 where a
    statistic is 0), computed in binary64 and rounded once to binary32."""
    a = _c(x_absmax, np.float32)
    b = _c(w_absmax, np.float32)
    if a.shape != b.shape:
        raise ValueError("x_absmax and w_absmax differ in shape")
    out = np.empty(a.shape, np.float32)
    _check(_load().oracle_smooth_factors(_p(a), _p(b), a.size, float(alpha), _p(out)), "smooth_factors")
    return out


def quantize_rows_smoothed(w, s):
    """Per-row INT8 quantisation of the folded rows w[r][k] * s[k]."""
    w = _c(w, np.float32)
    s = _c(s, np.float32)
    rows, K = w.shape
    if s.shape != (K,):
        raise ValueError("s must hold one factor per column")
    q = np.empty((rows, K), np.int8)
    sc = np.empty(rows, np.float32)
    _check(_load().oracle_quantize_rows_smoothed(_p(w), _p(s), rows, K, _p(q), _p(sc)), "quantize_rows_smoothed")
    return q, sc


def moe_forward_smooth(x_bits, Wr, bias, smooth, w13_q, s_w13, w2_q, s_w2, k, dump=()):
    """The layer with per-expert smoothing factors ``smooth [E, H]`` (w13_q
    folded with them).  ``dump`` may also name "s_slot" and "q_slot"."""
    x_bits = _c(x_bits, np.uint16)
    T, H = x_bits.shape
    w13_q = _c(w13_q, np.int8)
    E, two_i, _ = w13_q.shape
    I = two_i // 2
    smooth = _c(smooth, np.float32)
    if smooth.shape != (E, H):
        raise ValueError("smooth must be [E, H]")
    Wr = _c(Wr, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    s_w13 = _c(s_w13, np.float32)
    w2_q = _c(w2_q, np.int8)
    s_w2 = _c(s_w2, np.float32)
    y = np.empty((T, H), np.uint16)
    out = {}
    d = _Dump()
    for name in dump:
        if name in ("s_slot", "q_slot"):
            continue
        dt, shape = _DUMP_SPEC[name]
        arr = np.empty(shape(T, H, I, E, k), dt)
        out[name] = arr
        setattr(d, name, arr.ctypes.data)
    s_slot = np.empty(T * k, np.float32) if "s_slot" in dump else None
    q_slot = np.empty((T * k, H), np.int8) if "q_slot" in dump else None
    if s_slot is not None:
        out["s_slot"] = s_slot
    if q_slot is not None:
        out["q_slot"] = q_slot
    _check(_load().oracle_moe_forward_smooth(_p(x_bits), _p(Wr), _p(b), _p(smooth), _p(w13_q), _p(s_w13), _p(w2_q),
                                             _p(s_w2), T, H, I, E, k, _p(y), ctypes.byref(d), _p(s_slot), _p(q_slot)),
           "moe_forward_smooth")
    return (y, out) if dump else y
