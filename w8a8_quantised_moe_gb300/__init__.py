"""W8A8 quantised mixture-of-experts layer for GB300 (sm_103a).

Python front end of the C ABI in ``include/moe_w8a8.h``.  PyTorch provides
device memory and streams; every step of the layer runs in the CUDA library
``libmoe_w8a8.so`` (built in-tree by ``build.py``).  There is no CPU or
PyTorch fallback: without the library every call raises.

    import torch, w8a8_quantised_moe_gb300 as moe
    w13_q, w13_s = moe.quantize_weights(w13_fp32.view(-1, H))   # offline
    w2_q, w2_s = moe.quantize_weights(w2_fp32.view(-1, I))
    y = moe.forward(x, router_w, None, w13_q.view(E, 2 * I, H), w13_s.view(E, 2 * I),
                    w2_q.view(E, H, I), w2_s.view(E, H), top_k=2)
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import MoeError, STATUS

__all__ = [
    "MoeError", "STATUS", "quantize_weights", "workspace_size", "new_workspace", "forward", "forward_debug",
    "forward_host", "host_chunks", "quantize_weights_smoothed", "forward_smooth", "forward_fused",
    "fused_supported", "linear_workspace_size", "linear",
    "device_error", "set_wait_timeout_ns", "set_gemm_path", "GEMM_PATHS", "version",
    "fp8_quantize_weights", "fp8_forward", "fp8_forward_debug", "fp8_forward_host",
]


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t, dtype, shape, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous cuda {dtype} {tuple(shape)}, got {t.dtype} "
                         f"{tuple(t.shape)} on {t.device}")


def version() -> int:
    return _lib.load().moe_w8a8_version()


def set_wait_timeout_ns(ns: int) -> int:
    """Time limit of every in-kernel wait for later launches; returns the previous one."""
    return int(_lib.load().moe_w8a8_set_wait_timeout_ns(int(ns)))


# kernel choices of moe_w8a8_set_gemm_path
GEMM_PATHS = {"auto": -1, "wide": 0, "mid": 1, "narrow": 2, "pair": 3, "skinny": 4}


def set_gemm_path(path: str) -> str:
    """Force the GEMM kernel of later launches ("auto" restores the automatic
    choice); returns the previous setting.  A test hook: every path computes
    the same bits."""
    prev = _lib.load().moe_w8a8_set_gemm_path(GEMM_PATHS[path])
    if prev < -1:
        raise ValueError(path)
    return {v: k for k, v in GEMM_PATHS.items()}[prev]


def quantize_weights(w, stream=None):
    """Per-output-channel INT8 quantisation of fp32 ``w [rows, K]`` -> (int8 [rows, K], fp32 [rows])."""
    torch = _torch()
    rows, K = w.shape
    _need(w, torch.float32, (rows, K), "w")
    q = torch.empty((rows, K), dtype=torch.int8, device=w.device)
    s = torch.empty((rows,), dtype=torch.float32, device=w.device)
    _lib.check(_lib.load().moe_w8a8_quantize_weights(_ptr(w), rows, K, _ptr(q), _ptr(s), _stream(stream)),
               "moe_w8a8_quantize_weights")
    return q, s


def workspace_size(T, H, I, E, top_k) -> int:
    n = _lib.load().moe_w8a8_workspace_size(T, H, I, E, top_k)
    if n == 0:
        raise MoeError(-2, "moe_w8a8_workspace_size")
    return int(n)


def new_workspace(nbytes: int, device="cuda"):
    """A zeroed device workspace (the error word starts cleared)."""
    torch = _torch()
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def _forward_args(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, code_dtype=None):
    torch = _torch()
    code_dtype = torch.int8 if code_dtype is None else code_dtype
    T, H = x.shape
    E = router_w.shape[1]
    I = w2_q.shape[2] if w2_q.dim() == 3 else 0
    _need(x, torch.bfloat16, (T, H), "x")
    _need(router_w, torch.float32, (H, E), "router_w")
    if router_bias is not None:
        _need(router_bias, torch.float32, (E,), "router_bias")
    _need(w13_q, code_dtype, (E, 2 * I, H), "w13_q")
    _need(w13_scale, torch.float32, (E, 2 * I), "w13_scale")
    _need(w2_q, code_dtype, (E, H, I), "w2_q")
    _need(w2_scale, torch.float32, (E, H), "w2_scale")
    return T, H, I, E


def forward(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, workspace=None, out=None,
            stream=None):
    """The MoE layer: bf16 x [T, H] -> bf16 y [T, H] (see include/moe_w8a8.h)."""
    torch = _torch()
    T, H, I, E = _forward_args(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k)
    need = workspace_size(T, H, I, E, top_k)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    y = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (T, H), "out")
    _lib.check(_lib.load().moe_w8a8_forward(
        _ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(w13_q), _ptr(w13_scale), _ptr(w2_q), _ptr(w2_scale),
        T, H, I, E, top_k, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "moe_w8a8_forward")
    return y




def _need_host(t, dtype, shape, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda or t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous host {dtype} {tuple(shape)} (page-locked for the copies "
                         f"to overlap), got {t.dtype} {tuple(t.shape)} on {t.device}")

def host_chunks(T, H, I, E) -> int:
    """Token chunks ``forward_host`` takes when ``chunks`` is 0."""
    return int(_lib.load().moe_w8a8_host_chunks(T, H, I, E))


def _forward_host(fn, name, code_dtype, x_host, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k,
                  y_host, x_dev, y_dev, workspace, stream, copy_stream, chunks):
    torch = _torch()
    T, H = x_host.shape
    E = router_w.shape[1]
    I = w2_q.shape[2] if w2_q.dim() == 3 else 0
    _need_host(x_host, torch.bfloat16, (T, H), "x_host")
    _need(router_w, torch.float32, (H, E), "router_w")
    if router_bias is not None:
        _need(router_bias, torch.float32, (E,), "router_bias")
    _need(w13_q, code_dtype, (E, 2 * I, H), "w13_q")
    _need(w13_scale, torch.float32, (E, 2 * I), "w13_scale")
    _need(w2_q, code_dtype, (E, H, I), "w2_q")
    _need(w2_scale, torch.float32, (E, H), "w2_scale")
    dev = router_w.device
    if y_host is None:
        y_host = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    _need_host(y_host, torch.bfloat16, (T, H), "y_host")
    if x_dev is None:
        x_dev = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if y_dev is None:
        y_dev = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    _need(x_dev, torch.bfloat16, (T, H), "x_dev")
    _need(y_dev, torch.bfloat16, (T, H), "y_dev")
    if workspace is None:
        workspace = new_workspace(workspace_size(T, H, I, E, top_k), dev)
    cs = None if copy_stream is None else copy_stream.cuda_stream
    _lib.check(fn(
        _ptr(x_host), _ptr(router_w), _ptr(router_bias), _ptr(w13_q), _ptr(w13_scale), _ptr(w2_q), _ptr(w2_scale),
        T, H, I, E, top_k, _ptr(y_host), _ptr(x_dev), _ptr(y_dev), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream), cs, int(chunks)), name)
    return y_host


def forward_host(x_host, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, y_host=None, x_dev=None,
                 y_dev=None, workspace=None, stream=None, copy_stream=None, chunks=0):
    """The MoE layer on host-resident bf16 x [T, H] -> host bf16 y [T, H]:
    copies in and out inside the call, overlapped with compute on
    ``copy_stream`` (see include/moe_w8a8.h).  y_host is complete once
    ``stream`` is synchronised."""
    torch = _torch()
    return _forward_host(_lib.load().moe_w8a8_forward_host, "moe_w8a8_forward_host", torch.int8, x_host, router_w,
                         router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, y_host, x_dev, y_dev, workspace,
                         stream, copy_stream, chunks)

_DEBUG_FIELDS = {
    # name: (dtype, shape(T, H, I, E, k))
    "topk_ids": ("int32", lambda T, H, I, E, k: (T, k)),
    "topk_w": ("float32", lambda T, H, I, E, k: (T, k)),
    "offsets": ("int32", lambda T, H, I, E, k: (E + 1,)),
    "slot_of": ("int32", lambda T, H, I, E, k: (T, k)),
    "slot_token": ("int32", lambda T, H, I, E, k: (T * k,)),
    "s_x": ("float32", lambda T, H, I, E, k: (T,)),
    "q_x": ("int8", lambda T, H, I, E, k: (T, H)),
    "acc1": ("int32", lambda T, H, I, E, k: (T * k, 2 * I)),
    "h": ("float32", lambda T, H, I, E, k: (T * k, I)),
    "s_h": ("float32", lambda T, H, I, E, k: (T * k,)),
    "q_h": ("int8", lambda T, H, I, E, k: (T * k, I)),
    "acc2": ("int32", lambda T, H, I, E, k: (T * k, H)),
    "o": ("float32", lambda T, H, I, E, k: (T * k, H)),
    "s_slot": ("float32", lambda T, H, I, E, k: (T * k,)),
    "q_slot": ("int8", lambda T, H, I, E, k: (T * k, H)),
}


def forward_debug(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, fields=None,
                  workspace=None, stream=None):
    """``forward`` plus the intermediates named in ``fields`` (default: all)
    as device tensors.  Returns (y, dict)."""
    torch = _torch()
    T, H, I, E = _forward_args(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k)
    need = workspace_size(T, H, I, E, top_k)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    fields = tuple(_DEBUG_FIELDS) if fields is None else tuple(fields)
    bufs = _lib.DebugBuffers()
    out = {}
    for name in fields:
        dt, shape = _DEBUG_FIELDS[name]
        t = torch.zeros(shape(T, H, I, E, top_k), dtype=getattr(torch, dt), device=x.device)
        out[name] = t
        setattr(bufs, name, t.data_ptr())
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _lib.check(_lib.load().moe_w8a8_forward_debug(
        _ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(w13_q), _ptr(w13_scale), _ptr(w2_q), _ptr(w2_scale),
        T, H, I, E, top_k, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), ctypes.byref(bufs)), "moe_w8a8_forward_debug")
    return y, out



def fused_supported(T, H, I, E, top_k) -> bool:
    """Whether ``forward_fused`` takes the shape (few tokens: T <= 128)."""
    return bool(_lib.load().moe_w8a8_fused_supported(T, H, I, E, top_k))


def forward_fused(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, fields=(), workspace=None,
                  out=None, stream=None):
    """The MoE layer as one persistent kernel (few tokens; see
    include/moe_w8a8.h): the same result as ``forward`` bit for bit.  Returns
    y, or (y, dict of the intermediates named in ``fields``) when ``fields``
    is given (None: all)."""
    torch = _torch()
    T, H, I, E = _forward_args(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k)
    if workspace is None:
        workspace = new_workspace(workspace_size(T, H, I, E, top_k), x.device)
    y = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (T, H), "out")
    fields = tuple(_DEBUG_FIELDS) if fields is None else tuple(fields)
    bufs, dumps = None, {}
    if fields:
        bufs = _lib.DebugBuffers()
        for name in fields:
            dt, shape = _DEBUG_FIELDS[name]
            t = torch.zeros(shape(T, H, I, E, top_k), dtype=getattr(torch, dt), device=x.device)
            dumps[name] = t
            setattr(bufs, name, t.data_ptr())
    _lib.check(_lib.load().moe_w8a8_forward_fused(
        _ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(w13_q), _ptr(w13_scale), _ptr(w2_q), _ptr(w2_scale),
        T, H, I, E, top_k, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), ctypes.byref(bufs) if bufs is not None else None), "moe_w8a8_forward_fused")
    return (y, dumps) if fields else y

# ---- SmoothQuant-folded activations, calibrated per expert ------------------

def quantize_weights_smoothed(w, col_scale, stream=None):
    """Per-output-channel INT8 quantisation of fp32 ``w [rows, K]`` times the
    column factors ``col_scale [K]`` -> (int8 [rows, K], fp32 scales [rows])."""
    torch = _torch()
    rows, K = w.shape
    _need(w, torch.float32, (rows, K), "w")
    _need(col_scale, torch.float32, (K,), "col_scale")
    q = torch.empty((rows, K), dtype=torch.int8, device=w.device)
    s = torch.empty((rows,), dtype=torch.float32, device=w.device)
    _lib.check(_lib.load().moe_w8a8_quantize_weights_smoothed(_ptr(w), rows, K, _ptr(col_scale), _ptr(q), _ptr(s),
                                                              _stream(stream)), "moe_w8a8_quantize_weights_smoothed")
    return q, s


def forward_smooth(x, router_w, router_bias, smooth, w13_q, w13_scale, w2_q, w2_scale, top_k, fields=(),
                   workspace=None, out=None, stream=None):
    """The MoE layer with per-expert smoothing factors ``smooth [E, H]``
    (weights folded by ``quantize_weights_smoothed``).  Returns y, or (y,
    dict of the intermediates named in ``fields``) when ``fields`` is given."""
    torch = _torch()
    T, H, I, E = _forward_args(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k)
    _need(smooth, torch.float32, (E, H), "smooth")
    if workspace is None:
        workspace = new_workspace(workspace_size(T, H, I, E, top_k), x.device)
    y = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (T, H), "out")
    fields = tuple(_DEBUG_FIELDS) if fields is None else tuple(fields)
    bufs, dumps = None, {}
    if fields:
        bufs = _lib.DebugBuffers()
        for name in fields:
            dt, shape = _DEBUG_FIELDS[name]
            t = torch.zeros(shape(T, H, I, E, top_k), dtype=getattr(torch, dt), device=x.device)
            dumps[name] = t
            setattr(bufs, name, t.data_ptr())
    _lib.check(_lib.load().moe_w8a8_forward_smooth(
        _ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(smooth), _ptr(w13_q), _ptr(w13_scale), _ptr(w2_q),
        _ptr(w2_scale), T, H, I, E, top_k, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), ctypes.byref(bufs) if bufs is not None else None), "moe_w8a8_forward_smooth")
    return (y, dumps) if fields else y

def linear_workspace_size(M, N, K) -> int:
    n = _lib.load().moe_w8a8_linear_workspace_size(M, N, K)
    if n == 0:
        raise MoeError(-2, "moe_w8a8_linear_workspace_size")
    return int(n)


def linear(x, w_q, w_scale, workspace=None, out=None, stream=None):
    """W8A8 linear layer: bf16 x [M, K], int8 w_q [N, K], fp32 w_scale [N] -> bf16 [M, N]."""
    torch = _torch()
    M, K = x.shape
    N = w_q.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    _need(w_q, torch.int8, (N, K), "w_q")
    _need(w_scale, torch.float32, (N,), "w_scale")
    need = linear_workspace_size(M, N, K)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (M, N), "out")
    _lib.check(_lib.load().moe_w8a8_linear(_ptr(x), _ptr(w_q), _ptr(w_scale), M, N, K, _ptr(y), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream)),
               "moe_w8a8_linear")
    return y


def device_error(workspace, stream=None) -> int:
    """Synchronise the stream, read and clear the workspace's device error word (a status code)."""
    return int(_lib.load().moe_w8a8_device_error(_ptr(workspace), _stream(stream)))


# ---- FP8 (E4M3) variant: E4M3 codes travel as uint8 tensors ----------------

def fp8_quantize_weights(w, stream=None):
    """Per-output-channel E4M3 quantisation of fp32 ``w [rows, K]`` ->
    (E4M3 codes as uint8 [rows, K], fp32 scales [rows]); s = amax / 448."""
    torch = _torch()
    rows, K = w.shape
    _need(w, torch.float32, (rows, K), "w")
    q = torch.empty((rows, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((rows,), dtype=torch.float32, device=w.device)
    _lib.check(_lib.load().moe_w8a8_fp8_quantize_weights(_ptr(w), rows, K, _ptr(q), _ptr(s), _stream(stream)),
               "moe_w8a8_fp8_quantize_weights")
    return q, s


def fp8_forward(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, workspace=None, out=None,
                stream=None):
    """The FP8 MoE layer: bf16 x [T, H] -> bf16 y [T, H]; w13_q, w2_q E4M3 (uint8)."""
    torch = _torch()
    T, H, I, E = _forward_args(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, torch.uint8)
    need = workspace_size(T, H, I, E, top_k)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    y = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (T, H), "out")
    _lib.check(_lib.load().moe_w8a8_fp8_forward(
        _ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(w13_q), _ptr(w13_scale), _ptr(w2_q), _ptr(w2_scale),
        T, H, I, E, top_k, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "moe_w8a8_fp8_forward")
    return y


_DEBUG_FIELDS_FP8 = dict(_DEBUG_FIELDS, q_x=("uint8", _DEBUG_FIELDS["q_x"][1]),
                         q_slot=("uint8", _DEBUG_FIELDS["q_slot"][1]),
                         q_h=("uint8", _DEBUG_FIELDS["q_h"][1]), acc1=("float32", _DEBUG_FIELDS["acc1"][1]),
                         acc2=("float32", _DEBUG_FIELDS["acc2"][1]))


def fp8_forward_debug(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, fields=None,
                      workspace=None, stream=None):
    """``fp8_forward`` plus the intermediates named in ``fields`` (q_x, q_h:
    E4M3 codes; acc1, acc2: fp32 accumulators).  Returns (y, dict)."""
    torch = _torch()
    T, H, I, E = _forward_args(x, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, torch.uint8)
    need = workspace_size(T, H, I, E, top_k)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    fields = tuple(_DEBUG_FIELDS_FP8) if fields is None else tuple(fields)
    bufs = _lib.DebugBuffers()
    out = {}
    for name in fields:
        dt, shape = _DEBUG_FIELDS_FP8[name]
        t = torch.zeros(shape(T, H, I, E, top_k), dtype=getattr(torch, dt), device=x.device)
        out[name] = t
        setattr(bufs, name, t.data_ptr())
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _lib.check(_lib.load().moe_w8a8_fp8_forward_debug(
        _ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(w13_q), _ptr(w13_scale), _ptr(w2_q), _ptr(w2_scale),
        T, H, I, E, top_k, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), ctypes.byref(bufs)), "moe_w8a8_fp8_forward_debug")
    return y, out


def fp8_forward_host(x_host, router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, y_host=None,
                     x_dev=None, y_dev=None, workspace=None, stream=None, copy_stream=None, chunks=0):
    """``forward_host`` for the FP8 layer (w13_q, w2_q E4M3 as uint8)."""
    torch = _torch()
    return _forward_host(_lib.load().moe_w8a8_fp8_forward_host, "moe_w8a8_fp8_forward_host", torch.uint8, x_host,
                         router_w, router_bias, w13_q, w13_scale, w2_q, w2_scale, top_k, y_host, x_dev, y_dev,
                         workspace, stream, copy_stream, chunks)
