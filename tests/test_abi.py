"""The C ABI without a GPU: the library loads, exports every function that
include/moe_w8a8.h declares, and rejects bad arguments on the host before
anything is launched."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from w8a8_quantised_moe_gb300 import _lib
from w8a8_quantised_moe_gb300 import build as lib_build

HEADER = os.path.join(ROOT, "include", "moe_w8a8.h")
OK, INVALID, SHAPE, WS_SMALL = 0, -1, -2, -3
FAKE = 1 << 20  # an aligned, never dereferenced address


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_w8a8_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert sorted(_lib.EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_checked_build_compiles_and_exports_every_declared_symbol():
    """The checked build (-DMOE_CHECKED=1: data-derived indices range-checked
    in the kernels) is a separate library beside the normal one; it builds
    and loads here, and rejects the same bad arguments on the host."""
    checked = _lib.open_library(lib_build.build(checked=True))
    for name in declared_functions():
        assert hasattr(checked, name), name
    need = checked.moe_w8a8_linear_workspace_size(64, 256, 256)
    assert need > 0
    assert checked.moe_w8a8_linear(FAKE, FAKE, FAKE, 64, 256, 256, FAKE, FAKE, need - 1, None) == WS_SMALL
    assert checked.moe_w8a8_linear(FAKE, FAKE, FAKE, 64, 200, 256, FAKE, FAKE, need, None) == SHAPE


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.moe_w8a8_status_string(code).decode() == name
    assert lib.moe_w8a8_status_string(12345).decode() == "MOE_ERR_UNKNOWN"
    assert lib.moe_w8a8_version() >= 100


@pytest.mark.parametrize("shape", [
    (16, 100, 512, 8, 2),     # H not a multiple of 128
    (16, 256, 500, 8, 2),     # I not a multiple of 128
    (16, 256, 512, 0, 1),     # no experts
    (16, 256, 512, 257, 2),   # too many experts
    (16, 256, 512, 8, 0),     # top_k < 1
    (16, 256, 512, 8, 9),     # top_k > 8
    (16, 256, 512, 4, 5),     # top_k > E
    (-1, 256, 512, 8, 2),     # negative T
    (16, 32768, 512, 8, 2),   # H too large
])
def test_workspace_size_rejects_bad_shapes(lib, shape):
    assert lib.moe_w8a8_workspace_size(*shape) == 0


def test_workspace_size_grows_with_tokens(lib):
    a = lib.moe_w8a8_workspace_size(16, 256, 512, 8, 2)
    b = lib.moe_w8a8_workspace_size(32, 256, 512, 8, 2)
    assert 0 < a < b
    assert a % 256 == 0 and b % 256 == 0
    # the largest configuration stays a few GB
    big = lib.moe_w8a8_workspace_size(4096, 7168, 2048, 256, 8)
    assert 0 < big < 4 << 30


def _fwd(lib, T=16, H=256, I=512, E=8, k=2, ptrs=None, ws_bytes=None, bias=None):
    p = dict(x=FAKE, rw=FAKE, w13=FAKE, s13=FAKE, w2=FAKE, s2=FAKE, y=FAKE, ws=FAKE)
    p.update(ptrs or {})
    need = lib.moe_w8a8_workspace_size(T, H, I, E, k)
    return lib.moe_w8a8_forward(p["x"], p["rw"], bias, p["w13"], p["s13"], p["w2"], p["s2"], T, H, I, E, k,
                                p["y"], p["ws"], need if ws_bytes is None else ws_bytes, None)


def test_forward_rejects_bad_arguments_without_launching(lib):
    assert _fwd(lib, H=100) == SHAPE
    assert _fwd(lib, k=9) == SHAPE
    for name in ("x", "rw", "w13", "s13", "w2", "s2", "y", "ws"):
        assert _fwd(lib, ptrs={name: None}) == INVALID, name
        assert _fwd(lib, ptrs={name: FAKE + 4}) == INVALID, name  # misaligned
    assert _fwd(lib, bias=FAKE + 8) == INVALID
    assert _fwd(lib, ptrs={"ws": FAKE + 16}) == INVALID  # workspace must be 256-aligned
    assert _fwd(lib, ws_bytes=1024) == WS_SMALL


def test_forward_with_no_tokens_is_a_no_op(lib):
    # T == 0 passes every check and returns before touching the device
    assert _fwd(lib, T=0) == OK



def _fwd_host(lib, T=16, H=256, I=512, E=8, k=2, ptrs=None, ws_bytes=None, chunks=0, fn="moe_w8a8_forward_host"):
    p = dict(xh=FAKE, rw=FAKE, w13=FAKE, s13=FAKE, w2=FAKE, s2=FAKE, yh=FAKE, xd=FAKE, yd=FAKE, ws=FAKE)
    p.update(ptrs or {})
    need = lib.moe_w8a8_workspace_size(T, H, I, E, k)
    return getattr(lib, fn)(p["xh"], p["rw"], None, p["w13"], p["s13"], p["w2"], p["s2"], T, H, I, E, k, p["yh"],
                            p["xd"], p["yd"], p["ws"], need if ws_bytes is None else ws_bytes, None, None, chunks)


@pytest.mark.parametrize("fn", ["moe_w8a8_forward_host", "moe_w8a8_fp8_forward_host"])
def test_forward_host_rejects_bad_arguments_without_copying(lib, fn):
    assert _fwd_host(lib, H=100, fn=fn) == SHAPE
    for name in ("xh", "rw", "w13", "s13", "w2", "s2", "yh", "xd", "yd", "ws"):
        assert _fwd_host(lib, ptrs={name: None}, fn=fn) == INVALID, name
        assert _fwd_host(lib, ptrs={name: FAKE + 4}, fn=fn) == INVALID, name
    assert _fwd_host(lib, chunks=-1, fn=fn) == INVALID
    assert _fwd_host(lib, chunks=17, fn=fn) == INVALID
    assert _fwd_host(lib, ws_bytes=1024, fn=fn) == WS_SMALL
    assert _fwd_host(lib, T=0, fn=fn) == OK  # no tokens: nothing is copied or launched


def test_host_chunk_rule(lib):
    # prefill-shaped: x moves over the host link more slowly than HBM streams the weights -> 2
    assert lib.moe_w8a8_host_chunks(8192, 4096, 1536, 64) == 2
    # weights dominate (256 experts) or few tokens -> 1
    assert lib.moe_w8a8_host_chunks(4096, 7168, 2048, 256) == 1
    assert lib.moe_w8a8_host_chunks(64, 4096, 1536, 64) == 1
    assert lib.moe_w8a8_host_chunks(2047, 4096, 128, 1) == 1
    assert lib.moe_w8a8_host_chunks(0, 4096, 1536, 64) == 1
    assert lib.moe_w8a8_host_chunks(-1, 4096, 1536, 64) == 0

def test_linear_rejects_bad_arguments(lib):
    need = lib.moe_w8a8_linear_workspace_size(64, 256, 256)
    assert need > 0
    assert lib.moe_w8a8_linear_workspace_size(64, 100, 256) == 0
    assert lib.moe_w8a8_linear_workspace_size(64, 256, 0) == 0
    assert lib.moe_w8a8_linear(FAKE, FAKE, FAKE, 64, 256, 256, FAKE, FAKE, need - 1, None) == WS_SMALL
    assert lib.moe_w8a8_linear(None, FAKE, FAKE, 64, 256, 256, FAKE, FAKE, need, None) == INVALID
    assert lib.moe_w8a8_linear(FAKE, FAKE, FAKE, 64, 200, 256, FAKE, FAKE, need, None) == SHAPE
    assert lib.moe_w8a8_linear(FAKE, FAKE, FAKE, 0, 256, 256, FAKE, FAKE, need, None) == OK


def test_quantize_weights_argument_checks(lib):
    assert lib.moe_w8a8_quantize_weights(FAKE, 0, 64, FAKE, FAKE, None) == OK  # no rows
    assert lib.moe_w8a8_quantize_weights(FAKE, 4, 0, FAKE, FAKE, None) == SHAPE
    assert lib.moe_w8a8_quantize_weights(FAKE, -1, 64, FAKE, FAKE, None) == SHAPE
    assert lib.moe_w8a8_quantize_weights(None, 4, 64, FAKE, FAKE, None) == INVALID
    assert lib.moe_w8a8_quantize_weights(FAKE, 4, 64, FAKE + 1, FAKE, None) == INVALID


def test_device_error_rejects_bad_workspace(lib):
    assert lib.moe_w8a8_device_error(None, None) == INVALID
    assert lib.moe_w8a8_device_error(FAKE + 16, None) == INVALID


def test_wait_timeout_setting_round_trips(lib):
    prev = lib.moe_w8a8_set_wait_timeout_ns(12345)
    assert lib.moe_w8a8_set_wait_timeout_ns(prev) == 12345
    assert lib.moe_w8a8_set_wait_timeout_ns(0) == prev  # 0 restores the default
    assert lib.moe_w8a8_set_wait_timeout_ns(0) == 2_000_000_000


def test_python_front_end_fails_loudly_without_library(tmp_path, monkeypatch):
    import w8a8_quantised_moe_gb300 as moe
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError):
        _lib.load(str(tmp_path / "missing.so"))
    assert moe.__name__  # the package itself imports without the library


def test_smoothed_entry_points_reject_bad_arguments(lib):
    T, H, I, E, k = 16, 256, 512, 8, 2
    need = lib.moe_w8a8_workspace_size(T, H, I, E, k)

    def fwd(smooth=FAKE, T=T, x=FAKE):
        return lib.moe_w8a8_forward_smooth(x, FAKE, None, smooth, FAKE, FAKE, FAKE, FAKE, T, H, I, E, k, FAKE, FAKE,
                                           need, None, None)
    assert fwd(smooth=None) == INVALID
    assert fwd(smooth=FAKE + 4) == INVALID
    assert fwd(x=None) == INVALID
    assert fwd(T=0, smooth=None) == OK  # no tokens: nothing is read
    q = lib.moe_w8a8_quantize_weights_smoothed
    assert q(FAKE, 4, 128, None, FAKE, FAKE, None) == INVALID
    assert q(FAKE, 4, 128, FAKE + 4, FAKE, FAKE, None) == INVALID
    assert q(FAKE, 4, 0, FAKE, FAKE, FAKE, None) == SHAPE
    assert q(FAKE, 0, 128, FAKE, FAKE, FAKE, None) == OK


# ---- host-side fault injection (MOE_INJECT): every host status code ----

NOT_IMPL, CUDA = -6, -4


def test_injected_faults_take_each_host_error_path(lib, monkeypatch):
    need = lib.moe_w8a8_linear_workspace_size(64, 256, 256)
    monkeypatch.setenv("MOE_INJECT", "ws_short")
    assert _fwd(lib) == WS_SMALL
    assert _fwd_host(lib) == WS_SMALL
    assert lib.moe_w8a8_linear(FAKE, FAKE, FAKE, 64, 256, 256, FAKE, FAKE, need, None) == WS_SMALL
    monkeypatch.setenv("MOE_INJECT", "bad_ptr")
    assert _fwd(lib) == INVALID
    assert _fwd_host(lib) == INVALID
    assert lib.moe_w8a8_linear(FAKE, FAKE, FAKE, 64, 256, 256, FAKE, FAKE, need, None) == INVALID
    assert lib.moe_w8a8_linear_static(FAKE, FAKE, FAKE, 64, 256, 256, FAKE, None) == INVALID
    assert lib.moe_w8a8_quantize_weights(FAKE, 4, 64, FAKE, FAKE, None) == INVALID
    monkeypatch.setenv("MOE_INJECT", "launch_fail")
    assert _fwd(lib) == CUDA
    assert lib.moe_w8a8_linear(FAKE, FAKE, FAKE, 64, 256, 256, FAKE, FAKE, need, None) == CUDA
    assert lib.moe_w8a8_linear_static(FAKE, FAKE, FAKE, 64, 256, 256, FAKE, None) == CUDA
    assert lib.moe_w8a8_quantize_weights(FAKE, 4, 64, FAKE, FAKE, None) == CUDA
    assert lib.moe_w8a8_fp8_quantize_weights(FAKE, 4, 64, FAKE, FAKE, None) == CUDA
    # several faults at once: the argument checks come first
    monkeypatch.setenv("MOE_INJECT", "launch_fail,ws_short")
    assert _fwd(lib) == WS_SMALL
    # the checks themselves still run: a real shape error wins over an injected fault
    assert _fwd(lib, H=100) == SHAPE
    monkeypatch.delenv("MOE_INJECT")
    assert _fwd(lib, T=0) == OK


def _fused(lib, T=16, H=256, I=512, E=8, k=2, ptrs=None, ws_bytes=None):
    p = dict(x=FAKE, rw=FAKE, w13=FAKE, s13=FAKE, w2=FAKE, s2=FAKE, y=FAKE, ws=FAKE)
    p.update(ptrs or {})
    need = lib.moe_w8a8_workspace_size(T, H, I, E, k)
    return lib.moe_w8a8_forward_fused(p["x"], p["rw"], None, p["w13"], p["s13"], p["w2"], p["s2"], T, H, I, E, k,
                                      p["y"], p["ws"], need if ws_bytes is None else ws_bytes, None, None)


def test_fused_layer_shapes_and_argument_checks(lib, monkeypatch):
    ok = lib.moe_w8a8_fused_supported
    assert ok(1, 256, 128, 1, 1) and ok(64, 4096, 1536, 64, 2) and ok(128, 7168, 2048, 256, 8)
    assert ok(128, 16384, 16384, 256, 8)      # the largest layer
    assert not ok(129, 4096, 1536, 64, 2)     # more tokens than the few-token router takes
    assert not ok(64, 4096, 1544, 64, 2)      # not a shape of the forward at all
    assert not ok(64, 4032, 1536, 64, 2)      # H not a multiple of 128
    assert not ok(0, 4096, 1536, 64, 2)
    assert _fused(lib, T=129) == SHAPE
    assert _fused(lib, I=100) == SHAPE
    assert _fused(lib, T=0) == OK  # no tokens: nothing is launched
    for name in ("x", "rw", "w13", "s13", "w2", "s2", "y", "ws"):
        assert _fused(lib, ptrs={name: None}) == INVALID, name
        assert _fused(lib, ptrs={name: FAKE + 4}) == INVALID, name
    assert _fused(lib, ptrs={"ws": FAKE + 16}) == INVALID
    assert _fused(lib, ws_bytes=1024) == WS_SMALL
    monkeypatch.setenv("MOE_INJECT", "ws_short")
    assert _fused(lib) == WS_SMALL
    monkeypatch.setenv("MOE_INJECT", "bad_ptr")
    assert _fused(lib) == INVALID
    monkeypatch.setenv("MOE_INJECT", "launch_fail")
    assert _fused(lib) == CUDA


def test_fp8_layer_refuses_a_forced_int8_kernel(lib):
    T, H, I, E, k = 16, 256, 512, 8, 2
    need = lib.moe_w8a8_workspace_size(T, H, I, E, k)
    prev = lib.moe_w8a8_set_gemm_path(3)
    try:
        assert lib.moe_w8a8_fp8_forward(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, T, H, I, E, k, FAKE, FAKE, need,
                                        None) == NOT_IMPL
        assert _fwd_host(lib, fn="moe_w8a8_fp8_forward_host") == NOT_IMPL
    finally:
        lib.moe_w8a8_set_gemm_path(prev)


def test_every_host_status_code_is_produced():
    # the codes the tests above produce; the two device codes are produced on
    # the GPU (test_gpu_timeout.py) and by moe_w8a8_device_error
    produced = {OK, INVALID, SHAPE, WS_SMALL, CUDA, NOT_IMPL}
    device = {-5, -7}
    assert set(_lib.STATUS) == produced | device
