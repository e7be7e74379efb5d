"""The checked build (-DMOE_CHECKED=1): every index a kernel takes from data
(expert ids, slots, expert offsets, exact-path lists, gathered rows) is
range-checked, and one out of range sets the device error word
(MOE_ERR_DEVICE) instead of being read or written.  It stands in for a
memory checker, which this pool does not offer.

Checked through the C ABI of the checked library, loaded beside the normal
one:
  * on valid inputs it gives the normal build's results bit for bit (MoE
    layers on each GEMM kernel and quantiser form, with a router bias and
    top-8, the FP8 layer, the linear layer, the one-kernel layer) and leaves
    the error word clear; one layer is also compared with the oracle;
  * a slot index out of range, planted by its test hook after the quantiser
    (MOE_INJECT=bad_slot overwrites slot_of[0] with 0x7f7f7f7f), is caught by
    the combine's check: MOE_ERR_DEVICE, no fault, every other token's output
    unchanged, and the next call clean;
  * the normal build ignores that hook."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import _lib
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl
from gpu_helpers import Layer, assert_y_close, bf16_from_dev, bf16_to_dev

pytestmark = pytest.mark.gpu

OK, DEVICE = 0, -7
TINY = wl.CONFIGS["tiny"]
SHAPES = {
    "tiny": TINY,                                                        # dp4a GEMMs, CTA-per-token quantiser
    "mid": TINY.replace(T=300, H=512, I=384, E=8, k=2),                  # one-CTA tensor-core GEMMs
    "pair": TINY.replace(T=1500, H=1280, I=256, E=4, k=2),              # CTA pairs, two warps per token
    "decode": TINY.replace(T=64, H=1024, I=512, E=16, k=2),              # few rows per expert
    "top8": TINY.replace(T=600, H=256, I=128, E=256, k=8, bias="normal", bias_std=0.5),  # router bias, top-8
}


@pytest.fixture(scope="module")
def libs():
    lib_build.build()
    oracle.build()
    normal = _lib.load()
    checked = _lib.open_library(lib_build.build(checked=True))
    return normal, checked


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _forward(lib, layer, fp8=False, args=None):
    cfg = layer.cfg if layer is not None else None
    a = args if args is not None else layer.device_args()
    x, Wr, bias, w13, s13, w2, s2, k = a
    T, H = x.shape
    E, I2 = w13.shape[0], w13.shape[1]
    I = I2 // 2
    ws = moe.new_workspace(moe.workspace_size(T, H, I, E, k))
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    fn = lib.moe_w8a8_fp8_forward if fp8 else lib.moe_w8a8_forward
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    status = fn(ptr(x), ptr(Wr), ptr(bias), ptr(w13), ptr(s13), ptr(w2), ptr(s2), T, H, I, E, k, ptr(y),
                ptr(ws), ws.numel(), _stream())
    assert status == OK, status
    err = lib.moe_w8a8_device_error(ws.data_ptr(), _stream())
    return bf16_from_dev(y), err


@pytest.mark.parametrize("name", list(SHAPES))
def test_checked_build_equals_normal_build(libs, name):
    normal, checked = libs
    layer = Layer(SHAPES[name])
    y_n, e_n = _forward(normal, layer)
    y_c, e_c = _forward(checked, layer)
    assert e_n == OK and e_c == OK, (e_n, e_c)
    np.testing.assert_array_equal(y_c, y_n)
    if name == "mid":
        assert_y_close(y_c, layer.oracle())


def test_checked_build_equals_normal_build_fp8(libs):
    normal, checked = libs
    cfg = TINY.replace(T=1000, H=512, I=256, E=4, k=2)
    inp = wl.make_moe_inputs(cfg, 0)
    w13 = torch.stack([wl.expert_weight_fp32(cfg, "w13", e, 0) for e in range(cfg.E)]).cuda()
    w2 = torch.stack([wl.expert_weight_fp32(cfg, "w2", e, 0) for e in range(cfg.E)]).cuda()
    q13, s13 = moe.fp8_quantize_weights(w13.reshape(-1, cfg.H))
    q2, s2 = moe.fp8_quantize_weights(w2.reshape(-1, cfg.I))
    args = (bf16_to_dev(inp.x), torch.from_numpy(inp.Wr).cuda(), None, q13.reshape(cfg.E, 2 * cfg.I, cfg.H),
            s13.reshape(cfg.E, 2 * cfg.I), q2.reshape(cfg.E, cfg.H, cfg.I), s2.reshape(cfg.E, cfg.H), cfg.k)
    y_n, e_n = _forward(normal, None, fp8=True, args=args)
    y_c, e_c = _forward(checked, None, fp8=True, args=args)
    assert e_n == OK and e_c == OK, (e_n, e_c)
    np.testing.assert_array_equal(y_c, y_n)


def test_checked_build_equals_normal_build_linear(libs):
    normal, checked = libs
    M, N, K = 1500, 256, 1280
    x = wl.draw_activations(3, wl.LINEAR.cfg_id, M, K, max(1, K // 100))
    r = np.random.default_rng(3)
    xb = bf16_to_dev(x)
    w_q = torch.from_numpy(r.integers(-127, 128, (N, K)).astype(np.int8)).cuda()
    s_w = torch.from_numpy((r.random(N) * 1e-3 + 1e-4).astype(np.float32)).cuda()
    outs = []
    for lib in (normal, checked):
        ws = moe.new_workspace(moe.linear_workspace_size(M, N, K))
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert lib.moe_w8a8_linear(xb.data_ptr(), w_q.data_ptr(), s_w.data_ptr(), M, N, K, y.data_ptr(),
                                   ws.data_ptr(), ws.numel(), _stream()) == OK
        assert lib.moe_w8a8_device_error(ws.data_ptr(), _stream()) == OK
        outs.append(bf16_from_dev(y))
    np.testing.assert_array_equal(outs[1], outs[0])


FUSED_SHAPES = {  # T <= 128: the shapes the one-kernel layer takes
    "tiny": TINY,
    "decode": SHAPES["decode"],
    "top8": TINY.replace(T=100, H=256, I=128, E=256, k=8, bias="normal", bias_std=0.5),
}


@pytest.mark.parametrize("name", list(FUSED_SHAPES))
def test_checked_build_equals_normal_build_one_kernel_layer(libs, name):
    normal, checked = libs
    layer = Layer(FUSED_SHAPES[name])
    x, Wr, bias, w13, s13, w2, s2, k = layer.device_args()
    T, H = x.shape
    E, I = w13.shape[0], w13.shape[1] // 2
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    outs = []
    for lib in (normal, checked):
        ws = moe.new_workspace(moe.workspace_size(T, H, I, E, k))
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        assert lib.moe_w8a8_forward_fused(ptr(x), ptr(Wr), ptr(bias), ptr(w13), ptr(s13), ptr(w2), ptr(s2), T, H, I,
                                          E, k, ptr(y), ptr(ws), ws.numel(), _stream(), None) == OK
        assert lib.moe_w8a8_device_error(ws.data_ptr(), _stream()) == OK
        outs.append(bf16_from_dev(y))
    np.testing.assert_array_equal(outs[1], outs[0])
    y_multi, _ = _forward(normal, layer)
    np.testing.assert_array_equal(outs[0], y_multi)


def test_checked_build_reports_a_slot_out_of_range(libs, monkeypatch):
    normal, checked = libs
    layer = Layer(SHAPES["mid"])
    y_clean, _ = _forward(normal, layer)
    monkeypatch.setenv("MOE_INJECT", "bad_slot")
    y_bad, err = _forward(checked, layer)
    assert err == DEVICE
    # token 0 lost its first choice's contribution; every other token is exact
    np.testing.assert_array_equal(y_bad[1:], y_clean[1:])
    monkeypatch.delenv("MOE_INJECT")
    y_again, err = _forward(checked, layer)
    assert err == OK
    np.testing.assert_array_equal(y_again, y_clean)


def test_normal_build_ignores_the_bad_slot_hook(libs, monkeypatch):
    normal, _ = libs
    layer = Layer(SHAPES["mid"])
    y_clean, _ = _forward(normal, layer)
    monkeypatch.setenv("MOE_INJECT", "bad_slot")
    y, err = _forward(normal, layer)
    assert err == OK
    np.testing.assert_array_equal(y, y_clean)
