"""The one-kernel layer (moe_w8a8_forward_fused): router, top-k, routing
tables, quantisation, both expert GEMMs, requantisation and combine as the
phases of one cooperative launch.

Its arithmetic is the multi-kernel forward's, so the checks are bit for bit
against moe_w8a8_forward on the same inputs and workspace: y and every
intermediate of the debug dump (routing, slot maps, scales, codes, the raw
int32 accumulators of both GEMMs, h, o).  y is also compared with the oracle
directly.  Shapes: one token, a few tokens per expert, the 128-token maximum,
a single expert, 256 experts with top-8 and a router bias (most experts
empty), rows of h longer than 8192, the decode layer at full size, and the
256-expert layer's shape at 128 tokens.  Then
the failure path: with MOE_INJECT=stall one CTA skips a barrier arrival, the
2 ms wait limit runs out everywhere, MOE_ERR_DEVICE_TIMEOUT is reported, and
the next calls on the same workspace are exact again."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl
from gpu_helpers import Layer, assert_y_close, bf16_from_dev

pytestmark = pytest.mark.gpu

OK, TIMEOUT = 0, -5
TINY = wl.CONFIGS["tiny"]
SHAPES = {
    "tiny": TINY,
    "one_token": TINY.replace(T=1, H=512, I=256, E=8, k=2),
    "decode_like": TINY.replace(T=64, H=1024, I=512, E=16, k=2),
    "max_tokens": TINY.replace(T=128, H=512, I=384, E=64, k=4),
    "one_expert": TINY.replace(T=32, H=256, I=128, E=1, k=1),
    "top8_bias": TINY.replace(T=100, H=256, I=128, E=256, k=8, bias="normal", bias_std=0.5),
    "long_rows": TINY.replace(T=8, H=256, I=8320, E=2, k=1),  # rows of h longer than 8192
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    oracle.build()
    moe._lib.load()


def _both(layer, fields=None):
    cfg = layer.cfg
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y_p, d_p = moe.forward_debug(*layer.device_args(), fields=fields, workspace=ws)
    y_f, d_f = moe.forward_fused(*layer.device_args(), fields=fields, workspace=ws)
    assert moe.device_error(ws) == OK
    return bf16_from_dev(y_p), d_p, bf16_from_dev(y_f), d_f


@pytest.mark.parametrize("name", list(SHAPES))
def test_fused_equals_the_multi_kernel_forward_bit_for_bit(name):
    cfg = SHAPES[name]
    assert moe.fused_supported(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    layer = Layer(cfg)
    y_p, d_p, y_f, d_f = _both(layer)
    np.testing.assert_array_equal(y_f, y_p)
    for field in d_p:
        a, b = d_f[field].cpu().numpy(), d_p[field].cpu().numpy()
        np.testing.assert_array_equal(a.view(np.uint8), b.view(np.uint8), err_msg=field)
    assert_y_close(y_f, layer.oracle())


def test_fused_is_deterministic_and_shares_the_workspace():
    layer = Layer(SHAPES["decode_like"], seed=3)
    cfg = layer.cfg
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    ys = []
    for fused in (True, False, True, True):
        fn = moe.forward_fused if fused else moe.forward
        ys.append(bf16_from_dev(fn(*layer.device_args(), workspace=ws)))
        assert moe.device_error(ws) == OK
    for y in ys[1:]:
        np.testing.assert_array_equal(y, ys[0])


def test_fused_decode_layer_at_full_size():
    """T = 64, H = 4096, I = 1536, E = 64, top-2 (random int8 weights)."""
    cfg = wl.CONFIGS["decode"]
    inp = wl.make_moe_inputs(cfg, 0)
    g = torch.Generator().manual_seed(7)
    w13 = torch.randint(-127, 128, (cfg.E, 2 * cfg.I, cfg.H), dtype=torch.int8, generator=g)
    w2 = torch.randint(-127, 128, (cfg.E, cfg.H, cfg.I), dtype=torch.int8, generator=g)
    s13 = torch.rand((cfg.E, 2 * cfg.I), generator=g) * 1e-3 + 1e-4
    s2 = torch.rand((cfg.E, cfg.H), generator=g) * 1e-3 + 1e-4
    layer = Layer(cfg, weights=(w13.numpy(), s13.numpy(), w2.numpy(), s2.numpy()))
    fields = ("topk_ids", "offsets", "slot_token", "s_x", "h", "s_h", "q_h", "o")
    y_p, d_p, y_f, d_f = _both(layer, fields)
    np.testing.assert_array_equal(y_f, y_p)
    for field in fields:
        np.testing.assert_array_equal(d_f[field].cpu().numpy(), d_p[field].cpu().numpy(), err_msg=field)
    sel = np.arange(0, cfg.T, 8)  # the oracle on every 8th token
    y_o = oracle.moe_forward(inp.x[sel], inp.Wr, inp.bias, layer.w13_q, layer.s13, layer.w2_q, layer.s2, cfg.k)
    assert_y_close(y_f[sel], y_o)


def test_fused_wide_layer_at_128_tokens():
    """T = 128, H = 7168, I = 2048, E = 256, top-8 with a router bias (the
    256-expert layer's shape at the one-kernel layer's token limit; random
    int8 weights drawn on the device): bit for bit the multi-kernel layer."""
    cfg = wl.CONFIGS["wide"].replace(T=128)
    inp = wl.make_moe_inputs(cfg, 0)
    g = torch.Generator(device="cuda").manual_seed(11)
    w13 = torch.randint(-127, 128, (cfg.E, 2 * cfg.I, cfg.H), dtype=torch.int8, generator=g, device="cuda")
    w2 = torch.randint(-127, 128, (cfg.E, cfg.H, cfg.I), dtype=torch.int8, generator=g, device="cuda")
    s13 = torch.rand((cfg.E, 2 * cfg.I), generator=g, device="cuda") * 1e-3 + 1e-4
    s2 = torch.rand((cfg.E, cfg.H), generator=g, device="cuda") * 1e-3 + 1e-4
    x = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).view(torch.bfloat16).cuda()
    bias = None if inp.bias is None else torch.from_numpy(inp.bias).cuda()
    args = (x, torch.from_numpy(inp.Wr).cuda(), bias, w13, s13, w2, s2, cfg.k)
    assert moe.fused_supported(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    fields = ("topk_ids", "offsets", "slot_token", "s_h", "q_h")
    y_p, d_p = moe.forward_debug(*args, fields=fields, workspace=ws)
    y_f, d_f = moe.forward_fused(*args, fields=fields, workspace=ws)
    assert moe.device_error(ws) == OK
    np.testing.assert_array_equal(bf16_from_dev(y_f), bf16_from_dev(y_p))
    for field in fields:
        np.testing.assert_array_equal(d_f[field].cpu().numpy(), d_p[field].cpu().numpy(), err_msg=field)


def test_forced_timeout_in_the_fused_layer_then_exact_again(monkeypatch):
    layer = Layer(SHAPES["decode_like"])
    cfg = layer.cfg
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y_ref = bf16_from_dev(moe.forward(*layer.device_args(), workspace=ws))
    monkeypatch.setenv("MOE_INJECT", "stall")
    moe.set_wait_timeout_ns(2_000_000)
    try:
        moe.forward_fused(*layer.device_args(), workspace=ws)
        assert moe.device_error(ws) == TIMEOUT
    finally:
        monkeypatch.delenv("MOE_INJECT", raising=False)
        moe.set_wait_timeout_ns(0)
    assert moe.device_error(ws) == OK  # read and cleared
    for _ in range(2):  # the barrier words were left clear: exact again
        y = bf16_from_dev(moe.forward_fused(*layer.device_args(), workspace=ws))
        assert moe.device_error(ws) == OK
        np.testing.assert_array_equal(y, y_ref)
