"""Failure detection on the GPU, without faulting it.

* Forced timeouts: MOE_INJECT=stall makes the producer of every grouped
  GEMM launch first wait, with the library's own bounded wait, on a barrier
  that nothing completes (in a CTA pair, the even CTA's producer only).  With
  the wait limit set to 2 ms the wait runs out: the kernel records
  MOE_ERR_DEVICE_TIMEOUT in the workspace's error word, every role of the CTA
  (and of its pair peer, through the peer abort flag) gives up, the copies in
  flight are drained, tensor memory is freed and the kernel returns; nothing
  hangs and nothing traps.  The next call without the hook must be exact
  again.  Covered: the one-CTA INT8 GEMM, the CTA-pair INT8 GEMM, whole MoE
  forwards on both, and the FP8 layer's one-CTA and CTA-pair GEMMs.
  (A short limit alone does not force a timeout: mbarrier.try_wait suspends
  in hardware until the phase completes or a time limit passes, so waits of
  microseconds end inside the first polls.)
* A NaN in the activations (outside the layer's contract) makes every
  router logit of that token NaN: the top-k ranks NaN as -inf, so the
  routing stays valid, and the router records MOE_ERR_DEVICE.
* An injected launch failure (MOE_INJECT=launch_fail) returns MOE_ERR_CUDA
  without launching anything, and leaves the library usable.
"""
import numpy as np
import pytest
import torch

import oracle
import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import _lib
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl
from gpu_helpers import Layer, assert_y_close, bf16_from_dev, bf16_to_dev, gemm_path

pytestmark = pytest.mark.gpu

OK, CUDA, TIMEOUT, DEVICE = 0, -4, -5, -7
TINY = wl.CONFIGS["tiny"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    oracle.build()
    moe._lib.load()


class _Stall:
    """MOE_INJECT=stall and a 2 ms wait limit inside the block; neither after."""

    def __init__(self, monkeypatch):
        self.mp = monkeypatch

    def __enter__(self):
        self.mp.setenv("MOE_INJECT", "stall")
        moe.set_wait_timeout_ns(2_000_000)

    def __exit__(self, *exc):
        self.mp.delenv("MOE_INJECT", raising=False)
        moe.set_wait_timeout_ns(0)


def _linear_case(M, N, K, seed):
    x = wl.draw_activations(seed, wl.LINEAR.cfg_id, M, K, max(1, K // 100))
    r = np.random.default_rng(seed)
    w_q = r.integers(-127, 128, (N, K)).astype(np.int8)
    s_w = (r.random(N) * 1e-3 + 1e-4).astype(np.float32)
    return x, w_q, s_w


@pytest.mark.parametrize("path,shape", [("mid", (512, 512, 2048)), ("pair", (1024, 512, 2048))])
def test_forced_timeout_in_the_linear_gemm_then_exact_again(monkeypatch, path, shape):
    M, N, K = shape
    x, w_q, s_w = _linear_case(M, N, K, 11)
    dx, dw, ds = bf16_to_dev(x), torch.from_numpy(w_q).cuda(), torch.from_numpy(s_w).cuda()
    ws = moe.new_workspace(moe.linear_workspace_size(M, N, K))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with gemm_path(path):
        with _Stall(monkeypatch):
            moe.linear(dx, dw, ds, workspace=ws, out=y)
            assert moe.device_error(ws) == TIMEOUT
        assert moe.device_error(ws) == OK  # read and cleared
        for _ in range(2):  # exact again, and the error word stays clear
            y.zero_()
            moe.linear(dx, dw, ds, workspace=ws, out=y)
            assert moe.device_error(ws) == OK
            np.testing.assert_array_equal(bf16_from_dev(y), oracle.linear(x, w_q, s_w))


@pytest.mark.parametrize("path", ["auto", "mid"])  # auto: both expert GEMMs on CTA pairs
def test_forced_timeout_in_the_moe_forward_then_exact_again(monkeypatch, path):
    cfg = TINY.replace(T=600, H=512, I=384, E=4, k=2)
    layer = Layer(cfg)
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    y_o = layer.oracle()
    with gemm_path(path):
        with _Stall(monkeypatch):
            moe.forward(*layer.device_args(), workspace=ws, out=y)
            assert moe.device_error(ws) == TIMEOUT
        for _ in range(2):
            moe.forward(*layer.device_args(), workspace=ws, out=y)
            assert moe.device_error(ws) == OK
            assert_y_close(bf16_from_dev(y), y_o)


@pytest.mark.parametrize("name,cfg", [
    ("pair", TINY.replace(T=1000, H=512, I=256, E=4, k=2)),           # FP8 CTA-pair GEMMs
    ("one_cta", TINY.replace(T=40, H=512, I=256, E=32, k=2)),         # FP8 one-CTA GEMMs
])
def test_forced_timeout_in_the_fp8_gemms_then_clean_again(monkeypatch, name, cfg):
    inp = wl.make_moe_inputs(cfg, 0)
    w13 = np.stack([wl.expert_weight_fp32(cfg, "w13", e, 0).numpy() for e in range(cfg.E)])
    w2 = np.stack([wl.expert_weight_fp32(cfg, "w2", e, 0).numpy() for e in range(cfg.E)])
    q13, s13 = oracle.quantize_rows_fp8(w13.reshape(-1, cfg.H))
    q2, s2 = oracle.quantize_rows_fp8(w2.reshape(-1, cfg.I))
    q13, s13 = q13.reshape(cfg.E, 2 * cfg.I, cfg.H), s13.reshape(cfg.E, 2 * cfg.I)
    q2, s2 = q2.reshape(cfg.E, cfg.H, cfg.I), s2.reshape(cfg.E, cfg.H)
    args = (bf16_to_dev(inp.x), torch.from_numpy(inp.Wr).cuda(), None, torch.from_numpy(q13).cuda(),
            torch.from_numpy(s13).cuda(), torch.from_numpy(q2).cuda(), torch.from_numpy(s2).cuda(), cfg.k)
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    with _Stall(monkeypatch):
        moe.fp8_forward(*args, workspace=ws, out=y)
        assert moe.device_error(ws) == TIMEOUT
    y_o = oracle.moe_forward_fp8(inp.x, inp.Wr, None, q13, s13, q2, s2, cfg.k)
    moe.fp8_forward(*args, workspace=ws, out=y)
    assert moe.device_error(ws) == OK
    assert_y_close(bf16_from_dev(y), y_o)


@pytest.mark.parametrize("T", [100, 300])  # the few-token router, the tensor-core router
def test_nan_activation_is_reported_and_routing_stays_valid(T):
    cfg = TINY.replace(T=T, H=512, I=256, E=8, k=2)
    layer = Layer(cfg)
    bad = T // 3
    x = layer.x.copy()
    x[bad, 5] = 0x7FC0  # a bf16 quiet NaN
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y, d = moe.forward_debug(bf16_to_dev(x), *layer.device_args()[1:], workspace=ws,
                             fields=("topk_ids", "offsets", "slot_of"))
    assert moe.device_error(ws) == DEVICE
    ids = d["topk_ids"].cpu().numpy()
    assert ((ids >= 0) & (ids < cfg.E)).all()
    assert list(ids[bad]) == [0, 1]  # every logit ranks as -inf: ties to the lower index
    off = d["offsets"].cpu().numpy()
    assert off[0] == 0 and off[-1] == cfg.S and (np.diff(off) >= 0).all()
    assert sorted(d["slot_of"].cpu().numpy().ravel().tolist()) == list(range(cfg.S))
    # the other tokens are untouched: as the oracle computes them without the bad row
    keep = np.arange(T) != bad
    y_o = oracle.moe_forward(layer.x[keep], layer.Wr, layer.bias, layer.w13_q, layer.s13, layer.w2_q, layer.s2,
                             cfg.k)
    assert_y_close(bf16_from_dev(y)[keep], y_o)
    # the next call on clean input is clean
    moe.forward(*layer.device_args(), workspace=ws)
    assert moe.device_error(ws) == OK


def test_injected_launch_failure_launches_nothing(monkeypatch):
    cfg = TINY
    layer = Layer(cfg)
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    lib = _lib.load()
    torch.cuda.synchronize()
    before = lib.moe_w8a8_launch_count()
    monkeypatch.setenv("MOE_INJECT", "launch_fail")
    with pytest.raises(_lib.MoeError) as e:
        moe.forward(*layer.device_args(), workspace=ws)
    assert e.value.status == CUDA
    assert lib.moe_w8a8_launch_count() == before
    monkeypatch.delenv("MOE_INJECT")
    y = moe.forward(*layer.device_args(), workspace=ws)
    assert moe.device_error(ws) == OK
    assert_y_close(bf16_from_dev(y), layer.oracle())
