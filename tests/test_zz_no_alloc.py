"""moe_w8a8_linear_static: the W8A8 linear layer for callers that cannot
allocate device memory (a plugin whose host framework gives it no allocator,
or a serving loop that reserved all device memory for its own pool).  Its
scratch is a static device array inside the library.

Checked through the C ABI:
  * against moe_w8a8_linear, which takes a caller-allocated workspace, on two
    calls in a row with different shapes: bit-identical results, so nothing a
    call leaves in the shared scratch leaks into the next;
  * directly against the oracle on one call (y is exact there: the int32
    accumulators are exact and the bf16 epilogue is one rounding);
  * that repeated calls of several shapes leave the device's free memory
    unchanged, i.e. the entry point allocates nothing;
  * that its error-word query reports a clean state after good calls.

This file is named to be collected last, so that a run that stops at the
first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import _lib
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

OK, SHAPE = 0, -2
SHAPES = ((1, (300, 384, 1280)), (2, (1000, 256, 4096)), (3, (4, 512, 2048)))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    oracle.build()
    return _lib.load()


def _host_inputs(seed, M, N, K):
    x = wl.draw_activations(seed, wl.LINEAR.cfg_id, M, K, max(1, K // 100))
    r = np.random.default_rng(seed)
    w_q = r.integers(-127, 128, (N, K)).astype(np.int8)
    s_w = (r.random(N) * 1e-3 + 1e-4).astype(np.float32)
    return x, w_q, s_w


def _inputs(seed, M, N, K):
    x, w_q, s_w = _host_inputs(seed, M, N, K)
    xb = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    return xb, torch.from_numpy(w_q).cuda(), torch.from_numpy(s_w).cuda()


def _with_workspace(lib, xb, w_q, s_w):
    M, K = xb.shape
    N = w_q.shape[0]
    ws = moe.new_workspace(moe.linear_workspace_size(M, N, K))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert lib.moe_w8a8_linear(xb.data_ptr(), w_q.data_ptr(), s_w.data_ptr(), M, N, K, y.data_ptr(),
                               ws.data_ptr(), ws.numel(), st) == OK
    return y


def _static_into(lib, xb, w_q, s_w, y):
    M, K = xb.shape
    N = w_q.shape[0]
    st = torch.cuda.current_stream().cuda_stream
    assert lib.moe_w8a8_linear_static(xb.data_ptr(), w_q.data_ptr(), s_w.data_ptr(), M, N, K, y.data_ptr(),
                                      st) == OK
    return y


def _static(lib, xb, w_q, s_w):
    y = torch.empty((xb.shape[0], w_q.shape[0]), dtype=torch.bfloat16, device="cuda")
    return _static_into(lib, xb, w_q, s_w, y)


def test_static_scratch_linear_matches_workspace_linear_twice(lib):
    # two calls in a row with different shapes and inputs: the second must
    # not see anything the first left in the shared scratch
    for seed, (M, N, K) in SHAPES:
        xb, w_q, s_w = _inputs(seed, M, N, K)
        y_static = _static(lib, xb, w_q, s_w)
        y_ws = _with_workspace(lib, xb, w_q, s_w)
        torch.cuda.synchronize()
        assert torch.equal(y_static.view(torch.int16), y_ws.view(torch.int16)), (M, N, K)
    assert lib.moe_w8a8_linear_static_error(torch.cuda.current_stream().cuda_stream) == OK


def test_static_scratch_linear_matches_the_oracle(lib):
    M, N, K = 300, 384, 1280
    x, w_q, s_w = _host_inputs(7, M, N, K)
    xb = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    y = _static(lib, xb, torch.from_numpy(w_q).cuda(), torch.from_numpy(s_w).cuda())
    torch.cuda.synchronize()
    y_o = oracle.linear(x, w_q, s_w)
    assert np.array_equal(y.cpu().view(torch.int16).numpy().view(np.uint16), y_o)
    assert lib.moe_w8a8_linear_static_error(torch.cuda.current_stream().cuda_stream) == OK


def test_static_scratch_linear_allocates_nothing(lib):
    cases = [(_inputs(seed, M, N, K), torch.empty((M, N), dtype=torch.bfloat16, device="cuda"))
             for seed, (M, N, K) in SHAPES]
    for (xb, w_q, s_w), y in cases:  # warm-up: every kernel these shapes use is loaded
        _static_into(lib, xb, w_q, s_w, y)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        for (xb, w_q, s_w), y in cases:
            _static_into(lib, xb, w_q, s_w, y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert lib.moe_w8a8_linear_static_error(torch.cuda.current_stream().cuda_stream) == OK


def test_static_scratch_linear_rejects_shapes_beyond_its_capacity(lib):
    # 2048 x 4096 fp16 codes alone need 16 MiB: rejected before any launch
    assert lib.moe_w8a8_linear_static(1 << 20, 1 << 20, 1 << 20, 2048, 256, 4096, 1 << 20, None) == SHAPE
    assert lib.moe_w8a8_linear_static(1 << 20, 1 << 20, 1 << 20, 0, 256, 4096, 1 << 20, None) == OK
