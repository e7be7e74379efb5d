"""The host-resident entry points (moe_w8a8_forward_host and its FP8 form):
x copied in and y copied out inside the call, in token chunks overlapped
with compute on a second stream.  Each chunk is a whole forward of its
tokens, so the result must equal the device entry point run on each chunk,
bit for bit, and with one chunk the device entry point on the whole batch."""
import numpy as np
import pytest
import torch

import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl
from gpu_helpers import bf16_to_dev

pytestmark = pytest.mark.gpu

CFG = wl.CONFIGS["tiny"].replace(T=1000, H=512, I=256, E=8, k=2, bias="normal", bias_std=0.5)


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    moe._lib.load()


def _weights(fmt):
    quant = moe.fp8_quantize_weights if fmt == "fp8" else moe.quantize_weights
    w13 = [quant(wl.expert_weight_fp32(CFG, "w13", e, 0, device="cuda")) for e in range(CFG.E)]
    w2 = [quant(wl.expert_weight_fp32(CFG, "w2", e, 0, device="cuda")) for e in range(CFG.E)]
    return (torch.stack([q for q, _ in w13]), torch.stack([s for _, s in w13]),
            torch.stack([q for q, _ in w2]), torch.stack([s for _, s in w2]))


def _args(fmt):
    inp = wl.make_moe_inputs(CFG, 0)
    x_dev = bf16_to_dev(inp.x)
    Wr = torch.from_numpy(inp.Wr).cuda()
    bias = torch.from_numpy(inp.bias).cuda()
    return x_dev, (Wr, bias, *_weights(fmt), CFG.k)


def _per_chunk(fwd, x_dev, rest, n):
    T = x_dev.shape[0]
    outs = []
    for c in range(n):
        t0, t1 = T * c // n, T * (c + 1) // n
        outs.append(fwd(x_dev[t0:t1].contiguous(), *rest))
    return torch.cat(outs)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
@pytest.mark.parametrize("chunks", [1, 2, 3])
@pytest.mark.parametrize("two_streams", [True, False])
def test_forward_host_equals_device_forward_per_chunk(fmt, chunks, two_streams):
    fwd = moe.fp8_forward if fmt == "fp8" else moe.forward
    fwd_host = moe.fp8_forward_host if fmt == "fp8" else moe.forward_host
    x_dev, rest = _args(fmt)
    x_host = x_dev.cpu().pin_memory()
    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream() if two_streams else None
    y_host = torch.full(x_host.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    out = fwd_host(x_host, *rest, y_host=y_host, stream=stream, copy_stream=copy_stream, chunks=chunks)
    assert out.data_ptr() == y_host.data_ptr()
    stream.synchronize()
    ref = _per_chunk(fwd, x_dev, rest, chunks).cpu()
    torch.cuda.synchronize()
    assert torch.equal(y_host.view(torch.int16), ref.view(torch.int16))
    if chunks == 1:
        assert torch.equal(y_host.view(torch.int16), fwd(x_dev, *rest).cpu().view(torch.int16))


def test_forward_host_chooses_one_chunk_for_small_batches_and_repeats():
    x_dev, rest = _args("int8")
    assert moe.host_chunks(*x_dev.shape, CFG.I, CFG.E) == 1
    x_host = x_dev.cpu().pin_memory()
    copy_stream = torch.cuda.Stream()
    ws = moe.new_workspace(moe.workspace_size(CFG.T, CFG.H, CFG.I, CFG.E, CFG.k))
    y1 = moe.forward_host(x_host, *rest, workspace=ws, copy_stream=copy_stream)
    torch.cuda.current_stream().synchronize()  # y1 is complete once the compute stream is
    y1 = y1.clone()
    y2 = moe.forward_host(x_host, *rest, workspace=ws, copy_stream=copy_stream)
    torch.cuda.synchronize()
    assert moe.device_error(ws) == 0
    ref = moe.forward(x_dev, *rest).cpu()
    assert torch.equal(y1.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), ref.view(torch.int16))
