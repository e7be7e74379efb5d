"""Parity at the benchmark's full sizes (decode, prefill and wide MoE layers,
the 4096^3 linear layer, and the FP8 (E4M3) and SmoothQuant-folded variants
of the decode and prefill layers), in the launch configuration bench.py times: inputs
resident on the device, expert weights drawn in fp32 on the device and
quantised by the library, one plain forward.

The oracle cannot run these layers whole in a test's time, so it checks
sampled tokens one by one, and the full-size results are checked against
properties that hold at any size:

* every routing array is consistent (expert offsets are the prefix sums of
  the top-k counts, slots are a permutation, each slot lies in its expert's
  range, a token's experts are distinct);
* for the sampled tokens the router, the codes, both GEMMs' int32
  accumulators, the requantisation and the output epilogue are bit-exact
  against the oracle on the stage's input; h is within H_RTOL (expf);
* the sampled rows of y agree with the oracle's own end-to-end computation
  (from the oracle's h) within the layer's tolerance;
* the library's int8 weights of every sampled expert equal the oracle's
  quantisation of the same fp32 draws, so the oracle's weights are its own.

The FP8 layer is checked the same way, except that its fp32 accumulators
are bounded against the exact dot products of the E4M3 codes instead of
compared bit for bit.

Besides, y of every token of the decode and prefill layers (INT8), of every
token of the FP8 decode layer and 2048 tokens of the FP8 prefill layer, and of
256 tokens of the 256-expert layer is compared with the oracle's own
end-to-end forward on the same inputs, within the layer's tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl
from gpu_helpers import H_RTOL, TOPK_W_ATOL, assert_y_close, bf16_from_dev, bf16_to_dev

pytestmark = pytest.mark.gpu

# sampled tokens per layer (each brings up to k experts the oracle quantises)
SAMPLE = {"decode": 16, "prefill": 16, "wide": 4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    moe._lib.load()


def _device_weights(cfg, seed):
    w13_q = torch.empty((cfg.E, 2 * cfg.I, cfg.H), dtype=torch.int8, device="cuda")
    w13_s = torch.empty((cfg.E, 2 * cfg.I), dtype=torch.float32, device="cuda")
    w2_q = torch.empty((cfg.E, cfg.H, cfg.I), dtype=torch.int8, device="cuda")
    w2_s = torch.empty((cfg.E, cfg.H), dtype=torch.float32, device="cuda")
    for e in range(cfg.E):
        q, s = moe.quantize_weights(wl.expert_weight_fp32(cfg, "w13", e, seed, device="cuda"))
        w13_q[e].copy_(q)
        w13_s[e].copy_(s)
        q, s = moe.quantize_weights(wl.expert_weight_fp32(cfg, "w2", e, seed, device="cuda"))
        w2_q[e].copy_(q)
        w2_s[e].copy_(s)
    return w13_q, w13_s, w2_q, w2_s


def _oracle_expert(cfg, which, e, seed):
    """The oracle's quantisation of the same fp32 draws (drawn where the
    library's were, then copied to the host)."""
    return oracle.quantize_rows(wl.expert_weight_fp32(cfg, which, e, seed, device="cuda").cpu().numpy())


def _check_routing_arrays(cfg, ids, offsets, slot_of, slot_token):
    T, k, E = cfg.T, cfg.k, cfg.E
    S = T * k
    counts = np.bincount(ids.ravel(), minlength=E)
    assert offsets[0] == 0 and offsets[-1] == S
    np.testing.assert_array_equal(np.diff(offsets), counts)
    np.testing.assert_array_equal(np.sort(slot_of.ravel()), np.arange(S))
    np.testing.assert_array_equal(slot_token[slot_of], np.repeat(np.arange(T)[:, None], k, axis=1))
    expert_of_slot = np.searchsorted(offsets, slot_of, side="right") - 1
    np.testing.assert_array_equal(expert_of_slot, ids)
    assert (np.diff(np.sort(ids, axis=1), axis=1) > 0).all()  # distinct experts per token


@pytest.mark.parametrize("name", ["decode", "prefill", "wide"])
def test_full_size_layer_sampled_against_oracle(name):
    cfg = wl.CONFIGS[name]
    seed = 0
    inp = wl.make_moe_inputs(cfg, seed)
    x = bf16_to_dev(inp.x)
    Wr = torch.from_numpy(inp.Wr).cuda()
    bias = None if inp.bias is None else torch.from_numpy(inp.bias).cuda()
    w13_q, w13_s, w2_q, w2_s = _device_weights(cfg, seed)
    args = (x, Wr, bias, w13_q, w13_s, w2_q, w2_s, cfg.k)

    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y_plain = moe.forward(*args, workspace=ws)
    assert moe.device_error(ws) == 0
    y_dbg, dev = moe.forward_debug(*args, workspace=ws)
    assert moe.device_error(ws) == 0
    assert torch.equal(y_plain.view(torch.int16), y_dbg.view(torch.int16))

    ids = dev["topk_ids"].cpu().numpy()
    topk_w = dev["topk_w"].cpu().numpy()
    offsets = dev["offsets"].cpu().numpy()
    slot_of = dev["slot_of"].cpu().numpy()
    slot_token = dev["slot_token"].cpu().numpy()
    _check_routing_arrays(cfg, ids, offsets, slot_of, slot_token)

    tok = np.sort(np.random.default_rng(7).choice(cfg.T, SAMPLE[name], replace=False))
    ids_ref, w_ref, _ = oracle.router(inp.x[tok], inp.Wr, inp.bias, cfg.k)
    np.testing.assert_array_equal(ids[tok], ids_ref)
    np.testing.assert_allclose(topk_w[tok], w_ref, rtol=0, atol=TOPK_W_ATOL)
    q_ref, s_ref = oracle.quantize_rows_bf16(inp.x[tok])
    np.testing.assert_array_equal(dev["q_x"][tok].cpu().numpy(), q_ref)
    np.testing.assert_array_equal(dev["s_x"][tok].cpu().numpy(), s_ref)

    ref_w = {}
    for e in sorted(set(ids_ref.ravel().tolist())):
        ref_w[e] = (_oracle_expert(cfg, "w13", e, seed), _oracle_expert(cfg, "w2", e, seed))
        np.testing.assert_array_equal(w13_q[e].cpu().numpy(), ref_w[e][0][0])
        np.testing.assert_array_equal(w13_s[e].cpu().numpy(), ref_w[e][0][1])
        np.testing.assert_array_equal(w2_q[e].cpu().numpy(), ref_w[e][1][0])
        np.testing.assert_array_equal(w2_s[e].cpu().numpy(), ref_w[e][1][1])

    y_gpu = bf16_from_dev(y_dbg)[tok]
    y_ref = np.empty_like(y_gpu)
    for i, t in enumerate(tok):
        slots = slot_of[t]
        o_gpu = dev["o"][torch.from_numpy(slots).long().cuda()].cpu().numpy()
        o_own = np.empty_like(o_gpu)
        for j, s in enumerate(slots):
            (w13r, s13r), (w2r, s2r) = ref_w[int(ids_ref[i, j])]
            acc1 = oracle.gemm_s8(q_ref[i:i + 1], w13r)
            np.testing.assert_array_equal(dev["acc1"][s].cpu().numpy(), acc1[0])
            h_ref = oracle.epilogue_gate_up(acc1, s_ref[i:i + 1], s13r)
            h_gpu = dev["h"][s].cpu().numpy()
            np.testing.assert_allclose(h_gpu, h_ref[0], rtol=H_RTOL, atol=1e-30)
            # requantisation, GEMM2 and its epilogue on the GPU's own h: exact
            qh, sh = oracle.quantize_rows(h_gpu[None])
            np.testing.assert_array_equal(dev["q_h"][s].cpu().numpy(), qh[0])
            assert dev["s_h"][s].item() == sh[0]
            acc2 = oracle.gemm_s8(qh, w2r)
            np.testing.assert_array_equal(dev["acc2"][s].cpu().numpy(), acc2[0])
            np.testing.assert_array_equal(o_gpu[j], oracle.epilogue_scale(acc2, sh, s2r)[0])
            # the oracle's own path from its own h
            qh_o, sh_o = oracle.quantize_rows(h_ref)
            o_own[j] = oracle.epilogue_scale(oracle.gemm_s8(qh_o, w2r), sh_o, s2r)[0]
        # combine of the GPU's own o rows: exact; of the oracle's: the layer tolerance
        one = np.arange(cfg.k, dtype=np.int32)[None]
        np.testing.assert_array_equal(y_gpu[i], oracle.combine(o_gpu, one, topk_w[t][None])[0])
        y_ref[i] = oracle.combine(o_own, one, w_ref[i][None])[0]
    assert_y_close(y_gpu, y_ref)


def test_full_size_linear_sampled_against_oracle():
    cfg = wl.LINEAR
    seed = 0
    x_bits = wl.linear_activations(cfg, seed)
    w32 = wl.expert_weight_fp32(cfg, "linear", 0, seed, device="cuda")
    w_q, w_s = moe.quantize_weights(w32)
    y = moe.linear(bf16_to_dev(x_bits), w_q, w_s)
    torch.cuda.synchronize()
    wq_ref, ws_ref = oracle.quantize_rows(w32.cpu().numpy())
    np.testing.assert_array_equal(w_q.cpu().numpy(), wq_ref)
    np.testing.assert_array_equal(w_s.cpu().numpy(), ws_ref)
    rows = np.sort(np.random.default_rng(8).choice(cfg.M, 16, replace=False))
    np.testing.assert_array_equal(bf16_from_dev(y)[rows], oracle.linear(x_bits[rows], wq_ref, ws_ref))


# ---- the FP8 (E4M3) layer at the benchmark's sizes -------------------------

# fp32 accumulation of exact E4M3 products (the bound of the FP8 parity tests)
FP8_ACC_REL = 2.0 ** -16


def _fp8_device_weights(cfg, seed):
    code = torch.uint8
    w13_q = torch.empty((cfg.E, 2 * cfg.I, cfg.H), dtype=code, device="cuda")
    w13_s = torch.empty((cfg.E, 2 * cfg.I), dtype=torch.float32, device="cuda")
    w2_q = torch.empty((cfg.E, cfg.H, cfg.I), dtype=code, device="cuda")
    w2_s = torch.empty((cfg.E, cfg.H), dtype=torch.float32, device="cuda")
    for e in range(cfg.E):
        q, s = moe.fp8_quantize_weights(wl.expert_weight_fp32(cfg, "w13", e, seed, device="cuda"))
        w13_q[e].copy_(q)
        w13_s[e].copy_(s)
        q, s = moe.fp8_quantize_weights(wl.expert_weight_fp32(cfg, "w2", e, seed, device="cuda"))
        w2_q[e].copy_(q)
        w2_s[e].copy_(s)
    return w13_q, w13_s, w2_q, w2_s


def _assert_fp8_acc_close(acc, a_codes, w_codes):
    """acc within FP8_ACC_REL * sum |a_k w_k| of the exact dot products."""
    A = oracle.e4m3_decode(a_codes).astype(np.float64)
    W = oracle.e4m3_decode(w_codes).astype(np.float64)
    exact = A @ W.T  # exact: products are multiples of 2^-18 below 2^18
    mag = np.abs(A) @ np.abs(W).T
    err = np.abs(acc.astype(np.float64) - exact)
    assert (err <= FP8_ACC_REL * mag).all(), float((err / np.maximum(mag, 1e-300)).max())


@pytest.mark.parametrize("name", ["decode", "prefill", "wide"])
def test_full_size_fp8_layer_sampled_against_oracle(name):
    cfg = wl.CONFIGS[name]
    seed = 0
    inp = wl.make_moe_inputs(cfg, seed)
    x = bf16_to_dev(inp.x)
    Wr = torch.from_numpy(inp.Wr).cuda()
    bias = None if inp.bias is None else torch.from_numpy(inp.bias).cuda()
    w13_q, w13_s, w2_q, w2_s = _fp8_device_weights(cfg, seed)
    args = (x, Wr, bias, w13_q, w13_s, w2_q, w2_s, cfg.k)

    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y_plain = moe.fp8_forward(*args, workspace=ws)
    assert moe.device_error(ws) == 0
    y_dbg, dev = moe.fp8_forward_debug(*args, workspace=ws)
    assert moe.device_error(ws) == 0
    assert torch.equal(y_plain.view(torch.int16), y_dbg.view(torch.int16))

    ids = dev["topk_ids"].cpu().numpy()
    topk_w = dev["topk_w"].cpu().numpy()
    offsets = dev["offsets"].cpu().numpy()
    slot_of = dev["slot_of"].cpu().numpy()
    slot_token = dev["slot_token"].cpu().numpy()
    _check_routing_arrays(cfg, ids, offsets, slot_of, slot_token)

    tok = np.sort(np.random.default_rng(9).choice(cfg.T, SAMPLE[name], replace=False))
    ids_ref, w_ref, _ = oracle.router(inp.x[tok], inp.Wr, inp.bias, cfg.k)
    np.testing.assert_array_equal(ids[tok], ids_ref)
    np.testing.assert_allclose(topk_w[tok], w_ref, rtol=0, atol=TOPK_W_ATOL)
    q_ref, s_ref = oracle.quantize_rows_bf16_fp8(inp.x[tok])
    np.testing.assert_array_equal(dev["q_x"][tok].cpu().numpy(), q_ref)
    np.testing.assert_array_equal(dev["s_x"][tok].cpu().numpy(), s_ref)

    ref_w = {}
    for e in sorted(set(ids_ref.ravel().tolist())):
        w13 = wl.expert_weight_fp32(cfg, "w13", e, seed, device="cuda").cpu().numpy()
        w2 = wl.expert_weight_fp32(cfg, "w2", e, seed, device="cuda").cpu().numpy()
        ref_w[e] = (oracle.quantize_rows_fp8(w13), oracle.quantize_rows_fp8(w2))
        np.testing.assert_array_equal(w13_q[e].cpu().numpy(), ref_w[e][0][0])
        np.testing.assert_array_equal(w13_s[e].cpu().numpy(), ref_w[e][0][1])
        np.testing.assert_array_equal(w2_q[e].cpu().numpy(), ref_w[e][1][0])
        np.testing.assert_array_equal(w2_s[e].cpu().numpy(), ref_w[e][1][1])

    y_gpu = bf16_from_dev(y_dbg)[tok]
    y_ref = np.empty_like(y_gpu)
    for i, t in enumerate(tok):
        slots = slot_of[t]
        o_gpu = dev["o"][torch.from_numpy(slots).long().cuda()].cpu().numpy()
        o_own = np.empty_like(o_gpu)
        for j, s in enumerate(slots):
            (w13r, s13r), (w2r, s2r) = ref_w[int(ids_ref[i, j])]
            # GEMM1: within the fp32 accumulation bound of the exact dot products
            acc1 = dev["acc1"][s].cpu().numpy()[None]
            _assert_fp8_acc_close(acc1, q_ref[i:i + 1], w13r)
            # gate/up epilogue of the GPU's own accumulators: differs only through expf
            h_gpu = dev["h"][s].cpu().numpy()
            np.testing.assert_allclose(h_gpu, oracle.epilogue_gate_up_f32(acc1, s_ref[i:i + 1], s13r)[0],
                                       rtol=H_RTOL, atol=1e-30)
            # requantisation of the GPU's own h: exact; GEMM2 within the bound; its epilogue exact
            qh, sh = oracle.quantize_rows_fp8(h_gpu[None])
            np.testing.assert_array_equal(dev["q_h"][s].cpu().numpy(), qh[0])
            assert dev["s_h"][s].item() == sh[0]
            acc2 = dev["acc2"][s].cpu().numpy()[None]
            _assert_fp8_acc_close(acc2, qh, w2r)
            np.testing.assert_array_equal(o_gpu[j], oracle.epilogue_scale_f32(acc2, sh, s2r)[0])
            # the oracle's own path: exact sums, its own h
            h_own = oracle.epilogue_gate_up_f32(oracle.gemm_fp8(q_ref[i:i + 1], w13r), s_ref[i:i + 1], s13r)
            qh_o, sh_o = oracle.quantize_rows_fp8(h_own)
            o_own[j] = oracle.epilogue_scale_f32(oracle.gemm_fp8(qh_o, w2r), sh_o, s2r)[0]
        # combine of the GPU's own o rows: exact; of the oracle's: the layer tolerance
        one = np.arange(cfg.k, dtype=np.int32)[None]
        np.testing.assert_array_equal(y_gpu[i], oracle.combine(o_gpu, one, topk_w[t][None])[0])
        y_ref[i] = oracle.combine(o_own, one, w_ref[i][None])[0]
    assert_y_close(y_gpu, y_ref)


# ---- the SmoothQuant-folded layer at the benchmark's sizes ------------------

@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_full_size_smoothed_layer_sampled_against_oracle(name):
    cfg = wl.CONFIGS[name]
    seed = 0
    inp = wl.make_moe_inputs(cfg, seed)
    smooth = wl.smoothing_factors(cfg, seed)
    sm_dev = torch.from_numpy(smooth).cuda()
    w13_q = torch.empty((cfg.E, 2 * cfg.I, cfg.H), dtype=torch.int8, device="cuda")
    w13_s = torch.empty((cfg.E, 2 * cfg.I), dtype=torch.float32, device="cuda")
    w2_q = torch.empty((cfg.E, cfg.H, cfg.I), dtype=torch.int8, device="cuda")
    w2_s = torch.empty((cfg.E, cfg.H), dtype=torch.float32, device="cuda")
    for e in range(cfg.E):
        q, s = moe.quantize_weights_smoothed(wl.expert_weight_fp32(cfg, "w13", e, seed, device="cuda"), sm_dev[e])
        w13_q[e].copy_(q)
        w13_s[e].copy_(s)
        q, s = moe.quantize_weights(wl.expert_weight_fp32(cfg, "w2", e, seed, device="cuda"))
        w2_q[e].copy_(q)
        w2_s[e].copy_(s)
    x = bf16_to_dev(inp.x)
    Wr = torch.from_numpy(inp.Wr).cuda()
    bias = None if inp.bias is None else torch.from_numpy(inp.bias).cuda()
    args = (x, Wr, bias, sm_dev, w13_q, w13_s, w2_q, w2_s, cfg.k)
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y_plain = moe.forward_smooth(*args, workspace=ws)
    assert moe.device_error(ws) == 0
    names = ("topk_ids", "topk_w", "offsets", "slot_of", "slot_token", "s_slot", "q_slot", "acc1", "h", "s_h", "q_h",
             "acc2", "o")
    y_dbg, dev = moe.forward_smooth(*args, fields=names, workspace=ws)
    assert moe.device_error(ws) == 0
    assert torch.equal(y_plain.view(torch.int16), y_dbg.view(torch.int16))

    ids = dev["topk_ids"].cpu().numpy()
    topk_w = dev["topk_w"].cpu().numpy()
    slot_of = dev["slot_of"].cpu().numpy()
    _check_routing_arrays(cfg, ids, dev["offsets"].cpu().numpy(), slot_of, dev["slot_token"].cpu().numpy())

    tok = np.sort(np.random.default_rng(10).choice(cfg.T, SAMPLE[name], replace=False))
    ids_ref, w_ref, _ = oracle.router(inp.x[tok], inp.Wr, inp.bias, cfg.k)
    np.testing.assert_array_equal(ids[tok], ids_ref)
    np.testing.assert_allclose(topk_w[tok], w_ref, rtol=0, atol=TOPK_W_ATOL)
    ref_w = {}
    for e in sorted(set(ids_ref.ravel().tolist())):
        w13 = wl.expert_weight_fp32(cfg, "w13", e, seed, device="cuda").cpu().numpy()
        ref_w[e] = (oracle.quantize_rows_smoothed(w13, smooth[e]), _oracle_expert(cfg, "w2", e, seed))
        np.testing.assert_array_equal(w13_q[e].cpu().numpy(), ref_w[e][0][0])
        np.testing.assert_array_equal(w13_s[e].cpu().numpy(), ref_w[e][0][1])

    xf = oracle.bf16_to_f32(inp.x[tok])
    y_gpu = bf16_from_dev(y_dbg)[tok]
    y_ref = np.empty_like(y_gpu)
    for i, t in enumerate(tok):
        slots = slot_of[t]
        o_gpu = dev["o"][torch.from_numpy(slots).long().cuda()].cpu().numpy()
        o_own = np.empty_like(o_gpu)
        for j, s in enumerate(slots):
            e = int(ids_ref[i, j])
            (w13r, s13r), (w2r, s2r) = ref_w[e]
            # the slot's row: x times the binary32 reciprocals of its expert's factors, quantised per slot
            qx, sx = oracle.quantize_rows((xf[i] * (np.float32(1) / smooth[e]))[None])
            np.testing.assert_array_equal(dev["q_slot"][s].cpu().numpy(), qx[0])
            assert dev["s_slot"][s].item() == sx[0]
            acc1 = oracle.gemm_s8(qx, w13r)
            np.testing.assert_array_equal(dev["acc1"][s].cpu().numpy(), acc1[0])
            h_ref = oracle.epilogue_gate_up(acc1, sx, s13r)
            h_gpu = dev["h"][s].cpu().numpy()
            np.testing.assert_allclose(h_gpu, h_ref[0], rtol=H_RTOL, atol=1e-30)
            qh, sh = oracle.quantize_rows(h_gpu[None])
            np.testing.assert_array_equal(dev["q_h"][s].cpu().numpy(), qh[0])
            acc2 = oracle.gemm_s8(qh, w2r)
            np.testing.assert_array_equal(dev["acc2"][s].cpu().numpy(), acc2[0])
            np.testing.assert_array_equal(o_gpu[j], oracle.epilogue_scale(acc2, sh, s2r)[0])
            qh_o, sh_o = oracle.quantize_rows(h_ref)
            o_own[j] = oracle.epilogue_scale(oracle.gemm_s8(qh_o, w2r), sh_o, s2r)[0]
        one = np.arange(cfg.k, dtype=np.int32)[None]
        np.testing.assert_array_equal(y_gpu[i], oracle.combine(o_gpu, one, topk_w[t][None])[0])
        y_ref[i] = oracle.combine(o_own, one, w_ref[i][None])[0]
    assert_y_close(y_gpu, y_ref)


# ---- y of (nearly) every token against the oracle's own forward -------------

def _oracle_expert_weights(cfg, seed, experts, quant):
    """[E][...] weight arrays for the oracle: the experts in `experts`
    quantised by the oracle from the same fp32 draws, the rest zero (the
    oracle reads only the experts its tokens route to)."""
    code = np.uint8 if quant is oracle.quantize_rows_fp8 else np.int8
    w13_q = np.zeros((cfg.E, 2 * cfg.I, cfg.H), code)
    w13_s = np.zeros((cfg.E, 2 * cfg.I), np.float32)
    w2_q = np.zeros((cfg.E, cfg.H, cfg.I), code)
    w2_s = np.zeros((cfg.E, cfg.H), np.float32)
    for e in experts:
        w13_q[e], w13_s[e] = quant(wl.expert_weight_fp32(cfg, "w13", e, seed, device="cuda").cpu().numpy())
        w2_q[e], w2_s[e] = quant(wl.expert_weight_fp32(cfg, "w2", e, seed, device="cuda").cpu().numpy())
    return w13_q, w13_s, w2_q, w2_s


# the decode and prefill layers whole; 256 tokens of the 256-expert layer
# (its 11 GB of weights make the oracle's quantisation the cost, not its forward)
EVERY = {"decode": None, "prefill": None, "wide": 256}


@pytest.mark.parametrize("name", ["decode", "prefill", "wide"])
def test_full_size_layer_output_of_every_token_against_oracle(name):
    cfg = wl.CONFIGS[name]
    seed = 0
    inp = wl.make_moe_inputs(cfg, seed)
    args = (bf16_to_dev(inp.x), torch.from_numpy(inp.Wr).cuda(),
            None if inp.bias is None else torch.from_numpy(inp.bias).cuda(), *_device_weights(cfg, seed), cfg.k)
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y = moe.forward(*args, workspace=ws)
    assert moe.device_error(ws) == 0
    y_gpu = bf16_from_dev(y)
    del args, ws
    torch.cuda.empty_cache()
    n = EVERY[name]
    tok = np.arange(cfg.T) if n is None else np.sort(np.random.default_rng(11).choice(cfg.T, n, replace=False))
    ids_ref, _, _ = oracle.router(inp.x[tok], inp.Wr, inp.bias, cfg.k)
    weights = _oracle_expert_weights(cfg, seed, sorted(set(ids_ref.ravel().tolist())), oracle.quantize_rows)
    y_ref = oracle.moe_forward(inp.x[tok], inp.Wr, inp.bias, *weights, cfg.k)
    assert_y_close(y_gpu[tok], y_ref)


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_full_size_fp8_layer_output_of_many_tokens_against_oracle(name):
    cfg = wl.CONFIGS[name]
    seed = 0
    inp = wl.make_moe_inputs(cfg, seed)
    args = (bf16_to_dev(inp.x), torch.from_numpy(inp.Wr).cuda(),
            None if inp.bias is None else torch.from_numpy(inp.bias).cuda(), *_fp8_device_weights(cfg, seed), cfg.k)
    ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
    y = moe.fp8_forward(*args, workspace=ws)
    assert moe.device_error(ws) == 0
    y_gpu = bf16_from_dev(y)
    del args, ws
    torch.cuda.empty_cache()
    # the FP8 oracle sums in binary64 per product: 2048 of the prefill layer's tokens
    tok = np.arange(cfg.T) if cfg.T <= 2048 else np.sort(np.random.default_rng(12).choice(cfg.T, 2048, replace=False))
    ids_ref, _, _ = oracle.router(inp.x[tok], inp.Wr, inp.bias, cfg.k)
    weights = _oracle_expert_weights(cfg, seed, sorted(set(ids_ref.ravel().tolist())), oracle.quantize_rows_fp8)
    y_ref = oracle.moe_forward_fp8(inp.x[tok], inp.Wr, inp.bias, *weights, cfg.k)
    assert_y_close(y_gpu[tok], y_ref)
