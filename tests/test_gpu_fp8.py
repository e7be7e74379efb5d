"""Parity of the FP8 (E4M3) layer of the CUDA library with the CPU oracle,
stage by stage, on seeded inputs spanning several tiles and ragged tails.

Routing, slots, the E4M3 codes and their scales must match bit for bit
(they are integer decisions taken in binary32 on both sides).  The two
GEMMs are fp32 accumulations of exact E4M3 products on the tensor cores:
each accumulator must lie within ACC_REL * sum_k |a_k b_k| of the exact dot
product (the oracle's).  Every later stage is checked bit for bit on the
GPU's own input to it, and y end to end within the layer's tolerance."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl
from gpu_helpers import H_RTOL, assert_y_close, bf16_from_dev, bf16_to_dev

pytestmark = pytest.mark.gpu

# fp32 accumulation of K exact products: observed up to 2.4e-7 of sum |p| at
# K = 4096 on GB300; the bound leaves a wide margin (a sequential binary32
# sum could reach K * 2^-24 of it in the worst case).
ACC_REL = 2.0 ** -16


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    moe._lib.load()


TINY = wl.CONFIGS["tiny"]
CASES = {
    "tiny": TINY,
    # 75 rows per expert: ragged tiles
    "wide_tiles": TINY.replace(T=300, H=512, I=384, E=8, k=2),
    # 500 rows per expert: several 256-row tiles, ragged tails
    "tiles_256": TINY.replace(T=1000, H=512, I=256, E=4, k=2),
    # the benchmark layer's reduction lengths
    "long_k": TINY.replace(T=100, H=4096, I=1536, E=4, k=2, n_outlier=41),
    # a couple of rows per expert (decode-shaped)
    "decode_like": TINY.replace(T=40, H=1024, I=512, E=32, k=2),
    # router bias, top-4, skewed experts
    "top4_zipf": TINY.replace(T=500, H=384, I=256, E=16, k=4, bias="zipf", zipf_s=1.2),
    "one_token": TINY.replace(T=1, H=256, I=512, E=8, k=2),
    # the most experts and choices the library takes: 256 experts, top-8,
    # softmax-renormalised weights, router bias (few tokens: one-CTA tiles;
    # more: about 60 rows per expert)
    "experts_256_top8": TINY.replace(T=100, H=256, I=128, E=256, k=8, bias="normal", bias_std=0.5),
    "experts_256_top8_many": TINY.replace(T=2000, H=256, I=256, E=256, k=8, bias="normal", bias_std=0.5),
}


def _weights(cfg, seed=0):
    w13 = np.stack([wl.expert_weight_fp32(cfg, "w13", e, seed).numpy() for e in range(cfg.E)])
    w2 = np.stack([wl.expert_weight_fp32(cfg, "w2", e, seed).numpy() for e in range(cfg.E)])
    q13, s13 = oracle.quantize_rows_fp8(w13.reshape(-1, cfg.H))
    q2, s2 = oracle.quantize_rows_fp8(w2.reshape(-1, cfg.I))
    return (w13, q13.reshape(cfg.E, 2 * cfg.I, cfg.H), s13.reshape(cfg.E, 2 * cfg.I),
            q2.reshape(cfg.E, cfg.H, cfg.I), s2.reshape(cfg.E, cfg.H))


def _values(codes):
    return oracle.e4m3_decode(codes).astype(np.float64)


def _assert_acc_close(acc, a_codes, w_codes):
    A, W = _values(a_codes), _values(w_codes)
    exact = A @ W.T  # exact: products are multiples of 2^-18 below 2^18, sums stay below 2^35
    mag = np.abs(A) @ np.abs(W).T
    err = np.abs(acc.astype(np.float64) - exact)
    assert (err <= ACC_REL * mag).all(), float((err / np.maximum(mag, 1e-300)).max())


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_forward_matches_oracle_stage_by_stage(name):
    cfg = CASES[name]
    inp = wl.make_moe_inputs(cfg, 0)
    _, q13, s13, q2, s2 = _weights(cfg)
    names = ("topk_ids", "topk_w", "offsets", "slot_of", "slot_token", "s_x", "q_x", "acc1", "h", "s_h", "q_h",
             "acc2", "o")
    y_o, ref = oracle.moe_forward_fp8(inp.x, inp.Wr, inp.bias, q13, s13, q2, s2, cfg.k, dump=names)
    bias = None if inp.bias is None else torch.from_numpy(inp.bias).cuda()
    y_d, dev = moe.fp8_forward_debug(bf16_to_dev(inp.x), torch.from_numpy(inp.Wr).cuda(), bias,
                                     torch.from_numpy(q13).cuda(), torch.from_numpy(s13).cuda(),
                                     torch.from_numpy(q2).cuda(), torch.from_numpy(s2).cuda(), cfg.k)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in dev.items()}
    y_g = bf16_from_dev(y_d)
    # routing, slots, activation codes and scales: exact
    for k in ("topk_ids", "offsets", "slot_of", "slot_token", "s_x", "q_x"):
        np.testing.assert_array_equal(g[k], ref[k], err_msg=k)
    np.testing.assert_allclose(g["topk_w"], ref["topk_w"], rtol=0, atol=1e-6)
    off, tok = g["offsets"], g["slot_token"]
    for e in range(cfg.E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        # GEMM1: within the fp32 accumulation bound of the exact dot products
        _assert_acc_close(g["acc1"][a:b], g["q_x"][tok[a:b]], q13[e])
        # gate/up epilogue of the GPU's own accumulators: differs only through expf
        h = oracle.epilogue_gate_up_f32(g["acc1"][a:b], g["s_x"][tok[a:b]], s13[e])
        np.testing.assert_allclose(g["h"][a:b], h, rtol=H_RTOL, atol=1e-30)
        # GEMM2 on the GPU's own E4M3 h, then its epilogue on the GPU's accumulators: exact
        _assert_acc_close(g["acc2"][a:b], g["q_h"][a:b], q2[e])
        np.testing.assert_array_equal(g["o"][a:b], oracle.epilogue_scale_f32(g["acc2"][a:b], g["s_h"][a:b], s2[e]))
    # requantisation of the GPU's own h: exact
    q_h, s_h = oracle.quantize_rows_fp8(g["h"])
    np.testing.assert_array_equal(g["s_h"], s_h)
    np.testing.assert_array_equal(g["q_h"], q_h)
    # combine of the GPU's own o: exact; end to end: the layer's tolerance
    np.testing.assert_array_equal(y_g, oracle.combine(g["o"], g["slot_of"], g["topk_w"]))
    assert_y_close(y_g, y_o)


def test_fp8_quantize_weights_bit_exact():
    r = np.random.default_rng(11)
    w = (r.standard_normal((300, 1152)) * 0.02).astype(np.float32)
    w[7] = 0.0
    w[9, 3] = 5.0          # an outlier row
    w[11] = -w[11]
    w[13, :] = 2.0 ** -130  # a row whose scale is subnormal
    q_ref, s_ref = oracle.quantize_rows_fp8(w)
    q, s = moe.fp8_quantize_weights(torch.from_numpy(w).cuda())
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)


def test_fp8_plain_entry_equals_debug_entry_and_is_deterministic():
    cfg = CASES["tiles_256"]
    inp = wl.make_moe_inputs(cfg, 1)
    _, q13, s13, q2, s2 = _weights(cfg, 1)
    args = (bf16_to_dev(inp.x), torch.from_numpy(inp.Wr).cuda(), None, torch.from_numpy(q13).cuda(),
            torch.from_numpy(s13).cuda(), torch.from_numpy(q2).cuda(), torch.from_numpy(s2).cuda(), cfg.k)
    y1 = bf16_from_dev(moe.fp8_forward(*args))
    y2 = bf16_from_dev(moe.fp8_forward(*args))
    y3, _ = moe.fp8_forward_debug(*args, fields=("q_x",))
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(y1, bf16_from_dev(y3))
