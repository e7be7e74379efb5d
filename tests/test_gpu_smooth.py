"""Parity of the SmoothQuant-folded layer (per-expert smoothing factors) with
the CPU oracle: the folded weight quantiser bit for bit, and the layer stage
by stage -- routing, each slot's scale and codes and both GEMMs' int32
accumulators exact, h within the expf tolerance, every later stage exact on
the GPU's own input, y within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl
from gpu_helpers import H_RTOL, assert_y_close, bf16_from_dev, bf16_to_dev

pytestmark = pytest.mark.gpu

TINY = wl.CONFIGS["tiny"]
CASES = {
    "tiny": TINY,
    # a few rows per expert: the dp4a GEMMs
    "decode_like": TINY.replace(T=40, H=1024, I=512, E=32, k=2),
    # hundreds of rows per expert: the CTA-pair GEMMs, ragged tiles
    "pair_tiles": TINY.replace(T=1000, H=512, I=256, E=4, k=2),
    # router bias, top-4
    "top4_bias": TINY.replace(T=77, H=384, I=256, E=16, k=4, bias="normal", bias_std=0.5),
    # the most experts and choices the library takes: 256 experts, top-8, router bias
    "experts_256_top8": TINY.replace(T=100, H=256, I=128, E=256, k=8, bias="normal", bias_std=0.5),
    "experts_256_top8_many": TINY.replace(T=2000, H=256, I=256, E=256, k=8, bias="normal", bias_std=0.5),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    moe._lib.load()


def _factors(cfg, seed):
    r = np.random.default_rng(100 + seed)
    return np.exp(r.uniform(-1.5, 1.5, (cfg.E, cfg.H))).astype(np.float32)


def test_quantize_weights_smoothed_bit_exact():
    r = np.random.default_rng(21)
    for rows, K in ((300, 1152), (37, 130)):  # K % 4 != 0 takes the scalar path
        w = (r.standard_normal((rows, K)) * 0.02).astype(np.float32)
        w[3] = 0.0
        f = np.exp(r.uniform(-2, 2, K)).astype(np.float32)
        q_ref, s_ref = oracle.quantize_rows_smoothed(w, f)
        q, s = moe.quantize_weights_smoothed(torch.from_numpy(w).cuda(), torch.from_numpy(f).cuda())
        np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
        np.testing.assert_array_equal(s.cpu().numpy(), s_ref)


def _weights(cfg, smooth, seed=0):
    q13, s13, q2, s2 = [], [], [], []
    for e in range(cfg.E):
        w13 = wl.expert_weight_fp32(cfg, "w13", e, seed).numpy()
        w2 = wl.expert_weight_fp32(cfg, "w2", e, seed).numpy()
        a, b = oracle.quantize_rows_smoothed(w13, smooth[e]) if smooth is not None else oracle.quantize_rows(w13)
        q13.append(a), s13.append(b)
        a, b = oracle.quantize_rows(w2)
        q2.append(a), s2.append(b)
    return np.stack(q13), np.stack(s13), np.stack(q2), np.stack(s2)


@pytest.mark.parametrize("name", list(CASES))
def test_smoothed_forward_matches_oracle_stage_by_stage(name):
    cfg = CASES[name]
    inp = wl.make_moe_inputs(cfg, 0)
    smooth = _factors(cfg, 0)
    q13, s13, q2, s2 = _weights(cfg, smooth)
    names = ("topk_ids", "topk_w", "offsets", "slot_of", "slot_token", "s_slot", "q_slot", "acc1", "h", "s_h",
             "q_h", "acc2", "o")
    y_o, ref = oracle.moe_forward_smooth(inp.x, inp.Wr, inp.bias, smooth, q13, s13, q2, s2, cfg.k, dump=names)
    bias = None if inp.bias is None else torch.from_numpy(inp.bias).cuda()
    dev_args = [torch.from_numpy(a).cuda() for a in (q13, s13, q2, s2)]
    y_d, dev = moe.forward_smooth(bf16_to_dev(inp.x), torch.from_numpy(inp.Wr).cuda(), bias,
                                  torch.from_numpy(smooth).cuda(), *dev_args, cfg.k, fields=names)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in dev.items()}
    y_g = bf16_from_dev(y_d)
    for k in ("topk_ids", "offsets", "slot_of", "slot_token", "s_slot", "q_slot", "acc1"):
        np.testing.assert_array_equal(g[k], ref[k], err_msg=k)
    np.testing.assert_allclose(g["topk_w"], ref["topk_w"], rtol=0, atol=1e-6)
    np.testing.assert_allclose(g["h"], ref["h"], rtol=H_RTOL, atol=1e-30)
    q_h, s_h = oracle.quantize_rows(g["h"])
    np.testing.assert_array_equal(g["q_h"], q_h)
    np.testing.assert_array_equal(g["s_h"], s_h)
    off = g["offsets"]
    for e in range(cfg.E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        acc2 = oracle.gemm_s8(g["q_h"][a:b], q2[e])
        np.testing.assert_array_equal(g["acc2"][a:b], acc2)
        np.testing.assert_array_equal(g["o"][a:b], oracle.epilogue_scale(acc2, g["s_h"][a:b], s2[e]))
    np.testing.assert_array_equal(y_g, oracle.combine(g["o"], g["slot_of"], g["topk_w"]))
    assert_y_close(y_g, y_o)


def test_unit_factors_equal_the_plain_forward():
    cfg = CASES["pair_tiles"]
    inp = wl.make_moe_inputs(cfg, 1)
    q13, s13, q2, s2 = _weights(cfg, None, 1)
    args = [bf16_to_dev(inp.x), torch.from_numpy(inp.Wr).cuda(), None]
    w = [torch.from_numpy(a).cuda() for a in (q13, s13, q2, s2)]
    ones = torch.ones((cfg.E, cfg.H), dtype=torch.float32, device="cuda")
    y0 = moe.forward(*args, *w, cfg.k)
    y1 = moe.forward_smooth(*args, ones, *w, cfg.k)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
