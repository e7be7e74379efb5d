"""Parity of the CUDA library with the CPU oracle, stage by stage, on seeded
inputs that span several tiles and ragged tails.

Integer results (routing, slots, quantised codes, int32 accumulators) must
match bit for bit.  Float results are compared where the method is float:
h differs only through expf; every later stage is checked bit-exactly on the
GPU's own inputs to it (q_h from the GPU's h, acc2 from the GPU's q_h, o from
the GPU's acc2, y from the GPU's o), and end to end within the layer's
tolerance."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_quantised_moe_gb300 as moe
from w8a8_quantised_moe_gb300 import build as lib_build
from w8a8_quantised_moe_gb300 import workloads as wl
from gpu_helpers import (H_RTOL, Layer, assert_y_close, bf16_from_dev, bf16_to_dev, bits_to_f32,
                         gemm_path, y_errors)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib_build.build()
    moe._lib.load()


TINY = wl.CONFIGS["tiny"]
CASES = {
    "tiny": TINY,
    # 75 rows per expert: 128-row tiles, ragged tails
    "wide_tiles": TINY.replace(T=300, H=512, I=384, E=8, k=2),
    # 300 rows per expert: 256-row tiles, ragged tails
    "rows_256": TINY.replace(T=600, H=384, I=256, E=4, k=2),
    # 32-row tiles, router bias, top-4
    "top4_bias": TINY.replace(T=77, H=384, I=256, E=16, k=4, bias="normal", bias_std=0.5),
    # long reductions in both GEMMs
    "long_k": TINY.replace(T=100, H=1280, I=1152, E=4, k=2, n_outlier=13),
    "single_expert": TINY.replace(T=45, H=256, I=256, E=1, k=1),
    "one_token": TINY.replace(T=1, H=256, I=512, E=8, k=2),
    # about 500 rows per expert: CTA-pair tiles (192 rows), several per expert, ragged tails
    "pair_tiles": TINY.replace(T=1000, H=512, I=256, E=4, k=2),
    # CTA pairs with reductions longer than the stage ring in both GEMMs
    "pair_long_k": TINY.replace(T=800, H=1280, I=640, E=4, k=2, n_outlier=13),
    # CTA pairs under Zipf-skewed routing: experts from a few rows to several tiles
    "pair_skewed": TINY.replace(T=1200, H=256, I=256, E=8, k=2, bias="zipf", zipf_s=1.2),
    # about 125 rows per expert: one partial CTA-pair tile per expert
    "pair_one_tile": TINY.replace(T=500, H=512, I=256, E=8, k=2),
    # few-token router: an expert count that is not a multiple of 4 (router
    # weights staged 4 bytes at a time), top-3
    "odd_experts": TINY.replace(T=90, H=384, I=256, E=7, k=3),
    # few-token router at its largest T, 40 experts (padded logit tiles)
    "few_token_max": TINY.replace(T=128, H=512, I=256, E=40, k=3),
    # one token past it: the tensor-core router
    "tensor_router_min": TINY.replace(T=129, H=512, I=256, E=12, k=2),
    # the most experts and choices the library takes, few tokens
    "experts_256_top8": TINY.replace(T=100, H=256, I=128, E=256, k=8),
    # 256 experts, top-8, about 60 rows per expert: the one-CTA tensor-core GEMMs
    "experts_256_top8_many": TINY.replace(T=2000, H=256, I=256, E=256, k=8, bias="normal", bias_std=0.5),
}


def _stagewise(layer: Layer):
    cfg = layer.cfg
    names = ("topk_ids", "topk_w", "offsets", "slot_of", "slot_token", "s_x", "q_x", "acc1", "h",
             "s_h", "q_h", "acc2", "o")
    y_o, ref = layer.oracle(dump=names)
    y_d, dev = moe.forward_debug(*layer.device_args())
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in dev.items()}
    y_g = bf16_from_dev(y_d)

    # routing and permutation: exact
    np.testing.assert_array_equal(g["topk_ids"], ref["topk_ids"])
    np.testing.assert_allclose(g["topk_w"], ref["topk_w"], rtol=0, atol=1e-6)
    np.testing.assert_array_equal(g["offsets"], ref["offsets"])
    np.testing.assert_array_equal(g["slot_of"], ref["slot_of"])
    np.testing.assert_array_equal(g["slot_token"], ref["slot_token"])
    # activation quantisation: exact
    np.testing.assert_array_equal(g["s_x"], ref["s_x"])
    np.testing.assert_array_equal(g["q_x"], ref["q_x"])
    # GEMM1 accumulators: exact
    np.testing.assert_array_equal(g["acc1"], ref["acc1"])
    # h: float, differs only through expf
    np.testing.assert_allclose(g["h"], ref["h"], rtol=H_RTOL, atol=1e-30)
    # requantisation of the GPU's own h: exact
    q_h_ref, s_h_ref = oracle.quantize_rows(g["h"])
    np.testing.assert_array_equal(g["s_h"], s_h_ref)
    np.testing.assert_array_equal(g["q_h"], q_h_ref)
    # GEMM2 on the GPU's own q_h, then its epilogue: exact
    off = g["offsets"]
    for e in range(cfg.E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        acc2 = oracle.gemm_s8(g["q_h"][a:b], layer.w2_q[e])
        np.testing.assert_array_equal(g["acc2"][a:b], acc2)
        o = oracle.epilogue_scale(acc2, g["s_h"][a:b], layer.s2[e])
        np.testing.assert_array_equal(g["o"][a:b], o)
    # combine of the GPU's own o: exact
    y_stage = oracle.combine(g["o"], g["slot_of"], g["topk_w"])
    np.testing.assert_array_equal(y_g, y_stage)
    # end to end: the layer's tolerance
    assert_y_close(y_g, y_o)
    mismatch = int((g["q_h"] != ref["q_h"]).sum())
    return mismatch, y_errors(y_g, y_o)


@pytest.mark.parametrize("name", list(CASES))
def test_forward_matches_oracle_stage_by_stage(name):
    mismatch, (max_err, max_ref, mean_rel) = _stagewise(Layer(CASES[name], seed=0))
    cfg = CASES[name]
    # end-to-end q_h codes can differ only where expf moved h across a
    # rounding boundary: a vanishing fraction, each by one code
    assert mismatch <= max(2, cfg.T * cfg.k * cfg.I // 10000)


# every GEMM kernel on shapes from one row per expert to several tiles: the
# CUDA-core dp4a kernel (its automatic range is a few rows per expert, here
# also groups of hundreds of rows in chunks of 8), the one-CTA tensor-core
# kernels with 32-, 128- and 160-row tiles and the CTA-pair kernel
PATH_CASES = ("tiny", "one_token", "top4_bias", "long_k", "pair_skewed", "wide_tiles")


@pytest.mark.parametrize("path", ["skinny", "narrow", "mid", "wide", "pair"])
@pytest.mark.parametrize("name", PATH_CASES)
def test_forward_stage_by_stage_on_each_gemm_path(name, path):
    cfg = CASES[name]
    with gemm_path(path):
        mismatch, _ = _stagewise(Layer(cfg, seed=5))
    assert mismatch <= max(2, cfg.T * cfg.k * cfg.I // 10000)


def test_forward_all_tokens_to_one_expert():
    cfg = TINY.replace(T=150, H=256, I=256, E=6, k=1)
    layer = Layer(cfg, seed=2)
    layer.bias = np.array([0, 0, 0, 50, 0, 0], np.float32)  # every token picks expert 3
    layer.d_bias = torch.from_numpy(layer.bias).cuda()
    _stagewise(layer)


def test_forward_plain_entry_equals_debug_entry_and_is_deterministic():
    layer = Layer(CASES["wide_tiles"], seed=1)
    y1 = moe.forward(*layer.device_args())
    y2 = moe.forward(*layer.device_args())
    y3, _ = moe.forward_debug(*layer.device_args(), fields=("h",))
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))


def test_workspace_larger_than_needed_and_reused():
    big = Layer(CASES["wide_tiles"], seed=3)
    small = Layer(CASES["tiny"], seed=3)
    ws = moe.new_workspace(moe.workspace_size(300, 512, 384, 8, 2))
    y_big = moe.forward(*big.device_args(), workspace=ws)
    y_small = moe.forward(*small.device_args(), workspace=ws)
    assert moe.device_error(ws) == 0
    assert_y_close(bf16_from_dev(y_big), big.oracle())
    assert_y_close(bf16_from_dev(y_small), small.oracle())


def test_empty_batch_is_a_no_op():
    layer = Layer(TINY, seed=0)
    x0 = torch.empty((0, TINY.H), dtype=torch.bfloat16, device="cuda")
    y = moe.forward(x0, *layer.device_args()[1:])
    assert y.shape == (0, TINY.H)


# ------------------------------------------------------------------ weights

def test_quantize_weights_bit_exact():
    r = np.random.default_rng(11)
    w = (r.standard_normal((300, 520)) * 0.02).astype(np.float32)
    w[3] = 0.0
    w[5] *= 1e-30
    w[7] *= 1e20
    w[9, 17] = 5.0  # one dominant channel
    q_ref, s_ref = oracle.quantize_rows(w)
    q, s = moe.quantize_weights(torch.from_numpy(w).cuda())
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    # K not a multiple of 4 takes the scalar path
    q2, s2 = moe.quantize_weights(torch.from_numpy(w[:, :131].copy()).cuda())
    q2r, s2r = oracle.quantize_rows(w[:, :131])
    np.testing.assert_array_equal(q2.cpu().numpy(), q2r)
    np.testing.assert_array_equal(s2.cpu().numpy(), s2r)


# ------------------------------------------------------------------- linear

def _golden_linear_padded():
    """The hand-worked 2x4 example of tests/golden/linear_2x4.txt, zero-padded
    to K = N = 128 (padding changes neither the amax nor any sum)."""
    x = np.zeros((2, 128), np.float32)
    x[0, :4] = [1, -2, 0.5, 127]
    x[1, :4] = [63.5, -1.25, 0.75, -0.25]
    w = np.zeros((128, 128), np.int8)
    w[0, :4] = [1, 1, 1, 1]
    w[1, :4] = [-1, 0, 2, 1]
    s_w = np.ones(128, np.float32)
    s_w[:2] = [0.25, 0.125]
    return x, w, s_w


def test_linear_golden_example():
    x, w, s_w = _golden_linear_padded()
    xb = torch.from_numpy(x).to(torch.bfloat16).cuda()
    y = moe.linear(xb, torch.from_numpy(w).cuda(), torch.from_numpy(s_w).cuda())
    yf = y.float().cpu().numpy()
    np.testing.assert_array_equal(yf[:, :2], np.array([[31.5, 15.75], [15.875, -7.6875]], np.float32))
    assert (yf[:, 2:] == 0).all()


@pytest.mark.parametrize("M,N,K,path", [(1, 128, 128, "auto"), (37, 256, 384, "auto"), (300, 384, 1280, "auto"),
                                        (130, 128, 4096, "auto"), (500, 512, 1024, "auto"),
                                        (3, 384, 640, "auto"), (8, 1024, 2048, "auto"), (37, 256, 384, "skinny"),
                                        (9, 128, 1280, "narrow"), (5000, 128, 256, "auto"),
                                        (1500, 128, 1280, "auto"), (1300, 256, 2560, "auto"),
                                        (1250, 128, 7168, "auto")])
def test_linear_bit_exact(M, N, K, path):
    """M <= 8 rows take the dp4a kernel by default; 37 rows forced onto it
    pass in five chunks of up to 8 rows, the last one ragged; K = 384 and 640
    end on a half-filled 256-byte weight stage.  Above 8 rows per SM the
    quantiser takes one to eight warps per row by row length: 5000 x 256 one
    warp, 1500 x 1280 two, 1300 x 2560 four (2.5 vectors per lane: the
    warps' shares end unevenly), 1250 x 7168 eight; fewer rows take the
    CTA-per-token quantiser."""
    cfg = wl.LINEAR
    x = wl.draw_activations(7, cfg.cfg_id, M, K, max(1, K // 100))
    w32 = (np.random.default_rng(M + N + K).standard_normal((N, K)) * 0.02).astype(np.float32)
    w_q, s_w = oracle.quantize_rows(w32)
    y_ref = oracle.linear(x, w_q, s_w)
    with gemm_path(path):
        y = moe.linear(bf16_to_dev(x), torch.from_numpy(w_q).cuda(), torch.from_numpy(s_w).cuda())
    np.testing.assert_array_equal(bf16_from_dev(y), y_ref)


# --------------------------------------------------------------- exactness

@pytest.mark.parametrize("path", ["auto", "skinny"])
def test_int32_accumulators_exact_on_worst_case_inputs(path):
    """x = +-1 (every code +-127) against int8 weights spanning [-128, 127],
    K = 7168: the exact sums run far beyond 2^24, so any fp32 rounding in the
    tensor-core accumulation would show (and any int32 slip in the dp4a
    kernel)."""
    T, H, I = 64, 7168, 128
    r = np.random.default_rng(5)
    x = np.where(r.random((T, H)) < 0.5, -1.0, 1.0).astype(np.float32)
    x[:, :8] = 1.0  # some rows with long runs of one sign
    x[0, :] = 1.0
    xb = torch.from_numpy(x).to(torch.bfloat16)
    w13 = r.integers(-128, 128, (1, 2 * I, H)).astype(np.int8)
    w13[0, 0, :] = 127  # against row 0 of x: 7168 * 127 * 127 > 2^26
    w13[0, 1, :] = -128
    w2 = r.integers(-128, 128, (1, H, I)).astype(np.int8)
    s13 = np.full((1, 2 * I), 1e-6, np.float32)
    s2 = np.full((1, H), 1e-3, np.float32)
    Wr = np.zeros((H, 1), np.float32)
    args = (xb.cuda(), torch.from_numpy(Wr).cuda(), None, torch.from_numpy(w13).cuda(),
            torch.from_numpy(s13).cuda(), torch.from_numpy(w2).cuda(), torch.from_numpy(s2).cuda(), 1)
    with gemm_path(path):
        _, dev = moe.forward_debug(*args, fields=("q_x", "acc1", "q_h", "acc2"))
    q_x = dev["q_x"].cpu().numpy()
    assert (np.abs(q_x) == 127).all()
    ref1 = q_x.astype(np.int64) @ w13[0].astype(np.int64).T
    assert np.abs(ref1).max() > 2 ** 26
    np.testing.assert_array_equal(dev["acc1"].cpu().numpy(), ref1)
    q_h = dev["q_h"].cpu().numpy()
    ref2 = q_h.astype(np.int64) @ w2[0].astype(np.int64).T
    np.testing.assert_array_equal(dev["acc2"].cpu().numpy(), ref2)


def _boundary_rows(H):
    """Rows whose codes equal x (amax 127 -> s = 1): L1 = 2^17 and 2^17 + 1."""
    r = np.random.default_rng(9)
    rows = []
    for extra in (0, 1):
        mag = np.full(H, 64.0)
        mag[0] = 127.0
        mag[1:64] = 63.0  # 127 + 63*63 + 1984*64 = 131072
        if extra:
            mag[1] = 64.0  # 131073
        # row 0 positive (its weights -128 make every product -128 * |x|)
        sign = np.where(r.random(H) < 0.5, -1.0, 1.0) if extra else np.ones(H)
        sign[0] = 1.0
        rows.append(mag * sign)
    return np.array(rows, np.float32)


@pytest.mark.parametrize("path", ["narrow", "skinny"])
def test_exactness_certificate_boundary(path):
    """A positive row with L1 = 2^17 against weights -128 drives the partial
    sums down to exactly -2^24 on the tensor-core path; a row one above the
    bound goes to the exact CUDA-core path.  Both must be exact, and so must
    the dp4a kernel, which has no bound."""
    H, I = 2048, 128
    x = _boundary_rows(H)
    assert np.abs(x[0]).sum() == 2 ** 17 and np.abs(x[1]).sum() == 2 ** 17 + 1
    w13 = np.random.default_rng(3).integers(-128, 128, (1, 2 * I, H)).astype(np.int8)
    w13[0, 0] = -128   # partial sums of row 0 fall monotonically to -2^24
    w13[0, 1] = -128
    w13[0, 2] = 127
    w2 = np.random.default_rng(4).integers(-128, 128, (1, H, I)).astype(np.int8)
    args = (torch.from_numpy(x).to(torch.bfloat16).cuda(), torch.zeros((H, 1), device="cuda"), None,
            torch.from_numpy(w13).cuda(), torch.full((1, 2 * I), 1e-7, device="cuda"),
            torch.from_numpy(w2).cuda(), torch.full((1, H), 1e-3, device="cuda"), 1)
    with gemm_path(path):
        _, dev = moe.forward_debug(*args, fields=("q_x", "acc1", "q_h", "acc2"))
    q_x = dev["q_x"].cpu().numpy()
    np.testing.assert_array_equal(q_x, x.astype(np.int8))
    ref1 = q_x.astype(np.int64) @ w13[0].astype(np.int64).T
    assert ref1[0, 0] == -(2 ** 24)
    np.testing.assert_array_equal(dev["acc1"].cpu().numpy(), ref1)
    ref2 = dev["q_h"].cpu().numpy().astype(np.int64) @ w2[0].astype(np.int64).T
    np.testing.assert_array_equal(dev["acc2"].cpu().numpy(), ref2)


@pytest.mark.parametrize("path", ["narrow", "skinny"])
def test_second_gemm_exact_path(path):
    """Identical gate and up rows make h constant along I, so every q_h code
    is +-127 and L1(q_h) = 127 * 2048 is far above the bound: on the
    tensor-core kernel GEMM2 runs on the exact path for every row.  Compared
    with the oracle stage by stage."""
    cfg = TINY.replace(T=8, H=256, I=2048, E=2, k=1)
    layer = Layer(cfg, seed=4)
    layer.w13_q[:] = 1
    layer.d_w13 = torch.from_numpy(layer.w13_q).cuda()
    with gemm_path(path):
        mismatch, _ = _stagewise(layer)
        _, dev = moe.forward_debug(*layer.device_args(), fields=("q_h",))
    q_h = dev["q_h"].cpu().numpy()
    assert (np.abs(q_h.astype(np.int64)).sum(axis=1) > 2 ** 17).all()


def test_exact_path_mixed_rows_on_cta_pairs():
    """400 rows through one expert (CTA-pair tiles): four rows of +-1 (every
    code +-127, L1 far above the bound) take the exact CUDA-core path, the
    rest the tensor cores; both GEMMs' accumulators must be exact."""
    T, H, I = 400, 2048, 256
    r = np.random.default_rng(11)
    x = (r.standard_normal((T, H)) * 0.5).astype(np.float32)
    x[:4] = np.where(r.random((4, H)) < 0.5, -1.0, 1.0)
    w13 = r.integers(-128, 128, (1, 2 * I, H)).astype(np.int8)
    w2 = r.integers(-128, 128, (1, H, I)).astype(np.int8)
    args = (torch.from_numpy(x).to(torch.bfloat16).cuda(), torch.zeros((H, 1), device="cuda"), None,
            torch.from_numpy(w13).cuda(), torch.full((1, 2 * I), 1e-6, device="cuda"),
            torch.from_numpy(w2).cuda(), torch.full((1, H), 1e-3, device="cuda"), 1)
    _, dev = moe.forward_debug(*args, fields=("q_x", "acc1", "q_h", "acc2"))
    q_x = dev["q_x"].cpu().numpy()
    l1 = np.abs(q_x.astype(np.int64)).sum(axis=1)
    assert (l1[:4] > 2 ** 17).all() and (l1[4:] <= 2 ** 17).all()
    ref1 = q_x.astype(np.int64) @ w13[0].astype(np.int64).T
    np.testing.assert_array_equal(dev["acc1"].cpu().numpy(), ref1)
    q_h = dev["q_h"].cpu().numpy()
    ref2 = q_h.astype(np.int64) @ w2[0].astype(np.int64).T
    np.testing.assert_array_equal(dev["acc2"].cpu().numpy(), ref2)


def _f32_to_bf16_bits(x):
    """Round binary32 to bfloat16 bits, nearest-even (test-input construction)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def test_quantiser_every_bf16_value():
    """Every finite bf16 value v with |v| <= amax, quantised with the scale
    s = amax / 127 of ten row maxima: about 350 thousand quotients, dense near
    every half-integer where rint changes (the fast reciprocal path of the
    kernels decides those more than 2^-14 away, the division the rest).  The
    codes must equal the oracle's, which divides every element."""
    H = 4096
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    allf = bits_to_f32(allbits)
    finite = np.isfinite(allf)
    rows = []
    for amax in (1.0, 0.7, 1.3, 3.1, 100.0, 2e-3, 7e4, 0.0371, 5.9, 117.0):
        a_bits = _f32_to_bf16_bits(np.array([amax], np.float32))[0]
        a = bits_to_f32(np.array([a_bits], np.uint16))[0]
        vals = allbits[finite & (np.abs(allf) <= a)]
        n = H - 1
        pad = (-len(vals)) % n
        vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, n)
        rows.append(np.concatenate([np.full((vals.shape[0], 1), a_bits, np.uint16), vals], axis=1))
    x = np.concatenate(rows)
    T = x.shape[0]
    q_ref, s_ref = oracle.quantize_rows_bf16(x)
    I = 128
    w13 = np.zeros((1, 2 * I, H), np.int8)
    w2 = np.zeros((1, H, I), np.int8)
    args = (bf16_to_dev(x), torch.zeros((H, 1), device="cuda"), None, torch.from_numpy(w13).cuda(),
            torch.full((1, 2 * I), 1e-3, device="cuda"), torch.from_numpy(w2).cuda(),
            torch.full((1, H), 1e-3, device="cuda"), 1)
    _, dev = moe.forward_debug(*args, fields=("s_x", "q_x"))
    np.testing.assert_array_equal(dev["s_x"].cpu().numpy(), s_ref)
    np.testing.assert_array_equal(dev["q_x"].cpu().numpy(), q_ref)
    assert T * H > 300_000


def test_quantiser_rounding_boundaries():
    """Activation rows whose quotients x/s sit on or within a few ulp of the
    half-integers where rint changes (ties to even included): the codes must
    equal the oracle's, which divides exactly.  s = 1 and s = 2^-3 make
    x/s = m + 0.5 exact; other scales land the bf16-rounded quotients just
    either side of the boundaries."""
    H = 256
    rows = []
    r = np.random.default_rng(21)
    for amax in (127.0, 127.0 / 8, 3.0, 0.7, 1e-3, 5e4):
        s = np.float32(np.float32(amax) / np.float32(127.0))
        m = np.arange(-127, 127)  # (m + 0.5) * s stays within amax = 127 s
        v = np.concatenate([(m + 0.5) * np.float64(s), [0.0]])
        for jitter in (0.0, 1e-7, -1e-7, 1e-6, -1e-6):
            row = np.empty(H, np.float64)
            row[0] = amax  # fixes the row's amax
            row[1:] = v * (1.0 + jitter)
            r.shuffle(row[1:])
            bits = _f32_to_bf16_bits(row.astype(np.float32))
            # keep |x| <= amax after rounding: amax itself is exact in bf16 for the chosen values
            rows.append(bits)
    x = np.array(rows, np.uint16)
    xf = bits_to_f32(x)
    # amax of each row must stay the intended value after bf16 rounding
    assert (np.abs(xf).max(axis=1) == xf[:, 0]).all()
    T = x.shape[0]
    q_ref, s_ref = oracle.quantize_rows_bf16(x)
    # one expert, top-1: the codes of token t land in slot t
    I = 128
    w13 = np.zeros((1, 2 * I, H), np.int8)
    w2 = np.zeros((1, H, I), np.int8)
    args = (bf16_to_dev(x), torch.zeros((H, 1), device="cuda"), None, torch.from_numpy(w13).cuda(),
            torch.full((1, 2 * I), 1e-3, device="cuda"), torch.from_numpy(w2).cuda(),
            torch.full((1, H), 1e-3, device="cuda"), 1)
    _, dev = moe.forward_debug(*args, fields=("s_x", "q_x"))
    np.testing.assert_array_equal(dev["s_x"].cpu().numpy(), s_ref)
    np.testing.assert_array_equal(dev["q_x"].cpu().numpy(), q_ref)
    # the construction does hit ties: some quotients are exact half-integers
    ties = np.abs(xf[:, 1:] / s_ref[:, None] - np.round(xf[:, 1:] / s_ref[:, None])) == 0.5
    assert ties.sum() > 100
