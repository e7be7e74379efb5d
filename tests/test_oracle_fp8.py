"""Pins of the oracle's FP8 (E4M3) layer, on the CPU.

Each pin checks the oracle against something other than itself: values
worked by hand (tests/golden/e4m3.txt, "DeepSeek V4 950 FP8 inference on
H100" (lpnh.cn), section 2.1), PyTorch's float8_e4m3fn conversion (a library
routine), exact integer arithmetic for the GEMM, invariants of the
quantiser, and a brute-force dense evaluation of the whole layer.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3.txt")


def _golden():
    vals, codes = [], []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        v, c = line.split()[:2]
        vals.append(float(v))
        codes.append(int(c, 16))
    return np.array(vals, np.float32), np.array(codes, np.uint8)


def _torch_codes(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_values(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def test_e4m3_golden_table():
    v, c = _golden()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), c)


def test_e4m3_decode_every_code_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    nan = (codes & 0x7F) == 0x7F
    ours = oracle.e4m3_decode(codes)
    ref = _torch_values(codes)
    assert np.isnan(ours[nan]).all() and np.isnan(ref[nan]).all()
    np.testing.assert_array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_encode_against_torch():
    r = np.random.default_rng(3)
    x = np.concatenate([
        r.standard_normal(200_000).astype(np.float32) * np.float32(40.0),
        (r.random(50_000) * 0.03).astype(np.float32) * r.choice([-1, 1], 50_000).astype(np.float32),
        r.uniform(-463.9, 463.9, 50_000).astype(np.float32),
        # every midpoint between neighbouring finite codes, and one ulp either side
        *(lambda m: (m, np.nextafter(m, np.float32(np.inf)), np.nextafter(m, np.float32(-np.inf))))(
            ((oracle.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8)).astype(np.float64)
              + oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))) / 2).astype(np.float32)),
    ]).astype(np.float32)
    x = x[np.abs(x) < 464.0]  # torch's cast does not saturate; below 464 both round to nearest
    np.testing.assert_array_equal(oracle.e4m3_encode(x), _torch_codes(x))
    np.testing.assert_array_equal(oracle.e4m3_encode(-x), _torch_codes(-x))


def test_quantize_rows_fp8_invariants():
    r = np.random.default_rng(4)
    x = (r.standard_normal((64, 384)) * np.float32(3.0)).astype(np.float32)
    x[5] = 0.0
    x[7, 11] = 250.0  # an outlier
    q, s = oracle.quantize_rows_fp8(x)
    assert s[5] == 0 and (q[5] == 0).all()
    # s is the binary32 quotient amax / 448 and the amax element maps to +-448
    amax = np.abs(x).max(axis=1)
    np.testing.assert_array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    rows = np.arange(64) != 5
    arg = np.abs(x).argmax(axis=1)
    assert (oracle.e4m3_decode(q[rows, arg[rows]]) == np.sign(x[rows, arg[rows]]) * 448).all()
    # every code is the nearest E4M3 value to the quotient (torch's rounding)
    quot = (x[rows] / s[rows, None]).astype(np.float32)
    np.testing.assert_array_equal(q[rows], _torch_codes(quot))
    # relative error of a normal value at most 2^-4, absolute at most 2^-10 s below 2^-6 s
    deq = oracle.e4m3_decode(q[rows]).astype(np.float64) * s[rows, None]
    err = np.abs(deq - x[rows])
    bound = np.maximum(np.abs(x[rows]) * 2.0 ** -4, s[rows, None] * 2.0 ** -10) * (1 + 1e-6)
    assert (err <= bound).all()
    # sign symmetry and invariance under power-of-two scaling
    q2, s2 = oracle.quantize_rows_fp8(-x)
    np.testing.assert_array_equal(q2[rows], q[rows] ^ 0x80)
    q3, s3 = oracle.quantize_rows_fp8(x * np.float32(8.0))
    np.testing.assert_array_equal(q3, q)
    np.testing.assert_array_equal(s3, s * np.float32(8.0))


def _units(codes):
    """E4M3 values as exact integers in units of 2^-9 (torch's decode)."""
    v = _torch_values(codes).astype(np.float64) * 512.0
    assert (v == np.round(v)).all()
    return v.astype(np.int64)


def test_gemm_fp8_exact_against_integer_arithmetic():
    r = np.random.default_rng(5)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    for M, N, K in ((3, 5, 32), (17, 9, 1280), (4, 4, 8192)):
        a = r.choice(finite, (M, K))
        b = r.choice(finite, (N, K))
        exact = _units(a) @ _units(b).T  # units of 2^-18, |sum| < 2^53
        ref = (exact.astype(np.float64) * 2.0 ** -18).astype(np.float32)
        np.testing.assert_array_equal(oracle.gemm_fp8(a, b).view(np.uint32), ref.view(np.uint32))


def test_gemm_fp8_cancellation():
    # 448 * 448 - 448 * 448 + tiny: a binary32 running sum loses the tiny term,
    # the exact sum keeps it
    a = oracle.e4m3_encode(np.array([[448.0, 448.0, 2.0 ** -9]], np.float32))
    b = oracle.e4m3_encode(np.array([[448.0, -448.0, 2.0 ** -9]], np.float32))
    assert oracle.gemm_fp8(a, b)[0, 0] == np.float32(2.0 ** -18)


def test_epilogues_f32_match_the_int8_epilogues_on_integer_accumulators():
    r = np.random.default_rng(6)
    S, I, H = 7, 64, 96
    acc1 = r.integers(-2 ** 20, 2 ** 20, (S, 2 * I)).astype(np.int32)
    acc2 = r.integers(-2 ** 20, 2 ** 20, (S, H)).astype(np.int32)
    s_act = (r.random(S) * 0.01).astype(np.float32)
    s_w13 = (r.random(2 * I) * 0.001).astype(np.float32)
    s_w2 = (r.random(H) * 0.001).astype(np.float32)
    np.testing.assert_array_equal(oracle.epilogue_gate_up_f32(acc1.astype(np.float32), s_act, s_w13),
                                  oracle.epilogue_gate_up(acc1, s_act, s_w13))
    np.testing.assert_array_equal(oracle.epilogue_scale_f32(acc2.astype(np.float32), s_act, s_w2),
                                  oracle.epilogue_scale(acc2, s_act, s_w2))


@pytest.mark.parametrize("T,H,I,E,k", [(16, 256, 128, 8, 2), (23, 128, 256, 4, 3), (9, 128, 128, 1, 1)])
def test_moe_forward_fp8_equals_dense_brute_force(T, H, I, E, k):
    """Every expert evaluated on every token with numpy float64 products of
    torch-decoded codes, then the selected experts gathered and combined:
    the sparse oracle must agree bit for bit."""
    r = np.random.default_rng(T + H + I + E + k)
    x32 = r.standard_normal((T, H)).astype(np.float32)
    x = oracle.f32_to_bf16(x32)
    Wr = (r.standard_normal((H, E)) * 0.05).astype(np.float32)
    w13 = (r.standard_normal((E * 2 * I, H)) * 0.02).astype(np.float32)
    w2 = (r.standard_normal((E * H, I)) * 0.02).astype(np.float32)
    q13, s13 = oracle.quantize_rows_fp8(w13)
    q2, s2 = oracle.quantize_rows_fp8(w2)
    q13, s13 = q13.reshape(E, 2 * I, H), s13.reshape(E, 2 * I)
    q2, s2 = q2.reshape(E, H, I), s2.reshape(E, H)
    y, d = oracle.moe_forward_fp8(x, Wr, None, q13, s13, q2, s2, k, dump=("topk_ids", "topk_w"))

    ids, w = d["topk_ids"], d["topk_w"]
    qx, sx = oracle.quantize_rows_bf16_fp8(x)
    vx = _torch_values(qx).astype(np.float64)
    o_all = np.zeros((E, T, H), np.float32)
    for e in range(E):
        acc1 = (vx @ _torch_values(q13[e]).astype(np.float64).T).astype(np.float32)
        h = oracle.epilogue_gate_up_f32(acc1, sx, s13[e])
        qh, sh = oracle.quantize_rows_fp8(h)
        acc2 = (_torch_values(qh).astype(np.float64) @ _torch_values(q2[e]).astype(np.float64).T).astype(np.float32)
        o_all[e] = oracle.epilogue_scale_f32(acc2, sh, s2[e])
    # combine in top-k order, as the definition reads
    o_sel = np.stack([o_all[ids[:, j], np.arange(T)] for j in range(k)], axis=1)  # [T, k, H]
    slot_of = np.arange(T * k, dtype=np.int32).reshape(T, k)
    y_dense = oracle.combine(o_sel.reshape(T * k, H), slot_of, w)
    np.testing.assert_array_equal(y, y_dense)
