"""Pins of the oracle's SmoothQuant-folded layer (per-expert smoothing
factors), on the CPU.  "W8A8 quantisation of MiniMax-M3 on K100AI" (mhpn.cn),
section 2.2.  Each pin checks the oracle against something other than its own
code: values worked by hand, exact power-of-two invariances (smoothing by 2^j
commutes with every rounding of the layer, so the layer must not change), the
plain layer when every factor is 1, and a dense brute-force evaluation that
applies the factors per (token, expert) with numpy binary32 arithmetic."""
import numpy as np
import pytest

import oracle


def test_smooth_factors_worked_by_hand():
    xa = np.array([4, 9, 0, 2, 2, 5, 5], np.float32)
    wa = np.array([1, 4, 3, 0, 8, 7, 4], np.float32)
    # alpha = 1/2: sqrt(4)/sqrt(1) = 2, sqrt(9)/sqrt(4) = 1.5, zero statistics -> 1, sqrt(2/8) = 0.5
    np.testing.assert_array_equal(oracle.smooth_factors(xa[:5], wa[:5], 0.5), [2, 1.5, 1, 1, 0.5])
    # alpha = 1: the activation statistic alone; alpha = 0: one over the weight statistic
    np.testing.assert_array_equal(oracle.smooth_factors(xa[5:6], wa[5:6], 1.0), [5])
    np.testing.assert_array_equal(oracle.smooth_factors(xa[6:7], wa[6:7], 0.0), [0.25])


def test_quantize_rows_smoothed_unit_and_power_of_two_factors():
    r = np.random.default_rng(1)
    w = (r.standard_normal((48, 256)) * 0.02).astype(np.float32)
    q0, s0 = oracle.quantize_rows(w)
    q1, s1 = oracle.quantize_rows_smoothed(w, np.ones(256, np.float32))
    np.testing.assert_array_equal(q1, q0)
    np.testing.assert_array_equal(s1, s0)
    # one power of two for every column: the same codes, scales times 2^3
    q2, s2 = oracle.quantize_rows_smoothed(w, np.full(256, 8.0, np.float32))
    np.testing.assert_array_equal(q2, q0)
    np.testing.assert_array_equal(s2, s0 * np.float32(8))
    # a power of two per column: the fold is exact, so it is the quantiser of w * f
    f = (2.0 ** r.integers(-3, 4, 256)).astype(np.float32)
    q3, s3 = oracle.quantize_rows_smoothed(w, f)
    qr, sr = oracle.quantize_rows(w * f)
    np.testing.assert_array_equal(q3, qr)
    np.testing.assert_array_equal(s3, sr)


def _layer(T, H, I, E, k, seed):
    r = np.random.default_rng(seed)
    x32 = r.standard_normal((T, H)).astype(np.float32)
    x32[:, 3] *= 20  # an outlier channel
    x = oracle.f32_to_bf16(x32)
    Wr = (r.standard_normal((H, E)) * 0.05).astype(np.float32)
    w13 = (r.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32)
    w2 = (r.standard_normal((E, H, I)) * 0.02).astype(np.float32)
    return r, x, Wr, w13, w2


def _quantize_experts(w13, w2, smooth=None):
    E = w13.shape[0]
    q13, s13, q2, s2 = [], [], [], []
    for e in range(E):
        a, b = (oracle.quantize_rows(w13[e]) if smooth is None else oracle.quantize_rows_smoothed(w13[e], smooth[e]))
        q13.append(a), s13.append(b)
        a, b = oracle.quantize_rows(w2[e])
        q2.append(a), s2.append(b)
    return np.stack(q13), np.stack(s13), np.stack(q2), np.stack(s2)


NAMES = ("topk_ids", "topk_w", "offsets", "slot_of", "slot_token", "acc1", "h", "s_h", "q_h", "acc2", "o")


def test_unit_factors_give_the_plain_layer():
    _, x, Wr, w13, w2 = _layer(20, 128, 64, 6, 2, 3)
    q13, s13, q2, s2 = _quantize_experts(w13, w2)
    y0, d0 = oracle.moe_forward(x, Wr, None, q13, s13, q2, s2, 2, dump=NAMES + ("s_x", "q_x"))
    ones = np.ones((6, 128), np.float32)
    y1, d1 = oracle.moe_forward_smooth(x, Wr, None, ones, q13, s13, q2, s2, 2, dump=NAMES + ("s_slot", "q_slot"))
    np.testing.assert_array_equal(y1, y0)
    for n in NAMES:
        np.testing.assert_array_equal(d1[n], d0[n], err_msg=n)
    tok = d0["slot_token"]
    np.testing.assert_array_equal(d1["q_slot"], d0["q_x"][tok])
    np.testing.assert_array_equal(d1["s_slot"], d0["s_x"][tok])


def test_power_of_two_factors_leave_the_layer_unchanged():
    """s_e = 2^j_e on every channel: x / s and w * s are exact, the activation
    scale becomes s_x 2^-j_e and the weight scale s_w 2^j_e, the codes are the
    same, and the epilogue's two products give the same binary32 values."""
    T, H, I, E, k = 24, 128, 64, 5, 2
    _, x, Wr, w13, w2 = _layer(T, H, I, E, k, 4)
    j = np.array([-2, 0, 1, 3, -1])
    smooth = np.repeat((2.0 ** j).astype(np.float32)[:, None], H, axis=1)
    y0, d0 = oracle.moe_forward(x, Wr, None, *_quantize_experts(w13, w2), k, dump=("slot_token", "offsets", "s_x",
                                                                                  "q_x"))
    y1, d1 = oracle.moe_forward_smooth(x, Wr, None, smooth, *_quantize_experts(w13, w2, smooth), k,
                                       dump=("s_slot", "q_slot"))
    np.testing.assert_array_equal(y1, y0)
    tok, off = d0["slot_token"], d0["offsets"]
    np.testing.assert_array_equal(d1["q_slot"], d0["q_x"][tok])
    e_of_slot = np.searchsorted(off, np.arange(T * k), side="right") - 1
    np.testing.assert_array_equal(d1["s_slot"], d0["s_x"][tok] * (2.0 ** -j[e_of_slot]).astype(np.float32))


def test_smoothing_worked_by_hand():
    # one token, one expert: x = [2, -8, 1, 4], factors [1, 4, 0.5, 2] -> x / s = [2, -2, 2, 2]:
    # amax 2, s = 2/127, codes [127, -127, 127, 127]  (unsmoothed: amax 8, codes [32, -127, 16, 64])
    x = oracle.f32_to_bf16(np.array([[2, -8, 1, 4]], np.float32))
    Wr = np.ones((4, 1), np.float32)
    smooth = np.array([[1, 4, 0.5, 2]], np.float32)
    w13 = np.ones((1, 2, 4), np.float32)
    w2 = np.ones((1, 4, 1), np.float32)
    q13, s13, q2, s2 = _quantize_experts(w13, w2, smooth)
    _, d = oracle.moe_forward_smooth(x, Wr, None, smooth, q13, s13, q2, s2, 1, dump=("s_slot", "q_slot"))
    np.testing.assert_array_equal(d["q_slot"], [[127, -127, 127, 127]])
    assert d["s_slot"][0] == np.float32(2) / np.float32(127)
    _, d0 = oracle.moe_forward(x, Wr, None, *_quantize_experts(w13, w2), 1, dump=("q_x",))
    np.testing.assert_array_equal(d0["q_x"], [[32, -127, 16, 64]])


@pytest.mark.parametrize("T,H,I,E,k", [(16, 128, 64, 6, 2), (11, 256, 128, 4, 3)])
def test_sparse_smoothed_layer_equals_dense_brute_force(T, H, I, E, k):
    r, x, Wr, w13, w2 = _layer(T, H, I, E, k, 5 + T)
    smooth = np.exp(r.uniform(-1.5, 1.5, (E, H))).astype(np.float32)
    q13, s13, q2, s2 = _quantize_experts(w13, w2, smooth)
    y, d = oracle.moe_forward_smooth(x, Wr, None, smooth, q13, s13, q2, s2, k, dump=("topk_ids", "topk_w"))
    ids, tw = d["topk_ids"], d["topk_w"]
    xf = oracle.bf16_to_f32(x)
    o_sel = np.zeros((T, k, H), np.float32)
    for t in range(T):
        for jj in range(k):
            e = ids[t, jj]
            xs = xf[t] * (np.float32(1) / smooth[e])  # binary32 reciprocal, binary32 product
            qx, sx = oracle.quantize_rows(xs[None])
            acc1 = qx.astype(np.int64) @ q13[e].astype(np.int64).T
            h = oracle.epilogue_gate_up(acc1.astype(np.int32), sx, s13[e])
            qh, sh = oracle.quantize_rows(h)
            acc2 = qh.astype(np.int64) @ q2[e].astype(np.int64).T
            o_sel[t, jj] = oracle.epilogue_scale(acc2.astype(np.int32), sh, s2[e])[0]
    slot_of = np.arange(T * k, dtype=np.int32).reshape(T, k)
    np.testing.assert_array_equal(y, oracle.combine(o_sel.reshape(T * k, H), slot_of, tw))
