"""Pins for the CPU oracle: each test ties an oracle function to something
other than the oracle itself -- a hand-worked example, a closed form, an
invariant of the definition, a library routine, or brute force."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from w8a8_quantised_moe_gb300 import workloads as wl

from conftest import GOLDEN


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- quantiser

def _quant_golden():
    rows = []
    for line in _lines("quant_4x4.txt"):
        x, s, q = (part.split() for part in line.split("|"))
        rows.append(([float(v) for v in x], float(s[0]), [int(v) for v in q]))
    return rows


def test_quant_golden_4x4():
    rows = _quant_golden()
    x = np.array([r[0] for r in rows], np.float32)
    q, s = oracle.quantize_rows(x)
    np.testing.assert_array_equal(s, np.array([r[1] for r in rows], np.float32))
    np.testing.assert_array_equal(q, np.array([r[2] for r in rows], np.int8))
    # same rows through the bf16 entry (all values are exact in bf16)
    qb, sb = oracle.quantize_rows_bf16(_bf16_bits(x))
    np.testing.assert_array_equal(qb, q)
    np.testing.assert_array_equal(sb, s)


def _random_rows(seed, rows=64, K=777):
    r = np.random.default_rng(seed)
    x = r.standard_normal((rows, K)).astype(np.float32)
    x[:, r.choice(K, 8, replace=False)] *= 20
    x[3] *= 1e-30  # tiny magnitudes
    x[5] *= 1e30  # huge magnitudes
    x[7, :] = 0
    x[7, 11] = -3.0  # single non-zero
    return x


def test_quant_dequant_error_bound():
    """|q*s - x| <= s/2 per element (plus the rounding of x/s itself)."""
    x = _random_rows(1)
    q, s = oracle.quantize_rows(x)
    err = np.abs(q.astype(np.float64) * s[:, None].astype(np.float64) - x.astype(np.float64))
    bound = s[:, None].astype(np.float64) * (0.5 + 127 * 2.0 ** -23)
    assert (err <= bound).all()
    assert np.abs(q.astype(np.int32)).max() <= 127


def test_quant_amax_element_maps_to_127_and_scale_is_amax_over_127():
    x = _random_rows(2)
    q, s = oracle.quantize_rows(x)
    amax = np.abs(x).max(axis=1)
    np.testing.assert_array_equal(s, (amax / np.float32(127)).astype(np.float32))
    for r in range(x.shape[0]):
        if amax[r] == 0:
            assert (q[r] == 0).all() and s[r] == 0
            continue
        i = int(np.argmax(np.abs(x[r])))
        assert q[r, i] == (127 if x[r, i] > 0 else -127)


def test_quant_sign_symmetry_and_power_of_two_scaling():
    x = _random_rows(3)[:, :300]
    x = x[np.abs(x).max(axis=1) < 1e20]  # keep x * 2^8 finite
    q, s = oracle.quantize_rows(x)
    qn, sn = oracle.quantize_rows(-x)
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(sn, s)
    for p in (-8, 5):
        qp, sp = oracle.quantize_rows((x * np.float32(2.0 ** p)).astype(np.float32))
        np.testing.assert_array_equal(qp, q)
        np.testing.assert_array_equal(sp, (s * np.float32(2.0 ** p)).astype(np.float32))


def test_quant_exact_integer_multiples():
    """x = n * 2^-3 with max |n| = 127 has s = 2^-3 exactly and q = n."""
    r = np.random.default_rng(4)
    n = r.integers(-127, 128, size=(10, 256))
    n[:, 0] = 127
    x = (n * 0.125).astype(np.float32)
    q, s = oracle.quantize_rows(x)
    np.testing.assert_array_equal(s, np.full(10, 0.125, np.float32))
    np.testing.assert_array_equal(q, n.astype(np.int8))


def test_quant_bf16_entry_matches_widened_f32():
    bits = _bf16_bits(_random_rows(5))
    qb, sb = oracle.quantize_rows_bf16(bits)
    q, s = oracle.quantize_rows(_bits_to_f32(bits))
    np.testing.assert_array_equal(qb, q)
    np.testing.assert_array_equal(sb, s)


# -------------------------------------------------------------- bf16 helpers

def test_bf16_rounding_matches_torch():
    r = np.random.default_rng(6)
    x = np.concatenate([
        r.standard_normal(20000).astype(np.float32) * 10.0 ** r.integers(-30, 30, 20000),
        np.array([0.0, -0.0, 1.00390625, 1.01171875, -1.00390625, 3.0e38, -3.4e38, 1e-40,
                  np.inf, -np.inf], np.float32),
    ]).astype(np.float32)
    # exact half-way points between bf16 neighbours
    base = _bits_to_f32(r.integers(0x0080, 0x7f00, 5000).astype(np.uint16))
    x = np.concatenate([x, (base.view(np.uint32) | 0x8000).view(np.float32)])
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(oracle.bf16_to_f32(ours), _bits_to_f32(ours))


# ---------------------------------------------------------------- int GEMM

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 5, 33), (33, 64, 256), (5, 3, 4096)])
def test_gemm_matches_numpy_int64(M, N, K):
    r = np.random.default_rng(M * 1000 + N + K)
    a = r.integers(-128, 128, (M, K), dtype=np.int64).astype(np.int8)
    b = r.integers(-128, 128, (N, K), dtype=np.int64).astype(np.int8)
    a[0, :] = -128
    b[0, :] = -128
    acc = oracle.gemm_s8(a, b)
    ref = a.astype(np.int64) @ b.astype(np.int64).T
    np.testing.assert_array_equal(acc.astype(np.int64), ref)


def test_gemm_reports_int32_overflow():
    K = 131073  # 131073 * 128 * 128 > 2^31 - 1
    a = np.full((1, K), -128, np.int8)
    with pytest.raises(oracle.OracleError, match="overflow"):
        oracle.gemm_s8(a, a)
    # one below the bound still fits
    K = 131071
    a = np.full((1, K), -128, np.int8)
    assert int(oracle.gemm_s8(a, a)[0, 0]) == K * 16384


# ---------------------------------------------------------- linear epilogue

def _linear_golden():
    rec = {"x": [], "w": [], "s_w": [], "acc": [], "y": []}
    for line in _lines("linear_2x4.txt"):
        key, *vals = line.split()
        rec[key].append([float(v) for v in vals])
    return {k: np.array(v) for k, v in rec.items()}


def test_linear_golden_2x4():
    g = _linear_golden()
    x = _bf16_bits(g["x"].astype(np.float32))
    w_q = g["w"].astype(np.int8)
    s_w = g["s_w"][0].astype(np.float32)
    y, mid = oracle.linear(x, w_q, s_w, want_intermediates=True)
    np.testing.assert_array_equal(mid["q_x"], np.array([[1, -2, 0, 127], [127, -2, 2, 0]], np.int8))
    np.testing.assert_array_equal(mid["s_x"], np.array([1, 0.5], np.float32))
    np.testing.assert_array_equal(mid["acc"], g["acc"].astype(np.int32))
    np.testing.assert_array_equal(_bits_to_f32(y), g["y"].astype(np.float32))
    # the scale epilogue alone on the same accumulators
    out = oracle.epilogue_scale(g["acc"].astype(np.int32), mid["s_x"], s_w)
    np.testing.assert_array_equal(out, g["y"].astype(np.float32))


def test_epilogue_scale_closed_form():
    """(float(acc) * s_a) * s_w with power-of-two scales is exact."""
    r = np.random.default_rng(7)
    acc = r.integers(-2 ** 20, 2 ** 20, (9, 17)).astype(np.int32)
    s_a = (2.0 ** r.integers(-12, 4, 9)).astype(np.float32)
    s_w = (2.0 ** r.integers(-12, 4, 17)).astype(np.float32)
    out = oracle.epilogue_scale(acc, s_a, s_w)
    np.testing.assert_array_equal(out, (acc * s_a[:, None].astype(np.float64) * s_w[None, :]).astype(np.float32))


def test_epilogue_gate_up_closed_form():
    """h = silu(g) * u against binary64 g/(1+exp(-g)) * u, within the
    rounding of a handful of binary32 operations."""
    r = np.random.default_rng(8)
    S, I = 16, 64
    acc = r.integers(-300000, 300000, (S, 2 * I)).astype(np.int32)
    acc[0, :I] = 0  # g = 0 -> h = 0
    acc[1, I:] = 0  # u = 0 -> h = 0
    s_a = (r.random(S) * 1e-3 + 1e-4).astype(np.float32)
    s_w = (r.random(2 * I) * 1e-2 + 1e-3).astype(np.float32)
    h = oracle.epilogue_gate_up(acc, s_a, s_w)
    g = (acc[:, :I].astype(np.float32) * s_a[:, None]).astype(np.float32) * s_w[None, :I]
    u = (acc[:, I:].astype(np.float32) * s_a[:, None]).astype(np.float32) * s_w[None, I:]
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64))) * u.astype(np.float64)
    assert (h[0] == 0).all() and (h[1] == 0).all()
    rel = np.abs(h - ref) / np.maximum(np.abs(ref), 1e-30)
    assert rel.max() < 8 * 2.0 ** -24
    # large positive g: silu(g) = g exactly; large negative g: silu(g) -> 0
    big = np.zeros((2, 2), np.int32)
    big[0, 0], big[0, 1] = 2 ** 20, 3
    big[1, 0], big[1, 1] = -(2 ** 20), 3
    hb = oracle.epilogue_gate_up(big, np.ones(2, np.float32), np.ones(2, np.float32))
    assert hb[0, 0] == np.float32(2 ** 20 * 3)
    assert hb[1, 0] == 0.0


# ------------------------------------------------------------------ router

def _router_cases():
    for line in _lines("router_topk.txt"):
        parts = [p.split() for p in line.split("|")]
        logits = [float(v) for v in parts[0][2:]]
        k = int(parts[1][1])
        ids = [int(v) for v in parts[2][1:]]
        w = [float(v) for v in parts[3][1:]]
        yield logits, k, ids, w


@pytest.mark.parametrize("case", list(_router_cases()))
def test_router_golden(case):
    logits, k, ids, w = case
    E = len(logits)
    # one-hot activation on channel 0, router row 0 = the logits: exact logits
    H = 8
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    Wr = np.zeros((H, E), np.float32)
    Wr[0] = logits
    got_ids, got_w, got_l = oracle.router(_bf16_bits(x), Wr, None, k)
    np.testing.assert_array_equal(got_l[0], np.array(logits, np.float32))
    assert got_ids[0].tolist() == ids
    np.testing.assert_allclose(got_w[0], np.array(w), rtol=2 ** -23, atol=0)
    # the same logits split between a zero row product and a bias
    got_ids2, got_w2, _ = oracle.router(_bf16_bits(x * 0), Wr, np.array(logits, np.float32), k)
    assert got_ids2[0].tolist() == ids
    np.testing.assert_array_equal(got_w2, got_w)


def test_router_matches_library_routines():
    cfg = wl.CONFIGS["tiny"].replace(T=200, E=16, k=4)
    inp = wl.make_moe_inputs(cfg, seed=3)
    bias = (np.random.default_rng(9).standard_normal(cfg.E) * 0.5).astype(np.float32)
    ids, w, logits = oracle.router(inp.x, inp.Wr, bias, cfg.k)
    ref = wl.bf16_bits_to_f64(inp.x) @ inp.Wr.astype(np.float64) + bias.astype(np.float64)
    # logits: the binary64 dot product rounded once (BLAS may sum in another order)
    np.testing.assert_allclose(logits, ref.astype(np.float32), rtol=2.0 ** -23, atol=1e-7)
    order = np.argsort(-logits, axis=1, kind="stable")[:, : cfg.k]
    np.testing.assert_array_equal(ids, order)
    sel = np.take_along_axis(logits.astype(np.float64), order, axis=1)
    sm = np.exp(sel - sel[:, :1])
    sm /= sm.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, sm, rtol=1e-6)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-6)


# ------------------------------------------------------------- permutation

@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (37, 8, 2), (500, 64, 2), (300, 256, 8)])
def test_permute_matches_stable_argsort(T, E, k):
    r = np.random.default_rng(T + E + k)
    ids = np.stack([r.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, slot_of, slot_token = oracle.permute(ids, E)
    flat = ids.ravel()
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    order = np.argsort(flat, kind="stable")  # slots: experts ascending, then (t, j) order
    np.testing.assert_array_equal(slot_token, order // k)
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    np.testing.assert_array_equal(slot_of.ravel(), inv)
    # bijection onto [0, S), monotone offsets
    assert sorted(slot_of.ravel().tolist()) == list(range(T * k))
    assert (np.diff(offsets) >= 0).all() and offsets[-1] == T * k


def test_permute_empty_experts_and_single_expert():
    ids = np.zeros((5, 1), np.int32) + 3
    counts, offsets, slot_of, slot_token = oracle.permute(ids, 6)
    assert counts.tolist() == [0, 0, 0, 5, 0, 0]
    assert offsets.tolist() == [0, 0, 0, 0, 5, 5, 5]
    assert slot_of.ravel().tolist() == [0, 1, 2, 3, 4]
    assert slot_token.tolist() == [0, 1, 2, 3, 4]


# ----------------------------------------------------------------- combine

def test_combine_golden():
    for line in _lines("combine.txt"):
        w, o, y = ([float(v) for v in p.split()] for p in line.split("|"))
        k = len(w)
        o_rows = np.array(o, np.float32).reshape(k, 1)
        got = oracle.combine(o_rows, np.arange(k, dtype=np.int32).reshape(1, k), np.array([w], np.float32))
        assert _bits_to_f32(got)[0, 0] == np.float32(y[0]), line


def test_combine_single_expert_is_bf16_of_scaled_row():
    r = np.random.default_rng(10)
    o = r.standard_normal((6, 40)).astype(np.float32)
    slot_of = np.arange(6, dtype=np.int32)[::-1].reshape(6, 1).copy()
    w = np.ones((6, 1), np.float32)
    y = oracle.combine(o, slot_of, w)
    ref = torch.from_numpy(o[::-1].copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(y, ref)


# ------------------------------------------------------------ whole layer

def _tiny_layer(cfg, seed):
    inp = wl.make_moe_inputs(cfg, seed)
    w13 = np.stack([wl.expert_weight_fp32(cfg, "w13", e, seed).numpy() for e in range(cfg.E)])
    w2 = np.stack([wl.expert_weight_fp32(cfg, "w2", e, seed).numpy() for e in range(cfg.E)])
    w13_q, s13 = oracle.quantize_rows(w13.reshape(-1, cfg.H))
    w2_q, s2 = oracle.quantize_rows(w2.reshape(-1, cfg.I))
    return (inp, w13_q.reshape(cfg.E, 2 * cfg.I, cfg.H), s13.reshape(cfg.E, 2 * cfg.I),
            w2_q.reshape(cfg.E, cfg.H, cfg.I), s2.reshape(cfg.E, cfg.H))


@pytest.mark.parametrize("cfg", [
    wl.CONFIGS["tiny"],
    wl.CONFIGS["tiny"].replace(T=9, H=128, I=128, E=5, k=3, bias="normal", bias_std=0.5),
    wl.CONFIGS["tiny"].replace(T=4, H=128, I=256, E=1, k=1),
])
def test_sparse_equals_brute_force_dense(cfg):
    inp, w13_q, s13, w2_q, s2 = _tiny_layer(cfg, seed=0)
    y_sparse = oracle.moe_forward(inp.x, inp.Wr, inp.bias, w13_q, s13, w2_q, s2, cfg.k)
    y_dense = oracle.moe_forward_dense(inp.x, inp.Wr, inp.bias, w13_q, s13, w2_q, s2, cfg.k)
    np.testing.assert_array_equal(y_sparse, y_dense)


def test_forward_intermediates_satisfy_invariants():
    cfg = wl.CONFIGS["tiny"]
    inp, w13_q, s13, w2_q, s2 = _tiny_layer(cfg, seed=1)
    names = ("topk_ids", "topk_w", "offsets", "slot_of", "slot_token", "s_x", "q_x", "acc1", "h",
             "s_h", "q_h", "acc2", "o")
    y, d = oracle.moe_forward(inp.x, inp.Wr, inp.bias, w13_q, s13, w2_q, s2, cfg.k, dump=names)
    np.testing.assert_allclose(d["topk_w"].sum(axis=1), 1.0, atol=1e-6)
    S = cfg.T * cfg.k
    assert sorted(d["slot_of"].ravel().tolist()) == list(range(S))
    # integer accumulators against numpy's int64 matmul, slot by slot
    for s in range(S):
        t = d["slot_token"][s]
        e = int(np.searchsorted(d["offsets"], s, side="right") - 1)
        ref1 = w13_q[e].astype(np.int64) @ d["q_x"][t].astype(np.int64)
        np.testing.assert_array_equal(d["acc1"][s], ref1)
        ref2 = w2_q[e].astype(np.int64) @ d["q_h"][s].astype(np.int64)
        np.testing.assert_array_equal(d["acc2"][s], ref2)
    # dequantisation bound on the requantised h
    err = np.abs(d["q_h"] * d["s_h"][:, None].astype(np.float64) - d["h"])
    assert (err <= d["s_h"][:, None] * (0.5 + 1e-5)).all()
    # y is the bf16 of a convex combination of the expert rows
    o = d["o"][d["slot_of"]]  # [T, k, H]
    lo, hi = o.min(axis=1), o.max(axis=1)
    yf = _bits_to_f32(y)
    assert ((yf >= lo - np.abs(lo) * 2 ** -7 - 1e-30) & (yf <= hi + np.abs(hi) * 2 ** -7 + 1e-30)).all()


# -------------------------------------------------------------- workloads

def test_workload_gap_condition_holds():
    cfg = wl.CONFIGS["tiny"].replace(T=400, E=32, k=4)
    inp = wl.make_moe_inputs(cfg, seed=0)
    logits = wl.bf16_bits_to_f64(inp.x) @ inp.Wr.astype(np.float64)
    top = -np.sort(-logits, axis=1)[:, : cfg.k + 1]
    assert (np.diff(-top, axis=1) > wl.GAP_MIN).all()


def test_zipf_bias_gives_skewed_popularity():
    cfg = wl.CONFIGS["prefill"].replace(T=2048, H=512, n_outlier=5)
    inp = wl.make_moe_inputs(cfg, seed=0)
    ids, _, _ = oracle.router(inp.x, inp.Wr, inp.bias, cfg.k)
    shares = np.sort(wl.realised_shares(ids, cfg.E))[::-1]
    target = np.sort(wl.zipf_shares(cfg.E, cfg.zipf_s, 0, cfg.cfg_id))[::-1]
    assert abs(shares[:12].sum() - target[:12].sum()) < 0.05
    assert shares[0] > 0.15
