"""Seeded synthetic workloads for the W8A8 MoE layer.

This module only draws random inputs; it holds none of the method's
arithmetic (no quantisation, no expert GEMM, no epilogue, no combine).  The
tests, the benchmark and the smoke check take their inputs from here, for the
CUDA library and for the CPU oracle alike.

Recipes (shapes and distributions of the layer's workloads):

* activations ``x``: bf16, i.i.d. N(0, 1), with 1 % of the hidden channels
  (2 channels in the tiny layer) multiplied by 20 to model activation
  outliers ("a few dimensions far above the rest": "DeepSeek V4 950 FP8
  inference on H100", section 4.2);
* expert weights: fp32 N(0, 0.02^2), later quantised per output channel;
* router weights ``Wr`` [H, E]: N(0, 0.02^2) for the tiny layer, otherwise
  N(0, sigma^2) with sigma = 1/sqrt(sum_h var(x_h)) so that the routing
  logits are roughly N(0, 1);
* router bias: none (tiny, decode), a fitted bias that makes expert
  popularity follow Zipf(s) over a random ranking of the experts, fitted on
  the binary64 logits of the drawn activations (prefill),
  or N(0, 0.5^2) per expert (wide);
* the top-k gap condition: every token's k+1 largest logits (computed here
  in binary64 with numpy's matmul, purely to condition the draw) differ
  pairwise by more than 1e-3; offending token rows are redrawn, so that the
  choice of experts cannot depend on binary32 summation order.

Random streams: ``numpy.random.default_rng([seed, config id, tensor id,
sub-stream])`` for host tensors, and one seeded ``torch.Generator`` per
expert tensor (on the device that holds it) for expert weights.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GAP_MIN = 1e-3
OUTLIER_GAIN = 20.0
EXPERT_W_STD = 0.02

# tensor ids of the random streams
_T_X, _T_OUTL, _T_WR, _T_BIAS, _T_W13, _T_W2, _T_REDRAW, _T_ZIPF, _T_LIN_W, _T_SMOOTH = range(10)


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    cfg_id: int
    T: int
    H: int
    I: int
    E: int
    k: int
    n_outlier: int
    router_std: Optional[float]  # None: 1/sqrt(sum of channel variances)
    bias: str = "none"  # "none" | "zipf" | "normal"
    zipf_s: float = 0.0
    bias_std: float = 0.0

    @property
    def S(self) -> int:
        return self.T * self.k

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class LinearConfig:
    name: str
    cfg_id: int
    M: int
    K: int
    N: int
    n_outlier: int


CONFIGS = {
    "tiny": MoEConfig("tiny", 1, T=16, H=256, I=512, E=8, k=2, n_outlier=2, router_std=0.02),
    "decode": MoEConfig("decode", 3, T=64, H=4096, I=1536, E=64, k=2, n_outlier=41, router_std=None),
    "prefill": MoEConfig("prefill", 4, T=8192, H=4096, I=1536, E=64, k=2, n_outlier=41,
                         router_std=None, bias="zipf", zipf_s=1.2),
    "wide": MoEConfig("wide", 5, T=4096, H=7168, I=2048, E=256, k=8, n_outlier=72,
                      router_std=None, bias="normal", bias_std=0.5),
}
LINEAR = LinearConfig("linear", 2, M=4096, K=4096, N=4096, n_outlier=41)


def rng(seed: int, cfg_id: int, tensor_id: int, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, cfg_id, tensor_id, sub])


def _to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 draws to bf16 (torch's conversion) and return the bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to binary64 (exact: bf16 is the top half of a binary32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def outlier_channels(seed: int, cfg_id: int, H: int, n_outlier: int) -> np.ndarray:
    return np.sort(rng(seed, cfg_id, _T_OUTL).choice(H, size=n_outlier, replace=False))


def draw_activations(seed: int, cfg_id: int, T: int, H: int, n_outlier: int, sub: int = 0) -> np.ndarray:
    """bf16 bits [T, H]: N(0,1) with the outlier channels scaled by 20."""
    x = rng(seed, cfg_id, _T_X, sub).standard_normal((T, H), dtype=np.float32)
    x[:, outlier_channels(seed, cfg_id, H, n_outlier)] *= OUTLIER_GAIN
    return _to_bf16_bits(x)


def router_sigma(cfg: MoEConfig) -> float:
    if cfg.router_std is not None:
        return cfg.router_std
    var = (cfg.H - cfg.n_outlier) * 1.0 + cfg.n_outlier * OUTLIER_GAIN ** 2
    return float(1.0 / np.sqrt(var))


def zipf_shares(E: int, s: float, seed: int, cfg_id: int) -> np.ndarray:
    """Target share of assignments per expert: Zipf(s) over a random ranking."""
    p = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    perm = rng(seed, cfg_id, _T_ZIPF).permutation(E)
    shares = np.empty(E)
    shares[perm] = p
    return shares


def fit_zipf_bias(logits: np.ndarray, k: int, shares: np.ndarray, iters: int = 300,
                  eta: float = 0.1) -> np.ndarray:
    """Bias b with which the top-k of ``logits + b`` (the binary64 router
    logits of the drawn activations, one row per token) picks expert e with a
    share close to ``shares[e]``: damped fixed-point iteration
    b <- b + eta * (log target - log realised), keeping the best iterate."""
    n, E = logits.shape
    b = np.zeros(E)
    target = np.log(shares)
    best_err, best_b = np.inf, b.copy()
    for _ in range(iters):
        top = np.argpartition(-(logits + b), k - 1, axis=1)[:, :k]
        realised = np.maximum(np.bincount(top.ravel(), minlength=E), 0.5) / (n * k)
        err = np.abs(realised - shares).sum()
        if err < best_err:
            best_err, best_b = err, b.copy()
        b += eta * (target - np.log(realised))
        b -= b.mean()
    return best_b.astype(np.float32)


def _bad_gap_rows(x_bits: np.ndarray, Wr: np.ndarray, bias: Optional[np.ndarray], k: int) -> np.ndarray:
    logits = bf16_bits_to_f64(x_bits) @ Wr.astype(np.float64)
    if bias is not None:
        logits += bias.astype(np.float64)
    top = -np.sort(-logits, axis=1)[:, : k + 1]
    gaps = top[:, :-1] - top[:, 1:]
    return np.nonzero((gaps <= GAP_MIN).any(axis=1))[0]


@dataclasses.dataclass
class MoEInputs:
    cfg: MoEConfig
    x: np.ndarray  # bf16 bits [T, H]
    Wr: np.ndarray  # fp32 [H, E]
    bias: Optional[np.ndarray]  # fp32 [E] or None
    redrawn_rows: int
    seed: int


def make_moe_inputs(cfg: MoEConfig, seed: int = 0) -> MoEInputs:
    """Activations, router weights and bias for ``cfg``, with the gap condition enforced."""
    x = draw_activations(seed, cfg.cfg_id, cfg.T, cfg.H, cfg.n_outlier)
    Wr = (rng(seed, cfg.cfg_id, _T_WR).standard_normal((cfg.H, cfg.E), dtype=np.float32)
          * np.float32(router_sigma(cfg))).astype(np.float32)
    if cfg.bias == "none":
        bias = None
    elif cfg.bias == "normal":
        bias = (rng(seed, cfg.cfg_id, _T_BIAS).standard_normal(cfg.E) * cfg.bias_std).astype(np.float32)
    elif cfg.bias == "zipf":
        logits = bf16_bits_to_f64(x) @ Wr.astype(np.float64)
        bias = fit_zipf_bias(logits, cfg.k, zipf_shares(cfg.E, cfg.zipf_s, seed, cfg.cfg_id))
    else:
        raise ValueError(cfg.bias)
    outl = outlier_channels(seed, cfg.cfg_id, cfg.H, cfg.n_outlier)
    redrawn = 0
    bad = _bad_gap_rows(x, Wr, bias, cfg.k)
    sub = 0
    while bad.size:
        sub += 1
        if sub > 1000:
            raise RuntimeError("gap condition not met after 1000 redraw rounds")
        fresh = rng(seed, cfg.cfg_id, _T_REDRAW, sub).standard_normal((bad.size, cfg.H), dtype=np.float32)
        fresh[:, outl] *= OUTLIER_GAIN
        x[bad] = _to_bf16_bits(fresh)
        redrawn += bad.size
        bad = bad[_bad_gap_rows(x[bad], Wr, bias, cfg.k)]
    return MoEInputs(cfg, x, Wr, bias, redrawn, seed)


def expert_weight_seed(seed: int, cfg_id: int, which: str, e: int) -> int:
    tid = {"w13": _T_W13, "w2": _T_W2, "linear": _T_LIN_W}[which]
    return int(np.random.SeedSequence([seed, cfg_id, tid, e]).generate_state(1, np.uint64)[0] >> 1)


def expert_weight_fp32(cfg, which: str, e: int, seed: int = 0, device="cpu"):
    """fp32 torch tensor of one expert: w13 [2I, H] (gate rows then up rows),
    w2 [H, I]; for the linear config ``which='linear'`` gives w [N, K]."""
    import torch
    if which == "w13":
        shape = (2 * cfg.I, cfg.H)
    elif which == "w2":
        shape = (cfg.H, cfg.I)
    elif which == "linear":
        shape = (cfg.N, cfg.K)
    else:
        raise ValueError(which)
    g = torch.Generator(device=device)
    g.manual_seed(expert_weight_seed(seed, cfg.cfg_id, which, e))
    w = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return w.mul_(EXPERT_W_STD)


def smoothing_factors(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    """Per-expert, per-channel smoothing factors [E, H] for the layer with
    SmoothQuant-folded activations: log-uniform on [e^-1.5, e^1.5], seeded.
    (Calibrated factors need activation statistics of a trained model; these
    stand in for them.)"""
    r = rng(seed, cfg.cfg_id, _T_SMOOTH)
    return np.exp(r.uniform(-1.5, 1.5, (cfg.E, cfg.H))).astype(np.float32)


def linear_activations(cfg: LinearConfig, seed: int = 0) -> np.ndarray:
    return draw_activations(seed, cfg.cfg_id, cfg.M, cfg.K, cfg.n_outlier)


def realised_shares(topk_ids: np.ndarray, E: int) -> np.ndarray:
    counts = np.bincount(np.asarray(topk_ids).ravel(), minlength=E)
    return counts / counts.sum()
