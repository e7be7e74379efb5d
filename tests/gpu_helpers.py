"""Shared helpers of the GPU parity tests: moving seeded inputs to the device,
running the oracle on the same inputs, and the float tolerances."""
import contextlib

import numpy as np
import torch

import oracle
from w8a8_quantised_moe_gb300 import workloads as wl

# Output tolerance of the layer: max |y - y_oracle| <= 1e-2 * max |y_oracle|
# and sum |y - y_oracle| / sum |y_oracle| <= 2e-3.
Y_MAX_REL = 1e-2
Y_MEAN_REL = 2e-3
# h differs from the oracle only through expf (CUDA: <= 2 ulp; glibc: < 1 ulp)
# feeding one division and one multiply: a few ulp of binary32.
H_RTOL = 2e-6
# Router top-k weights: the GPU accumulates each logit (H products, exact on
# the tensor cores) in binary32 in a fixed order; the oracle sums in binary64
# and rounds once.  At H = 4096-7168 the logits differ by up to ~1e-5, and a
# softmax weight moves by at most a quarter of that.
TOPK_W_ATOL = 1e-5


@contextlib.contextmanager
def gemm_path(name: str):
    """Force the library's GEMM kernel ("auto", "skinny", "narrow", "mid",
    "wide", "pair") inside the block; the automatic choice afterwards."""
    import w8a8_quantised_moe_gb300 as moe
    moe.set_gemm_path(name)
    try:
        yield
    finally:
        moe.set_gemm_path("auto")


def bf16_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_from_dev(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def y_errors(y_bits: np.ndarray, y_ref_bits: np.ndarray):
    y = bits_to_f32(y_bits).astype(np.float64)
    r = bits_to_f32(y_ref_bits).astype(np.float64)
    max_err = np.abs(y - r).max() if y.size else 0.0
    max_ref = np.abs(r).max() if r.size else 0.0
    mean_rel = np.abs(y - r).sum() / max(np.abs(r).sum(), 1e-30)
    return max_err, max_ref, mean_rel


def assert_y_close(y_bits, y_ref_bits):
    max_err, max_ref, mean_rel = y_errors(y_bits, y_ref_bits)
    assert max_err <= Y_MAX_REL * max_ref, (max_err, max_ref)
    assert mean_rel <= Y_MEAN_REL, mean_rel


class Layer:
    """Seeded inputs of one layer shape: host copies for the oracle, device
    copies for the library.  Expert weights are drawn in fp32 and quantised
    by the oracle; the device gets the oracle's int8 weights and scales."""

    def __init__(self, cfg: wl.MoEConfig, seed: int = 0, weights=None):
        self.cfg = cfg
        inp = wl.make_moe_inputs(cfg, seed)
        self.x, self.Wr, self.bias = inp.x, inp.Wr, inp.bias
        if weights is None:
            w13 = np.stack([wl.expert_weight_fp32(cfg, "w13", e, seed).numpy() for e in range(cfg.E)])
            w2 = np.stack([wl.expert_weight_fp32(cfg, "w2", e, seed).numpy() for e in range(cfg.E)])
            q13, s13 = oracle.quantize_rows(w13.reshape(-1, cfg.H))
            q2, s2 = oracle.quantize_rows(w2.reshape(-1, cfg.I))
            weights = (q13.reshape(cfg.E, 2 * cfg.I, cfg.H), s13.reshape(cfg.E, 2 * cfg.I),
                       q2.reshape(cfg.E, cfg.H, cfg.I), s2.reshape(cfg.E, cfg.H))
        self.w13_q, self.s13, self.w2_q, self.s2 = weights
        self.d_x = bf16_to_dev(self.x)
        self.d_Wr = torch.from_numpy(self.Wr).cuda()
        self.d_bias = None if self.bias is None else torch.from_numpy(self.bias).cuda()
        self.d_w13 = torch.from_numpy(self.w13_q).cuda()
        self.d_s13 = torch.from_numpy(self.s13).cuda()
        self.d_w2 = torch.from_numpy(self.w2_q).cuda()
        self.d_s2 = torch.from_numpy(self.s2).cuda()

    def device_args(self):
        return (self.d_x, self.d_Wr, self.d_bias, self.d_w13, self.d_s13, self.d_w2, self.d_s2, self.cfg.k)

    def oracle(self, dump=()):
        return oracle.moe_forward(self.x, self.Wr, self.bias, self.w13_q, self.s13, self.w2_q, self.s2,
                                  self.cfg.k, dump=dump)
