"""Seeded synthetic inputs shared by the oracle-side and GPU-side tests and the benchmark.

This module holds no arithmetic of the Relation operator: it only draws
Gaussian tensors from a fixed seed, scales them, and rounds them to the
requested storage dtype.  Both sides of a parity check get the same rounded
tensors (the oracle upcasts them exactly to float64).

Recipe (workloads of the paper's models: head width 48-128, T 128-16384,
B*H independent heads): tensors are [B, H, T, d], drawn in float32 on the CPU
with ``torch.Generator().manual_seed(seed)`` and ``torch.randn``, multiplied by
``scale``, then rounded to nearest-even bf16 when dtype is bf16.  Default seeds
42/43/44/45 for P1/P2/V/dY (42 is the first of the paper's paired seeds).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEEDS = {"P1": 42, "P2": 43, "V": 44, "dY": 45}


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype, Self temperature, count coefficient."""

    name: str
    B: int
    H: int
    T: int
    d: int
    dtype: torch.dtype
    tau_S: float
    lam: float
    causal: bool = True
    p_scale: float = 1.0  # multiplies P1 and P2
    backward: bool = False
    seeds: dict = field(default_factory=lambda: dict(SEEDS))


def gaussian(shape, seed: int, scale: float = 1.0, dtype: torch.dtype = torch.float32) -> torch.Tensor:
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(dtype)


def make(w: Workload, with_dy: bool | None = None) -> dict:
    """CPU tensors P1, P2, V (and dY when backward) for workload ``w``."""
    shape = (w.B, w.H, w.T, w.d)
    out = {
        "P1": gaussian(shape, w.seeds["P1"], w.p_scale, w.dtype),
        "P2": gaussian(shape, w.seeds["P2"], w.p_scale, w.dtype),
        "V": gaussian(shape, w.seeds["V"], 1.0, w.dtype),
    }
    if with_dy if with_dy is not None else w.backward:
        out["dY"] = gaussian(shape, w.seeds["dY"], 1.0, w.dtype)
    return out


# The five workloads: single-head fp32 (T=128, d=64); the 10M-decoder forward
# (B8 H8 T1024 d64); the large-|U| forward (P1,P2 ~ N(0,1) * 3 / d^(1/4), tau 0.5);
# forward+backward at B8 H12 T2048 d64; long context B1 H32 T16384 d128.
# lambda = 0.5 is the paper's initial value of the per-layer count coefficient.
WORKLOADS = {
    "single_head_fp32": Workload("single_head_fp32", 1, 1, 128, 64, torch.float32, 1.0, 0.5),
    "mhr_fwd_T1024": Workload("mhr_fwd_T1024", 8, 8, 1024, 64, torch.bfloat16, 1.0, 0.5),
    "mhr_fwd_T4096_large_u": Workload("mhr_fwd_T4096_large_u", 4, 16, 4096, 64, torch.bfloat16, 0.5, 0.5,
                                      p_scale=3.0 / 64 ** 0.25),
    "mhr_fwd_bwd_T2048": Workload("mhr_fwd_bwd_T2048", 8, 12, 2048, 64, torch.bfloat16, 1.0, 0.5, backward=True),
    "mhr_fwd_bwd_T16384_d128": Workload("mhr_fwd_bwd_T16384_d128", 1, 32, 16384, 128, torch.bfloat16, 1.0, 0.5,
                                        backward=True),
    # The paper's other model widths ("Ask Self, Ask Others", Table 2: 8 heads of 48 at
    # T=1024, 8 of 80 at T=4096; Appendix F.1: the Hybrid model's 8 heads of 60 at
    # T=2048), forward+backward with the paper's tau_S = 2 and lambda = 0.5.
    "paper_d48_T1024": Workload("paper_d48_T1024", 16, 8, 1024, 48, torch.bfloat16, 2.0, 0.5, backward=True),
    "paper_d60_T2048": Workload("paper_d60_T2048", 16, 8, 2048, 60, torch.bfloat16, 2.0, 0.5, backward=True),
    "paper_d80_T4096": Workload("paper_d80_T4096", 4, 8, 4096, 80, torch.bfloat16, 2.0, 0.5, backward=True),
    # The headline shape: the large-|U| forward workload run forward+backward.
    "mhr_fwd_bwd_T4096": Workload("mhr_fwd_bwd_T4096", 4, 16, 4096, 64, torch.bfloat16, 0.5, 0.5,
                                  p_scale=3.0 / 64 ** 0.25, backward=True),
}


# ---------------------------------------------------------------- Linear Relation
# Inputs of Linear Relation ("Ask Self, Ask Others", Sec. 5.2): P1, P2, I~ as above
# (bf16) plus the float32 log-retention G <= 0.  G is drawn with the statistics of its
# parameterisation at initialisation (eq.(16), the caller's projection, not part of the
# operator): g = -a * softplus(0.5 z + b) with a ~ U(1, 16) per (head, channel),
# softplus(b) log-uniform in [1e-3, 1e-1] per (head, channel), z ~ N(0, 1) per entry;
# ``g_scale`` multiplies the result (strong or weak retention cases).
LINEAR_G_SEED = 46


@dataclass(frozen=True)
class LinearWorkload:
    name: str
    B: int
    H: int
    T: int
    d: int
    tau_S: float = 2.0
    g_scale: float = 1.0
    backward: bool = False


def linear_retention(B: int, H: int, T: int, d: int, seed: int = LINEAR_G_SEED, g_scale: float = 1.0) -> torch.Tensor:
    g = torch.Generator().manual_seed(int(seed))
    a = 1.0 + 15.0 * torch.rand(1, H, 1, d, generator=g)
    sp_b = torch.exp(torch.empty(1, H, 1, d).uniform_(float(torch.log(torch.tensor(1e-3))),
                                                     float(torch.log(torch.tensor(1e-1))), generator=g))
    b = torch.log(torch.expm1(sp_b))  # inverse softplus
    z = torch.randn(B, H, T, d, generator=g)
    return (-g_scale * a * torch.nn.functional.softplus(0.5 * z + b)).to(torch.float32)


def linear_gate_inputs(B: int, H: int, T: int, d: int, seed: int = LINEAR_G_SEED, g_scale: float = 1.0):
    """The draws behind linear_retention() as the inputs of the KDA-style gate: the per-token
    projection output R = z / 2 [B, H, T, d] and the per-head channel parameters
    A_log = log(g_scale * a), dt_bias = b [H, d] (float32), so that
    -exp(A_log) * softplus(R + dt_bias) reproduces linear_retention() with the same seed."""
    g = torch.Generator().manual_seed(int(seed))
    a = 1.0 + 15.0 * torch.rand(1, H, 1, d, generator=g)
    sp_b = torch.exp(torch.empty(1, H, 1, d).uniform_(float(torch.log(torch.tensor(1e-3))),
                                                     float(torch.log(torch.tensor(1e-1))), generator=g))
    b = torch.log(torch.expm1(sp_b))
    z = torch.randn(B, H, T, d, generator=g)
    return ((0.5 * z).to(torch.float32), torch.log(g_scale * a).reshape(H, d).to(torch.float32),
            b.reshape(H, d).to(torch.float32))


def make_linear(w: LinearWorkload) -> dict:
    """CPU tensors P1, P2, I (bf16), G (float32) and, when backward, dY (bf16); [B, H, T, d]."""
    shape = (w.B, w.H, w.T, w.d)
    out = {
        "P1": gaussian(shape, SEEDS["P1"], 1.0, torch.bfloat16),
        "P2": gaussian(shape, SEEDS["P2"], 1.0, torch.bfloat16),
        "I": gaussian(shape, SEEDS["V"], 1.0, torch.bfloat16),
        "G": linear_retention(w.B, w.H, w.T, w.d, g_scale=w.g_scale),
    }
    if w.backward:
        out["dY"] = gaussian(shape, SEEDS["dY"], 1.0, torch.bfloat16)
    return out


# The Hybrid model's Linear Relation layers (Appendix F.1: 8 heads of width 60, T = 2048,
# micro-batch 16) and the longest context its long-context runs pass (Appendix I.2,
# Table 28: T = 32768, micro-batch 1).
LINEAR_WORKLOADS = {
    "linear_d60_T2048": LinearWorkload("linear_d60_T2048", 16, 8, 2048, 60, backward=True),
    "linear_d60_T32768": LinearWorkload("linear_d60_T32768", 1, 8, 32768, 60, backward=True),
}
