"""Seeded synthetic inputs for the norm-quant and GEMM workloads.

This module only draws random numbers and shapes them into bf16 tensors on
the host.  It holds none of the method's arithmetic, so both the CUDA path
and the CPU oracle can be fed from it.

Shapes follow the MiniMax-M3 serving pages: hidden size N = H = 6144, the
o_proj contraction K = 2048 and the dense down_proj contraction K = 3072 per
tensor-parallel rank (vLLM PR #64659, "GEMM-RS microbenchmark" table: TP4,
N=6144, o_proj K=2048, down_proj K=3072, M = 128 ... 32768 tokens).  The
model and the SpeedBench prompts the pages measure with are not available, so
these seeded tensors stand in for them.

Every tensor gets its own ``torch.Generator`` seeded from (seed, tag), so a
tensor can be regenerated without drawing the others first.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HIDDEN = 6144          # N of both projections and the norm width H
K_OPROJ = 2048
K_DOWN = 3072
EPS = 1e-6
M_SWEEP = (128, 512, 768, 1024, 1536, 2048, 4096, 8192, 16384, 32768)

_TAGS = {"A": 1, "W": 2, "rowscale": 3, "x": 4, "w": 5, "outlier": 6, "zeroblk": 7}


def _gen(seed: int, tag: str, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 1_000_003 + _TAGS[tag] * 7919 + sub) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal_bf16(shape, std: float, seed: int, tag: str, sub: int = 0) -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded to bf16 (round-to-nearest-even)."""
    t = torch.randn(*shape, generator=_gen(seed, tag, sub), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def uniform_bf16(shape, lo: float, hi: float, seed: int, tag: str, sub: int = 0) -> torch.Tensor:
    t = torch.rand(*shape, generator=_gen(seed, tag, sub), dtype=torch.float32)
    return (t * (hi - lo) + lo).to(torch.bfloat16)


def log_uniform_row_scales(rows: int, lo: float, hi: float, seed: int) -> torch.Tensor:
    """Per-row multipliers exp(U(ln lo, ln hi)) (fp32), spreading the UE8M0 exponents."""
    u = torch.rand(rows, generator=_gen(seed, "rowscale"), dtype=torch.float32)
    return torch.exp(u * (math.log(hi) - math.log(lo)) + math.log(lo))


def gemm_operands(m: int, k: int, seed: int = 0, n: int = HIDDEN, a_std: float = 1.0,
                  w_std: float = 0.02, row_scales: torch.Tensor | None = None):
    """A (m x k) activations and W (n x k) weights, both bf16 row-major."""
    a = torch.randn(m, k, generator=_gen(seed, "A", k), dtype=torch.float32)
    if a_std != 1.0:
        a.mul_(a_std)
    if row_scales is not None:
        a.mul_(row_scales[:m, None])
    w = normal_bf16((n, k), w_std, seed, "W", k)
    return a.to(torch.bfloat16), w


def norm_inputs(m: int, h: int = HIDDEN, seed: int = 0, row_scales: torch.Tensor | None = None,
                outlier_frac: float = 0.0, outlier_mult: float = 50.0,
                zero_block_frac: float = 0.0, zero_first_row: bool = False):
    """x (m x h) bf16 residual rows ~ N(0,1) and the gain w (h,) bf16 ~ U(-0.1, 0.1).

    Optional stressors: a seeded set of round(outlier_frac*h) channels multiplied
    by outlier_mult; a seeded fraction of (row, 32-element block) pairs set to
    zero; row 0 set to zero.
    """
    x = torch.randn(m, h, generator=_gen(seed, "x"), dtype=torch.float32)
    if row_scales is not None:
        x.mul_(row_scales[:m, None])
    if outlier_frac > 0.0:
        n_out = round(outlier_frac * h)
        ch = torch.randperm(h, generator=_gen(seed, "outlier"))[:n_out]
        x[:, ch] *= outlier_mult
    if zero_block_frac > 0.0:
        nblk = h // 32
        total = m * nblk
        n_zero = int(total * zero_block_frac)
        pick = torch.randperm(total, generator=_gen(seed, "zeroblk"))[:n_zero]
        xb = x.view(m, nblk, 32)
        xb[pick // nblk, pick % nblk, :] = 0.0
    if zero_first_row and m > 0:
        x[0].zero_()
    w = uniform_bf16((h,), -0.1, 0.1, seed, "w")
    return x.to(torch.bfloat16), w


@dataclass
class Workload:
    """One named configuration: GEMM shapes plus the norm-quant shape."""
    name: str
    m: int
    ks: tuple
    norm_rows: int
    row_scales: bool = False
    stress: bool = False
    n: int = HIDDEN
    h: int = HIDDEN
    eps: float = EPS
    notes: str = ""
    extra: dict = field(default_factory=dict)

    def gemm(self, k: int, seed: int = 0):
        rs = log_uniform_row_scales(self.m, 0.1, 10.0, seed) if self.row_scales else None
        return gemm_operands(self.m, k, seed, n=self.n, row_scales=rs)

    def norm(self, seed: int = 0):
        rs = log_uniform_row_scales(self.norm_rows, 0.1, 10.0, seed) if self.row_scales else None
        if self.stress:
            return norm_inputs(self.norm_rows, self.h, seed, outlier_frac=0.01, outlier_mult=50.0,
                               zero_block_frac=1.0 / 128.0, zero_first_row=True)
        return norm_inputs(self.norm_rows, self.h, seed, row_scales=rs)


WORKLOADS = {
    "m128": Workload("m128", 128, (K_OPROJ,), 128,
                     notes="o_proj at 128 tokens; norm-quant 128x6144"),
    "m1024": Workload("m1024", 1024, (K_OPROJ, K_DOWN), 1024,
                      notes="o_proj and down_proj at 1024 tokens; norm-quant 1024x6144"),
    "m4096_rowscale": Workload("m4096_rowscale", 4096, (K_OPROJ, K_DOWN), 4096, row_scales=True,
                               notes="rows scaled by LogUniform(0.1, 10) to spread UE8M0 exponents"),
    "m32768_stress": Workload("m32768_stress", 32768, (K_DOWN,), 32768, stress=True,
                              notes="down_proj at 32768 tokens; norm-quant with 61 outlier channels "
                                    "x50, 1/128 of 32-blocks zero, row 0 zero"),
}


def sweep_workload(m: int, k: int) -> Workload:
    return Workload(f"sweep_m{m}_k{k}", m, (k,), m, notes="M sweep, plain N(0,1) activations")


def get_workload(name: str) -> Workload:
    """A named workload, or sweep_m<M>_k<K> for a point of the M x K sweep."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("sweep_m") and "_k" in name:
        m, k = name[len("sweep_m"):].split("_k")
        return sweep_workload(int(m), int(k))
    raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)} or sweep_m<M>_k<K>")
