"""Seeded synthetic workloads for the causal LLA forward.

This module only draws inputs: it holds none of the method's arithmetic, imports neither the
CUDA binding nor the oracle, and is the one piece of code that both sides (the GPU path's tests
and bench, and the float64 oracle's tests) share.

All draws use ``torch.Generator().manual_seed(seed)`` on the CPU, in float32 unless noted, in
the order q, k, v, each shaped [B, H, T, d]. bf16 workloads are drawn in float32 and rounded
(round-to-nearest-even) to bf16; the oracle then reads the rounded values exactly.

The five workloads are the benchmark shapes of the causal LLA forward:

1. tiny: B1 H1 T128 d=dv=16, fp32, i.i.d. N(0,1), h=4, lambda=1e-2, seed 0.
2. small: B2 H4 T1024 d=dv=32, bf16, i.i.d. N(0,1), h=sqrt(32), lambda=1e-2, seed 1.
3. headline: B4 H8 T4096 d=dv=64, bf16, i.i.d. N(0,1), h=8, lambda=1e-2, seed 2.
4. stress: B1 H8 T2048 d=dv=64, fp32; per head, keys of rank 8 plus 1e-3 isotropic noise,
   shifted along the first latent direction so that half of the queries lie beyond every key;
   values an affine map of the keys plus 0.01 noise; lambda in {1e-4, 1e-2, 1} and
   h in {0.5, 1, 2} * sqrt(64); seed 3.
5. long: B1 H16 T16384 d=dv=64, bf16, i.i.d. N(0,1), h=8, lambda=1e-2, seed 4; checked
   against the oracle on 256 sampled query positions.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_iid", "make_stress", "sample_rows"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dv: int
    dtype: str            # "f32" or "bf16": the input/output element type
    seed: int
    kind: str             # "iid" or "stress"
    h: float = 0.0        # kernel bandwidth (single point)
    lam: float = 0.0      # ridge (single point)
    sweep: tuple = field(default_factory=tuple)  # ((lam, h), ...) for the stress workload
    oracle_rows: int = 0  # 0 = every row is checked; else the number of sampled rows

    @property
    def points(self):
        """(lam, h) pairs this workload is run at."""
        return self.sweep if self.sweep else ((self.lam, self.h),)

    @property
    def queries(self) -> int:
        return self.B * self.H * self.T

    def describe(self) -> str:
        return f"B{self.B} H{self.H} T{self.T} d{self.d} dv{self.dv} {self.dtype}"

    def recipe(self) -> str:
        """How the inputs are drawn, in a few words."""
        if self.kind == "stress":
            return ("rank-8 keys + 1e-3 noise, half the queries outside the key cloud, "
                    "v = A k + c + 0.01 N(0,1)")
        return "i.i.d. N(0,1) q/k/v"


WORKLOADS = {
    1: Workload("tiny", 1, 1, 128, 16, 16, "f32", 0, "iid", h=4.0, lam=1e-2),
    2: Workload("small", 2, 4, 1024, 32, 32, "bf16", 1, "iid", h=math.sqrt(32.0), lam=1e-2),
    3: Workload("headline", 4, 8, 4096, 64, 64, "bf16", 2, "iid", h=8.0, lam=1e-2),
    4: Workload("stress", 1, 8, 2048, 64, 64, "f32", 3, "stress",
                sweep=tuple((lam, f * 8.0) for lam in (1e-4, 1e-2, 1.0) for f in (0.5, 1.0, 2.0))),
    5: Workload("long", 1, 16, 16384, 64, 64, "bf16", 4, "iid", h=8.0, lam=1e-2, oracle_rows=256),
}


def _cast(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "f32":
        return x.to(torch.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def make_iid(B, H, T, d, dv, dtype, seed):
    """q, k ~ N(0,1) [B,H,T,d], v ~ N(0,1) [B,H,T,dv], drawn in that order from one generator."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, T, d, generator=g, dtype=torch.float32)
    k = torch.randn(B, H, T, d, generator=g, dtype=torch.float32)
    v = torch.randn(B, H, T, dv, generator=g, dtype=torch.float32)
    return _cast(q, dtype), _cast(k, dtype), _cast(v, dtype)


def make_probe(B, H, T, d, dtype, seed):
    """Parallax probe r ~ N(0, 1/d) [B,H,T,d] from its own generator (seed), so that r . k has
    unit variance for unit-variance keys; q, k, v of the same workload are unchanged by it."""
    g = torch.Generator().manual_seed(seed)
    r = torch.randn(B, H, T, d, generator=g, dtype=torch.float32) / math.sqrt(d)
    return _cast(r, dtype)


def make_stress(B, H, T, d, dv, dtype, seed, rank: int = 8, key_noise: float = 1e-3,
                value_noise: float = 0.01, return_u1: bool = False):
    """Ill-conditioned keys, half of the queries outside the key cloud, near-affine values.

    Per (b, h), in this draw order from one float64 generator: an orthonormal basis
    U [d, rank] (QR of a Gaussian), latent key coordinates and key noise, latent query
    coordinates and query noise, A [dv, d] ~ N(0, 1/d), c [dv] ~ N(0, 1), value noise.
    k = U g + key_noise * n; q likewise; then every key is moved along u_1 by
    median_i(q_i . u_1) - min_j(k_j . u_1), which puts half of the queries beyond all keys
    along u_1. v = A k + c + value_noise * n. With return_u1, also returns the shift directions
    u_1 [B, H, d] (float64).
    """
    g = torch.Generator().manual_seed(seed)
    f64 = torch.float64
    qs, ks, vs, us = [], [], [], []
    for _ in range(B * H):
        U, _ = torch.linalg.qr(torch.randn(d, rank, generator=g, dtype=f64))
        gk = torch.randn(T, rank, generator=g, dtype=f64)
        nk = torch.randn(T, d, generator=g, dtype=f64)
        gq = torch.randn(T, rank, generator=g, dtype=f64)
        nq = torch.randn(T, d, generator=g, dtype=f64)
        A = torch.randn(dv, d, generator=g, dtype=f64) / math.sqrt(d)
        c = torch.randn(dv, generator=g, dtype=f64)
        nv = torch.randn(T, dv, generator=g, dtype=f64)
        k = gk @ U.T + key_noise * nk
        q = gq @ U.T + key_noise * nq
        u1 = U[:, 0]
        k = k + (torch.median(q @ u1) - torch.min(k @ u1)) * u1
        v = k @ A.T + c + value_noise * nv
        qs.append(q), ks.append(k), vs.append(v), us.append(u1)
    shape = lambda xs, w: torch.stack(xs).reshape(B, H, T, w)  # noqa: E731
    out = (_cast(shape(qs, d), dtype), _cast(shape(ks, d), dtype), _cast(shape(vs, dv), dtype))
    return out + (torch.stack(us).reshape(B, H, d),) if return_u1 else out


def make_inputs(w: Workload):
    """CPU tensors (q, k, v) for a workload, in its element type."""
    if w.kind == "iid":
        return make_iid(w.B, w.H, w.T, w.d, w.dv, w.dtype, w.seed)
    if w.kind == "stress":
        return make_stress(w.B, w.H, w.T, w.d, w.dv, w.dtype, w.seed)
    raise ValueError(w.kind)


def sample_rows(BH: int, T: int, n: int, seed: int):
    """Sorted flat query indices (bh * T + i) for sampled checks.

    Always includes the first and last position of the first and last head; the rest are drawn
    without replacement, uniformly over all (bh, i), from a generator seeded with ``seed``.
    """
    total = BH * T
    if n >= total:
        return list(range(total))
    must = sorted({0, T - 1, (BH - 1) * T, total - 1})
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(total, generator=g).tolist()
    chosen = set(must)
    for r in perm:
        if len(chosen) >= n:
            break
        chosen.add(r)
    return sorted(chosen)
