"""Seeded synthetic inputs for the GPTQ fold + q4tp sweep.

This module only draws inputs; it holds none of the method's arithmetic.
Both the CUDA path (tests, bench) and the oracle consume the bytes it
returns, so a parity check always compares the two on identical inputs.

Workload shapes follow the fold/sweep pages' own workload (one Hessian group
of a 27B model's ``down_proj``: n = 17408 input channels, 5120 rows), plus
smaller groups of the same structure:

* ``X`` [n, T] ~ N(0, 1), each channel (row) scaled by a lognormal(0, sigma)
  factor; a few outlier channels are multiplied by 100 (about 10^4 x energy)
  and a few dead channels are zero rows (they never fire);
* ``H = X X^T / T`` in f32, stored as the upper triangle by rows
  (``n (n + 1) / 2`` floats; row r starts at ``r (2n - r + 1) / 2``);
* ``W`` [rows, n] ~ N(0, w_std^2) in f32.

Randomness comes from ``torch.Generator`` seeded per tensor, on the device
the caller asks for, so a CUDA run and a CPU run of the same seed draw
different (but each reproducible) numbers; every comparison feeds the same
drawn bytes to both sides.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Config:
    name: str
    n: int
    rows: int
    T: int
    w_std: float
    sigma: float
    n_outlier: int
    n_dead: int
    lam: float = 0.01
    seed: int = 0


CONFIGS = {
    "tiny": Config("tiny", 256, 64, 1024, 0.02, 1.0, 2, 2),
    "n4096": Config("n4096", 4096, 4096, 8192, 0.02, 1.0, 8, 4),
    "n14336": Config("n14336", 14336, 4096, 16384, 0.02, 1.5, 32, 16),
    "n17408": Config("n17408", 17408, 5120, 32768, 0.015, 1.5, 64, 16),
}


def config(name: str, **kw) -> Config:
    """A named workload, optionally with fields replaced (seed, T, n, ...)."""
    return replace(CONFIGS[name], **kw)


def rank_deficient(cfg: Config) -> Config:
    """The same group drawn from T = n/2 samples: H has rank n/2, so the
    undamped Hessian is singular (drives the damping-retry path)."""
    return replace(cfg, T=max(1, cfg.n // 2), name=cfg.name + "_rankdef")


def _gen(device, seed: int, salt: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + salt)
    return g


def channel_plan(cfg: Config, device="cpu"):
    """Per-channel scale, outlier and dead index sets (drawn without replacement)."""
    g = _gen("cpu", cfg.seed, 1)
    perm = torch.randperm(cfg.n, generator=g)
    dead = perm[: cfg.n_dead].sort().values
    outl = perm[cfg.n_dead : cfg.n_dead + cfg.n_outlier].sort().values
    scale = torch.exp(cfg.sigma * torch.randn(cfg.n, generator=g, dtype=torch.float64)).to(torch.float32)
    scale[outl] *= 100.0
    scale[dead] = 0.0
    return scale.to(device), outl.to(device), dead.to(device)


def make_x(cfg: Config, device="cpu") -> torch.Tensor:
    scale, _, _ = channel_plan(cfg, device)
    g = _gen(device, cfg.seed, 2)
    x = torch.randn(cfg.n, cfg.T, generator=g, device=device, dtype=torch.float32)
    x.mul_(scale[:, None])
    return x


def make_h(cfg: Config, device="cpu") -> torch.Tensor:
    """Dense f32 H = X X^T / T (symmetric, n x n)."""
    x = make_x(cfg, device)
    prev = None
    if x.is_cuda:
        prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False
    try:
        h = (x @ x.T).div_(float(cfg.T))
    finally:
        if prev is not None:
            torch.backends.cuda.matmul.allow_tf32 = prev
    del x
    return h


def pack_upper(h: torch.Tensor) -> torch.Tensor:
    """Upper triangle of a square matrix by rows: (0,0..n-1), (1,1..n-1), ..."""
    n = h.shape[0]
    out = torch.empty(n * (n + 1) // 2, dtype=h.dtype, device=h.device)
    off = 0
    for r in range(n):
        out[off : off + n - r] = h[r, r:]
        off += n - r
    return out


def make_h_packed(cfg: Config, device="cpu") -> torch.Tensor:
    return pack_upper(make_h(cfg, device)).contiguous()


def make_w(cfg: Config, device="cpu") -> torch.Tensor:
    g = _gen(device, cfg.seed, 3)
    w = torch.randn(cfg.rows, cfg.n, generator=g, device=device, dtype=torch.float32)
    return w.mul_(cfg.w_std)


def make_problem(cfg: Config, device="cpu"):
    """(H_packed f32 [n(n+1)/2], W f32 [rows, n]) for one group."""
    return make_h_packed(cfg, device), make_w(cfg, device)
