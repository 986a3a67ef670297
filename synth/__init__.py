"""Seeded synthetic KV inputs.

This module only draws random numbers.  It holds none of the cache's
arithmetic (no projection, quantisation, packing or fitting), so that the
float64 oracle and the GPU path can both consume the very same inputs
without sharing any code of the method.

The recipe follows the workloads of the projected-and-quantized KV cache:

* spectral rows  x_t = mu + sum_k sigma_k g_{t,k} u_k + 0.01 eps_t with
  mu ~ N(0, 0.5^2), U = Q of the QR of a seeded Gaussian matrix,
  sigma_k = k^(-alpha), g, eps ~ N(0, 1);
* optional outlier channels: a seeded ~2 % of the channels scaled by 8
  after generation;
* Gaussian keys whose coordinates are, with probability 1 %, replaced by a
  Student-t (nu = 3) draw.

Every generator is a pure function of ``(seed, key...)`` through
``torch.Generator`` seeded from ``numpy.random.SeedSequence``.  The same
call on the same device gives the same numbers; CPU and CUDA streams differ
(tests generate on the CPU and copy to the GPU).
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "make_generator",
    "spectral_basis",
    "spectral_rows",
    "outlier_channels",
    "kv_spectral",
    "group_spectral",
    "heavy_tailed_keys",
    "to_dtype",
]

_DTYPES = {
    "f32": torch.float32,
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "f64": torch.float64,
}


def make_generator(seed: int, *key: int, device="cpu") -> torch.Generator:
    """A torch generator whose state depends only on ``(seed, *key)``."""
    ss = np.random.SeedSequence([int(seed)] + [int(k) for k in key])
    g = torch.Generator(device=device)
    g.manual_seed(int(ss.generate_state(1, dtype=np.uint64)[0] & 0x7FFF_FFFF_FFFF_FFFF))
    return g


def spectral_basis(d_in: int, gen: torch.Generator, device="cpu", dtype=torch.float64):
    """Draw (mu, U): mu ~ N(0, 0.5^2) and an orthogonal U from a QR factorisation."""
    mu = 0.5 * torch.randn(d_in, generator=gen, device=device, dtype=dtype)
    g = torch.randn(d_in, d_in, generator=gen, device=device, dtype=dtype)
    q, _ = torch.linalg.qr(g.cpu())        # small factorisation on the host
    return mu, q.to(device)


def spectral_rows(mu, U, n: int, alpha: float, gen: torch.Generator, noise: float = 0.01):
    """n rows of mu + sum_k k^-alpha g_k u_k + noise * eps (same device/dtype as U)."""
    d_in = U.shape[0]
    k = torch.arange(1, d_in + 1, device=U.device, dtype=U.dtype)
    sigma = k.pow(-alpha)
    g = torch.randn(n, d_in, generator=gen, device=U.device, dtype=U.dtype)
    eps = torch.randn(n, d_in, generator=gen, device=U.device, dtype=U.dtype)
    return mu + (g * sigma) @ U.T + noise * eps


def outlier_channels(d_in: int, count: int, gen: torch.Generator) -> torch.Tensor:
    """A seeded choice of ``count`` distinct channels (sorted)."""
    perm = torch.randperm(d_in, generator=gen)
    return torch.sort(perm[:count]).values


def to_dtype(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(_DTYPES[dtype])


def kv_spectral(B: int, H: int, S: int, D: int, alpha: float, seed: int, tensor: int,
                n_outliers: int = 0, dtype: str = "f32", device="cpu",
                work_dtype=torch.float64) -> torch.Tensor:
    """[B, H, S, D] rows; each (b, h) has its own (mu, U) and outlier channels.

    ``tensor`` separates K (0) from V (1).
    """
    out = torch.empty(B, H, S, D, dtype=_DTYPES[dtype], device=device)
    for b in range(B):
        for h in range(H):
            gen = make_generator(seed, tensor, b, h, device=device)
            mu, U = spectral_basis(D, gen, device=device, dtype=work_dtype)
            x = spectral_rows(mu, U, S, alpha, gen)
            if n_outliers:
                cgen = make_generator(seed, tensor, b, h, 7919)
                ch = outlier_channels(D, n_outliers, cgen).to(device)
                x[:, ch] *= 8.0
            out[b, h] = x.to(out.dtype)
    return out


def group_spectral(B: int, H: int, S: int, D: int, heads_per_group: int, alpha: float,
                   seed: int, tensor: int, n_outliers: int = 0, dtype: str = "bf16",
                   device="cpu", work_dtype=torch.float64) -> torch.Tensor:
    """[B, H, S, D] rows where each head group's concatenated row (D_in =
    heads_per_group * D) comes from one D_in-dimensional spectral model that
    every batch entry of the group shares (independent draws per batch)."""
    assert H % heads_per_group == 0
    d_in = heads_per_group * D
    out = torch.empty(B, H, S, D, dtype=_DTYPES[dtype], device=device)
    for g in range(H // heads_per_group):
        bgen = make_generator(seed, tensor, g, device=device)
        mu, U = spectral_basis(d_in, bgen, device=device, dtype=work_dtype)
        ch = None
        if n_outliers:
            ch = outlier_channels(d_in, n_outliers, make_generator(seed, tensor, g, 7919)).to(device)
        for b in range(B):
            gen = make_generator(seed, tensor, g, b + 1, device=device)
            x = spectral_rows(mu, U, S, alpha, gen)
            if ch is not None:
                x[:, ch] *= 8.0
            x = x.view(S, heads_per_group, D).permute(1, 0, 2)
            out[b, g * heads_per_group:(g + 1) * heads_per_group] = x.to(out.dtype)
    return out


def heavy_tailed_keys(B: int, H: int, S: int, D: int, seed: int, p_heavy: float = 0.01,
                      nu: float = 3.0, dtype: str = "f16", device="cpu",
                      work_dtype=torch.float32) -> torch.Tensor:
    """[B, H, S, D] N(0, 1) entries, each replaced with probability ``p_heavy``
    by a Student-t(nu) draw (t = N / sqrt(Chi2_nu / nu))."""
    out = torch.empty(B, H, S, D, dtype=_DTYPES[dtype], device=device)
    for b in range(B):
        gen = make_generator(seed, 2, b, device=device)
        n = torch.randn(H, S, D, generator=gen, device=device, dtype=work_dtype)
        z = torch.randn(H, S, D, generator=gen, device=device, dtype=work_dtype)
        chi2 = torch.zeros_like(z)
        for _ in range(int(nu)):
            chi2 += torch.randn(H, S, D, generator=gen, device=device, dtype=work_dtype) ** 2
        t = z / torch.sqrt(chi2 / nu)
        pick = torch.rand(H, S, D, generator=gen, device=device, dtype=work_dtype) < p_heavy
        out[b] = torch.where(pick, t, n).to(out.dtype)
    return out
