"""Prefill calibration: fit the frozen layer parameters from prefill rows.

This runs once per layer before the hot path (the kvtc_cache page fits the
local PCA basis and the bit allocation on the first call and freezes them;
the palu_cache page fits one projection per head group at prefill).  The
per-(b, h) uniform fit runs on the GPU in libkvc (kvc_fit_uniform); the
shared and head-group fits, whose pooled rows reach D_in = 1024, use PyTorch
linear algebra in float64.  The hot path itself (append / fetch) runs only in
libkvc's kernels.

    params = fit_uniform(x[:, :, :512], r=32, choices=(0, 2, 4, 8), budget=128)
    layer = KVCacheLayer("uniform", B, H, D, capacity=S, **params)
"""
from __future__ import annotations

import math

import numpy as np
import torch

__all__ = ["pca", "fit_uniform", "fit_uniform_shared", "fit_group",
           "rotation", "gaussian_codebook"]


def pca(rows: torch.Tensor):
    """Batched PCA of rows [N, S, D_in] -> (mean [N, D_in], eigenvalues [N, D_in]
    descending, eigenvectors [N, D_in, D_in] as columns), float64.  Signs are
    fixed so that each vector's largest-magnitude entry is positive."""
    X = rows.to(torch.float64)
    mean = X.mean(dim=1)
    Xc = X - mean[:, None, :]
    C = Xc.transpose(1, 2) @ Xc / X.shape[1]
    lam, U = torch.linalg.eigh(C.cpu())      # small symmetric eigenproblems, on the host
    lam, U = lam.to(X.device), U.to(X.device)
    lam, U = lam.flip(-1), U.flip(-1)
    piv = U.abs().argmax(dim=1, keepdim=True)
    sign = torch.sign(torch.gather(U, 1, piv))
    sign[sign == 0] = 1
    return mean, lam, U * sign


def _min_step(Z: torch.Tensor, bits: np.ndarray):
    lo = Z.min(dim=0).values
    hi = Z.max(dim=0).values
    levels = torch.tensor((2.0 ** bits) - 1.0, dtype=torch.float64, device=Z.device)
    step = torch.clamp((hi - lo) / torch.clamp(levels, min=1.0), min=1e-8)
    keep = torch.tensor(bits > 0, device=Z.device)
    return torch.where(keep, lo, 0.0), torch.where(keep, step, 0.0)


def fit_uniform(x_fit: torch.Tensor, r: int, choices, budget: int) -> dict:
    """One basis per (b, h) from prefill rows x_fit [B, H, S_fit, D] (device),
    fitted on the GPU by libkvc's kvc_fit_uniform (covariance, Jacobi
    eigendecomposition, DP allocation, frozen minimum and step, in float64);
    returns the uniform layer's parameters as host arrays."""
    from . import fit_uniform as device_fit

    B, H, S, D = x_fit.shape
    out = device_fit(x_fit, S, r, choices, budget)
    torch.cuda.synchronize(x_fit.device)
    return dict(V=out["V"].cpu().numpy(), mean=out["mean"].cpu().numpy(),
                bits=out["bits"].cpu().numpy(), qmin=out["qmin"].cpu().numpy(),
                qstep=out["qstep"].cpu().numpy(), basis_of=np.arange(B * H, dtype=np.int32))


def fit_uniform_shared(x_fit: torch.Tensor, r: int, bits_each: int) -> dict:
    """One basis per KV head shared by the batch, every kept component at
    ``bits_each`` bits (the uniform 2- and 4-bit allocations of a sweep)."""
    B, H, S, D = x_fit.shape
    rows = x_fit.permute(1, 0, 2, 3).reshape(H, B * S, D)
    mean, lam, U = pca(rows)
    V32 = U[:, :, :r].to(torch.float32)
    m32 = mean.to(torch.float32)
    bits = np.full(r, bits_each, dtype=np.int64)
    los, sts = [], []
    for h in range(H):
        Z = (rows[h].to(torch.float64) - m32[h].double()) @ V32[h].double()
        lo, st = _min_step(Z, bits)
        los.append(lo), sts.append(st)
    return dict(V=V32.cpu().numpy(), mean=m32.cpu().numpy(),
                bits=np.tile(bits, (H, 1)).astype(np.uint8),
                qmin=torch.stack(los).to(torch.float32).cpu().numpy(),
                qstep=torch.stack(sts).to(torch.float32).cpu().numpy(),
                basis_of=np.array([h for b in range(B) for h in range(H)], dtype=np.int32))


def fit_group(x_fit: torch.Tensor, heads_per_group: int, r: int, hi_bit=4, lo_bit=2,
              hi_fraction=0.25, group_size=32) -> dict:
    """One projection per head group (rows pooled over batch and tokens)."""
    B, H, S, D = x_fit.shape
    Hg = H // heads_per_group
    rows = (x_fit.reshape(B, Hg, heads_per_group, S, D).permute(1, 0, 3, 2, 4)
            .reshape(Hg, B * S, heads_per_group * D))
    mean, lam, U = pca(rows)
    n_hi = int(math.ceil(hi_fraction * r))
    bits = np.array([hi_bit] * n_hi + [lo_bit] * (r - n_hi), dtype=np.uint8)
    return dict(V=U[:, :, :r].to(torch.float32).cpu().numpy(),
                mean=mean.to(torch.float32).cpu().numpy(), bits=np.tile(bits, (Hg, 1)),
                basis_of=np.array([g for b in range(B) for g in range(Hg)], dtype=np.int32),
                heads_per_group=heads_per_group, group_size=group_size)


def rotation(d: int, seed: int) -> np.ndarray:
    """Seeded orthogonal d x d rotation (QR of a seeded Gaussian, diag(R) > 0)."""
    g = torch.Generator().manual_seed(seed)
    G = torch.randn(d, d, generator=g, dtype=torch.float64)
    Q, R = torch.linalg.qr(G)
    return (Q * torch.sign(torch.diagonal(R))).to(torch.float32).numpy()


def gaussian_codebook(bits: int, sigma: float, iters: int = 2000) -> np.ndarray:
    """Lloyd-Max centroids for N(0, sigma^2), ascending, fp32."""
    n = 1 << bits
    c = torch.linspace(-2.0, 2.0, n, dtype=torch.float64)
    sq2 = math.sqrt(2.0)
    for _ in range(iters):
        t = torch.cat([torch.tensor([-math.inf], dtype=torch.float64), 0.5 * (c[1:] + c[:-1]),
                       torch.tensor([math.inf], dtype=torch.float64)])
        pdf = torch.exp(-0.5 * t * t) / math.sqrt(2 * math.pi)
        pdf = torch.nan_to_num(pdf, nan=0.0)
        cdf = 0.5 * (1 + torch.erf(t / sq2))
        new = (pdf[:-1] - pdf[1:]) / (cdf[1:] - cdf[:-1])
        if torch.max(torch.abs(new - c)) < 1e-14:
            c = new
            break
        c = new
    return (sigma * c).to(torch.float32).numpy()
