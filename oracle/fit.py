"""One-time fit of the frozen layer parameters (float64, CPU).

Test infrastructure only -- see ``oracle/__init__.py``.

Everything here runs once, at prefill, before the hot path: the pages fit
the basis and the bit allocation on the first call and freeze them
(kvtc_cache page, module docstring, "NOT PATH-DEPENDENT" and "Design").
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "pca_fit",
    "dp_allocate",
    "brute_force_allocate",
    "allocation_distortion",
    "uniform_params",
    "palu_bits",
    "lloyd_max_gaussian",
    "seeded_rotation",
]


def pca_fit(X):
    """Local PCA of prefill rows ``X`` [S, D_in] -> (mean, lam, U).

    kvtc_cache page, module docstring "Design", prefill step 1 (local PCA of
    the prefill batch, stored as ``V`` and ``mean``), and
    ``KVTCKVCache.update_and_fetch`` (the batched local-PCA fit that returns
    ``(L, V, mean, variances)``).  palu_cache page, "Design", prefill step 2
    (one shared projection per head group, fitted on the group's rows).

    The principal directions are the eigenvectors of the covariance
    C = (X - mean)^T (X - mean) / S, sorted by eigenvalue, largest first.
    Each eigenvector's sign is fixed so that its largest-magnitude entry is
    positive (the pages leave the sign open; any fixed rule gives the same
    reconstruction).
    """
    X = np.asarray(X, dtype=np.float64)
    S = X.shape[0]
    if X.ndim != 2 or S < 2:
        raise ValueError("the fit needs at least two prefill rows")
    mean = X.mean(axis=0)
    Xc = X - mean
    C = (Xc.T @ Xc) / S
    lam, U = np.linalg.eigh(C)
    order = np.argsort(-lam, kind="stable")
    lam = lam[order]
    U = U[:, order]
    pivot = np.argmax(np.abs(U), axis=0)
    sign = np.sign(U[pivot, np.arange(U.shape[1])])
    sign[sign == 0] = 1.0
    return mean, lam, U * sign


def allocation_distortion(lam, bits) -> float:
    """The distortion proxy sum_k lam_k 2^(-2 b_k); a 0-bit component costs lam_k.

    kvtc_cache page, module docstring (the "analytic distortion proxy" the
    dynamic programme minimises).
    """
    lam = np.asarray(lam, dtype=np.float64)
    b = np.asarray(bits, dtype=np.float64)
    return float(np.sum(lam * np.power(2.0, -2.0 * b)))


def dp_allocate(lam, choices, budget: int) -> np.ndarray:
    """Discrete per-component bit allocation by dynamic programming.

    kvtc_cache page, module docstring: a "DP-optimal, discrete,
    per-component bit allocation (may drop a component entirely, i.e. assign
    it 0 bits)" under ``kvtc_bit_budget`` total bits per token, with bit
    widths from ``kvtc_bit_choices``.

    Minimises sum_k lam_k 2^(-2 b_k) over b_k in ``choices`` subject to
    sum_k b_k <= budget.  cost[k][c] is the least distortion of components
    k..r-1 given c bits still free; the allocation is read forward from
    component 0 with all ``budget`` bits free.  Among equal costs the
    smallest width wins (choices are scanned in ascending order with a
    strict comparison).
    """
    if budget < 0:
        raise ValueError("bit budget must be >= 0")
    lam = np.asarray(lam, dtype=np.float64)
    r = lam.shape[0]
    choices = sorted(set(int(c) for c in choices))
    if any(c < 0 for c in choices):
        raise ValueError("bit widths must be >= 0")
    cost = np.full((r + 1, budget + 1), np.inf)
    cost[r, :] = 0.0
    for k in range(r - 1, -1, -1):
        for b in choices:
            if b > budget:
                continue
            cand = np.full(budget + 1, np.inf)
            cand[b:] = lam[k] * 2.0 ** (-2 * b) + cost[k + 1, : budget + 1 - b]
            cost[k] = np.minimum(cost[k], cand)
    if not np.isfinite(cost[0, budget]):
        raise ValueError("no allocation fits the budget with these choices")
    bits = np.zeros(r, dtype=np.int64)
    free = budget
    for k in range(r):
        best_b, best_v = None, np.inf
        for b in choices:
            if b > free:
                continue
            v = lam[k] * 2.0 ** (-2 * b) + cost[k + 1, free - b]
            if v < best_v:
                best_b, best_v = b, v
        bits[k] = best_b
        free -= best_b
    return bits


def brute_force_allocate(lam, choices, budget: int):
    """Every feasible allocation, enumerated: returns (min distortion, list of minimisers).

    Only for small r (the dynamic programme's check).
    """
    import itertools

    lam = np.asarray(lam, dtype=np.float64)
    choices = sorted(set(int(c) for c in choices))
    best, arg = np.inf, []
    for combo in itertools.product(choices, repeat=lam.shape[0]):
        if sum(combo) > budget:
            continue
        d = allocation_distortion(lam, combo)
        if d < best:
            best, arg = d, [combo]
        elif d == best:
            arg.append(combo)
    return best, arg


def uniform_params(Z_fit, bits):
    """Frozen per-component minimum and step from the fit rows' latents.

    kvtc_cache page, ``_TensorKVTC._requantize`` (``quantize_component`` gives
    each surviving component a minimum ``lo`` and a step ``scale``).  Here they
    are taken once, from the prefill latents, and frozen:
    lo_k = min_t z_{t,k}; step_k = max((max_t z_{t,k} - lo_k) / (2^b_k - 1), 1e-8).
    Dropped (0-bit) components get lo = step = 0 (never used).
    """
    Z = np.asarray(Z_fit, dtype=np.float64)
    bits = np.asarray(bits)
    lo = np.zeros(bits.shape[0])
    step = np.zeros(bits.shape[0])
    for k, b in enumerate(bits):
        if b == 0:
            continue
        lo[k] = Z[:, k].min()
        step[k] = max((Z[:, k].max() - lo[k]) / (2.0 ** int(b) - 1.0), 1e-8)
    return lo, step


def palu_bits(r: int, hi_bit: int, lo_bit: int, hi_fraction: float) -> np.ndarray:
    """Mixed-bit split: the top ceil(hi_fraction * r) components (largest
    variance first) at ``hi_bit``, the rest at ``lo_bit``.

    palu_cache page, ``PALUKVCache`` parameters ``palu_hi_bit``,
    ``palu_lo_bit``, ``palu_hi_fraction`` ("Design", prefill step 3:
    mixed-bit quantisation of the [S, r] latents).
    """
    n_hi = int(math.ceil(hi_fraction * r))
    return np.array([hi_bit] * n_hi + [lo_bit] * (r - n_hi), dtype=np.int64)


def _phi(x: float) -> float:
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def _Phi(x: float) -> float:
    return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def lloyd_max_gaussian(levels: int, sigma: float = 1.0, tol: float = 1e-13,
                       max_iter: int = 100000) -> np.ndarray:
    """Lloyd-Max scalar codebook (ascending centroids) for N(0, sigma^2).

    turboquant_cache page, class docstring and ``TurboQuantMSE(d, b, seed,
    store)``: keys are quantised coordinate-wise against a scalar codebook of
    2^b centroids; after a random rotation each coordinate of a unit vector
    is close to N(0, 1/d).

    Lloyd's iteration: thresholds are the midpoints of adjacent centroids,
    each centroid is the conditional mean of the Gaussian on its cell,
    E[X | a < X < b] = sigma (phi(a/s) - phi(b/s)) / (Phi(b/s) - Phi(a/s)),
    repeated until the largest move is below ``tol`` (relative to sigma).
    """
    c = np.linspace(-2.0, 2.0, levels)
    for _ in range(max_iter):
        t = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))
        new = np.empty_like(c)
        for j in range(levels):
            a, b = t[j], t[j + 1]
            pa = 0.0 if np.isinf(a) else _phi(a)
            pb = 0.0 if np.isinf(b) else _phi(b)
            Pa = 0.0 if a == -np.inf else _Phi(a)
            Pb = 1.0 if b == np.inf else _Phi(b)
            new[j] = (pa - pb) / (Pb - Pa)
        done = np.max(np.abs(new - c)) < tol
        c = new
        if done:
            break
    return sigma * c


def seeded_rotation(d: int, seed: int) -> np.ndarray:
    """Seeded d x d orthogonal rotation.

    turboquant_cache page, ``TurboQuantMSE(d=d, b=b, seed=seed, ...)`` (a
    seeded, deterministic rotation; the page does not show the seed-to-matrix
    map).  Here: Q of the QR factorisation of a standard Gaussian matrix drawn
    from ``numpy.random.default_rng(seed)``, with column signs chosen so that
    diag(R) > 0, which makes the map unique.
    """
    G = np.random.default_rng(seed).standard_normal((d, d))
    Q, R = np.linalg.qr(G)
    return Q * np.sign(np.diag(R))
