"""CPU checks of the calibration helpers (rank_quantized_kv_gb300.calib).

The calibration runs once per layer, outside the hot path: the Lloyd-Max
codebook and the seeded rotation of the codebook mode (turboquant_cache page,
``TurboQuantMSE``), the shared-basis uniform fit and the head-group fit
(kvtc_cache page, "Design", prefill step 1; palu_cache page, "Design",
prefill steps 2-3).  These tests pin the helpers to printed values and closed
forms, and compare them with the oracle's float64 restatements of the same
steps.
"""
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

from oracle import fit
from rank_quantized_kv_gb300 import calib

GOLDEN = Path(__file__).parent / "golden"


def _rows(n, s, d, seed):
    """Rows with a decaying spectrum (well-separated eigenvalues) and a mean."""
    g = np.random.default_rng(seed)
    U, _ = np.linalg.qr(g.standard_normal((d, d)))
    sig = 3.0 * np.arange(1, d + 1, dtype=np.float64) ** -1.0
    X = g.standard_normal((n, s, d)) * sig @ U.T + g.normal(0.0, 0.5, size=(n, 1, d))
    return X


def test_codebook_matches_max_table():
    table = json.loads((GOLDEN / "lloyd_max_gaussian.json").read_text())["levels"]
    for levels, row in table.items():
        n = int(levels)
        c = calib.gaussian_codebook(int(math.log2(n)), 1.0).astype(np.float64)
        assert c.shape == (n,)
        assert np.all(np.diff(c) > 0)                            # ascending
        assert np.allclose(c, -c[::-1], atol=1e-6)               # symmetric
        assert np.allclose(c[n // 2:], row["outputs"], atol=6e-4)


def test_codebook_closed_forms_and_scaling():
    # one bit: the centroids are +-E|X| = +-sqrt(2/pi) sigma
    c = calib.gaussian_codebook(1, 0.3)
    assert c[1] == pytest.approx(0.3 * math.sqrt(2 / math.pi), rel=1e-6)
    # centroids scale with sigma (the TurboQuant codebook is for N(0, 1/d))
    c1 = calib.gaussian_codebook(3, 1.0)
    cs = calib.gaussian_codebook(3, 128 ** -0.5)
    assert np.allclose(cs, c1 * 128 ** -0.5, rtol=1e-6)
    assert calib.gaussian_codebook(3, 1.0).dtype == np.float32


def test_codebook_matches_the_oracle():
    for bits in (1, 2, 3, 4):
        c = calib.gaussian_codebook(bits, 128 ** -0.5).astype(np.float64)
        o = fit.lloyd_max_gaussian(1 << bits, sigma=128 ** -0.5)
        # the helper returns fp32: within one fp32 rounding of the float64 fixed point
        assert np.allclose(c, o, rtol=2 ** -23, atol=1e-12)


def test_rotation_is_orthogonal_and_seeded():
    R = calib.rotation(128, 1234).astype(np.float64)
    assert R.shape == (128, 128)
    assert np.abs(R.T @ R - np.eye(128)).max() < 1e-5
    assert abs(abs(np.linalg.det(R)) - 1.0) < 1e-4
    assert np.array_equal(calib.rotation(128, 1234), calib.rotation(128, 1234))
    assert not np.allclose(calib.rotation(128, 1234), calib.rotation(128, 1235))


def test_pca_matches_the_oracle():
    X = _rows(3, 400, 16, seed=5)
    mean, lam, U = calib.pca(torch.from_numpy(X))
    for i in range(X.shape[0]):
        m_o, l_o, U_o = fit.pca_fit(X[i])
        assert np.allclose(mean[i].numpy(), m_o, atol=1e-12)
        assert np.allclose(lam[i].numpy(), l_o, rtol=1e-9, atol=1e-12)
        # the same sign rule (largest-magnitude entry positive) on both sides
        assert np.allclose(U[i].numpy(), U_o, atol=1e-8)


def test_pca_recovers_a_planted_covariance():
    # rows +-a e_k for each k: mean 0, covariance diag(a_k^2) / D exactly
    d = 6
    a = np.array([6.0, 5.0, 4.0, 3.0, 2.0, 1.0])
    rows = np.concatenate([np.diag(a), -np.diag(a)])[None]
    mean, lam, U = calib.pca(torch.from_numpy(rows))
    assert np.allclose(mean.numpy(), 0.0)
    assert np.allclose(lam[0].numpy(), a ** 2 / d, rtol=1e-12)
    assert np.allclose(np.abs(U[0].numpy()), np.eye(d), atol=1e-12)
    assert np.all(U[0].numpy().max(axis=0) > 0)


def test_min_step_matches_the_oracle():
    g = np.random.default_rng(3)
    Z = g.standard_normal((200, 12)) * np.linspace(0.1, 4.0, 12)
    Z[:, 5] = 2.5                                                # a constant column
    bits = np.array([8, 4, 4, 2, 2, 2, 1, 0, 0, 3, 2, 1])
    lo, st = calib._min_step(torch.from_numpy(Z), bits)
    lo_o, st_o = fit.uniform_params(Z, bits)
    assert np.array_equal(lo.numpy(), lo_o)
    assert np.array_equal(st.numpy(), st_o)
    assert st.numpy()[5] == 1e-8                                 # the step's floor


def test_fit_uniform_shared_on_cpu():
    B, H, S, D, r = 2, 3, 128, 16, 6
    x = torch.from_numpy(_rows(B * H, S, D, seed=11).reshape(B, H, S, D))
    p = calib.fit_uniform_shared(x, r, 4)
    assert p["V"].shape == (H, D, r) and p["V"].dtype == np.float32
    assert np.array_equal(p["bits"], np.full((H, r), 4, dtype=np.uint8))
    assert list(p["basis_of"]) == [h for _ in range(B) for h in range(H)]
    for h in range(H):
        rows = x[:, h].reshape(B * S, D).numpy()
        m_o, _, U_o = fit.pca_fit(rows)
        assert np.allclose(p["mean"][h], m_o, atol=1e-6)
        assert np.allclose(p["V"][h], U_o[:, :r], atol=1e-6)
        # the frozen min/step come from the latents of the fp32 basis and mean
        Z = (rows - p["mean"][h].astype(np.float64)) @ p["V"][h].astype(np.float64)
        lo_o, st_o = fit.uniform_params(Z, np.full(r, 4))
        assert np.allclose(p["qmin"][h], lo_o, rtol=1e-6, atol=1e-7)
        assert np.allclose(p["qstep"][h], st_o, rtol=1e-6)


def test_fit_group_on_cpu():
    B, H, S, D, r, hpg = 2, 4, 64, 8, 6, 2
    x = torch.from_numpy(_rows(B * H, S, D, seed=21).reshape(B, H, S, D))
    p = calib.fit_group(x, hpg, r, hi_bit=4, lo_bit=2, hi_fraction=0.25, group_size=2)
    Hg = H // hpg
    assert p["V"].shape == (Hg, hpg * D, r)
    assert np.array_equal(p["bits"], np.tile(fit.palu_bits(r, 4, 2, 0.25), (Hg, 1)))
    assert list(p["basis_of"]) == [g for _ in range(B) for g in range(Hg)]
    assert p["heads_per_group"] == hpg and p["group_size"] == 2
    for gi in range(Hg):
        # a group's rows: its heads' channels side by side, pooled over batch and tokens
        rows = np.concatenate([x[:, gi * hpg + j].reshape(B * S, D).numpy()
                               for j in range(hpg)], axis=1)
        m_o, _, U_o = fit.pca_fit(rows)
        assert np.allclose(p["mean"][gi], m_o, atol=1e-6)
        assert np.allclose(p["V"][gi], U_o[:, :r], atol=1e-6)
