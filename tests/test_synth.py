"""CPU checks that the seeded input generators follow their stated recipe.

Spectral rows x = mu + sum_k k^-alpha g_k u_k + 0.01 eps (mu ~ N(0, 0.25),
U orthogonal), outlier channels scaled by 8 after generation, and Gaussian
keys with 1 % of the coordinates replaced by Student-t(3) draws.  Every
statistic is taken on fixed seeds, so the outcomes are deterministic.
"""
import math

import numpy as np
import torch

import synth


def test_generators_are_pure_functions_of_the_key():
    a = torch.randn(4, generator=synth.make_generator(5, 1, 2))
    b = torch.randn(4, generator=synth.make_generator(5, 1, 2))
    c = torch.randn(4, generator=synth.make_generator(5, 1, 3))
    assert torch.equal(a, b) and not torch.equal(a, c)
    x1 = synth.kv_spectral(1, 2, 16, 8, 1.0, seed=3, tensor=0)
    x2 = synth.kv_spectral(1, 2, 16, 8, 1.0, seed=3, tensor=0)
    v = synth.kv_spectral(1, 2, 16, 8, 1.0, seed=3, tensor=1)
    assert torch.equal(x1, x2) and not torch.equal(x1, v)     # K and V are independent draws


def test_spectral_basis_is_orthogonal():
    mu, U = synth.spectral_basis(64, synth.make_generator(1))
    assert torch.allclose(U.T @ U, torch.eye(64, dtype=U.dtype), atol=1e-12)
    assert 0.35 < mu.std().item() < 0.65                        # N(0, 0.5^2), 64 draws


def test_spectral_rows_have_the_stated_spectrum():
    d, n, alpha = 8, 40000, 1.0
    gen = synth.make_generator(9)
    mu, U = synth.spectral_basis(d, gen)
    X = synth.spectral_rows(mu, U, n, alpha, gen)
    Z = (X - mu) @ U                                            # coordinates along u_k
    var = Z.var(dim=0).numpy()
    want = np.arange(1, d + 1, dtype=np.float64) ** (-2 * alpha) + 0.01 ** 2
    assert np.allclose(var, want, rtol=0.03)
    assert np.allclose(Z.mean(dim=0).numpy(), 0.0, atol=4 * math.sqrt(want[0] / n))


def test_outlier_channels_are_the_plain_rows_times_eight():
    plain = synth.kv_spectral(2, 2, 32, 128, 1.0, seed=4, tensor=0, dtype="f32")
    out = synth.kv_spectral(2, 2, 32, 128, 1.0, seed=4, tensor=0, n_outliers=3, dtype="f32")
    for b in range(2):
        for h in range(2):
            ch = synth.outlier_channels(128, 3, synth.make_generator(4, 0, b, h, 7919))
            assert len(set(ch.tolist())) == 3
            rest = torch.ones(128, dtype=torch.bool)
            rest[ch] = False
            assert torch.equal(out[b, h][:, ch], 8.0 * plain[b, h][:, ch])
            assert torch.equal(out[b, h][:, rest], plain[b, h][:, rest])


def _max_cross_corr(p, q):
    """Largest |correlation| between a channel of p [S, D] and one of q."""
    p0, q0 = p - p.mean(0), q - q.mean(0)
    c = p0.T @ q0 / p.shape[0]
    return (c / (p0.std(0)[:, None] * q0.std(0)[None, :])).abs().max().item()


def test_group_rows_share_one_model_per_group():
    B, H, S, D, hpg = 3, 4, 4000, 4, 2
    x = synth.group_spectral(B, H, S, D, hpg, 1.0, seed=6, tensor=0, dtype="f32").double()
    assert x.shape == (B, H, S, D)
    # the heads of one group are slices of one D_in = 8 model (correlated
    # channels); heads of different groups are independent draws
    for b in range(B):
        assert _max_cross_corr(x[b, 0], x[b, 1]) > 0.5
        assert _max_cross_corr(x[b, 2], x[b, 3]) > 0.5
        assert _max_cross_corr(x[b, 0], x[b, 2]) < 5 / math.sqrt(S)
    # each batch entry is a fresh draw of its group's model: the same channel
    # means, different rows
    m = x[:, 0:2].mean(dim=2)                                   # [B, hpg, D]
    assert torch.allclose(m[0], m[1], atol=0.1) and torch.allclose(m[0], m[2], atol=0.1)
    assert not torch.equal(x[0, 0], x[1, 0])


def test_heavy_tailed_keys_mix():
    k = synth.heavy_tailed_keys(2, 4, 4096, 64, seed=8, dtype="f32").reshape(-1).double()
    n = k.numel()                                               # 2.1 M coordinates
    med = k.abs().median().item()
    assert abs(med - 0.6745) < 0.01                             # the Gaussian bulk
    # P(|t_3| > 6) = 0.00927 against 2e-9 for N(0, 1): the tail is the 1 % t draws
    tail = (k.abs() > 6).sum().item()
    want = n * 0.01 * 0.00927
    assert 0.6 * want < tail < 1.4 * want
