"""GPU parity of the on-device prefill fit (kvc_fit_uniform) against the
float64 oracle fit (oracle/fit.py: pca_fit, dp_allocate, uniform_params).

What is unique is compared, at the precision the arithmetic allows:
* eigenvalues: within 1e-12 lam_max (both solvers are backward stable in
  float64: |error| <= c n eps ||C||);
* the fp32 mean: within one fp32 ulp (the two sums run in different orders);
* each kept eigenvector whose eigenvalue is separated from its neighbours:
  within 1e-6 + 1e3 D eps lam_max / gap (fp32 rounding plus the float64
  perturbation bound of an eigenvector, eps ||C|| / gap);
* the DP allocation on the device's own eigenvalues: the oracle's, bit for
  bit (same arithmetic on the same numbers); on the oracle's eigenvalues:
  the same widths wherever no near-tie decides;
* the minimum and step on the device's own V and mean: within one fp32 ulp
  plus 1e-12 max_t ||x_t - mean|| (float64 sums in different orders).
Then a layer built from the device fit stores the oracle's codes.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import codec, fit
from oracle.layer import OracleLayer

from kvc_cases import MISMATCH_RATE, compare_codes, oracle_kwargs

pytestmark = pytest.mark.gpu

EPS = 2.0 ** -52


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rank_quantized_kv_gb300 as kvc

    kvc.load_library()
    return kvc


def _dev():
    return torch.device("cuda:0")


def _f32_close(a, b, extra=0.0):
    a = np.asarray(a, dtype=np.float64)
    b32 = np.asarray(b, dtype=np.float32)
    tol = np.spacing(np.abs(b32)).astype(np.float64) + extra
    return np.abs(a - b32.astype(np.float64)) <= tol


def _check_fit(out, x64, S_fit, r, choices, budget, decisive=True):
    """Compare every slot of a device fit with the oracle's fit of the same rows."""
    B, H, _, D = x64.shape
    g = {k: v.cpu().numpy() for k, v in out.items() if k != "workspace"}
    for s in range(B * H):
        b, h = divmod(s, H)
        X = x64[b, h, :S_fit]
        mean, lam, U = fit.pca_fit(X)
        scale = max(lam[0], 1e-300)
        lam_g = g["lam"][s]
        assert np.max(np.abs(lam_g - lam)) <= 1e-12 * scale, f"slot {s}: eigenvalues"
        assert _f32_close(g["mean"][s], mean.astype(np.float32)).all(), f"slot {s}: mean"
        V_g = g["V"][s].astype(np.float64)
        for k in range(r):
            left = lam[k - 1] - lam[k] if k > 0 else np.inf
            right = lam[k] - lam[k + 1] if k + 1 < D else np.inf
            gap = min(left, right)
            if gap <= 1e-8 * scale:
                continue  # the vector is not unique to this precision
            tol = 1e-6 + 1e3 * D * EPS * scale / gap
            err = np.max(np.abs(V_g[:, k] - U[:, k]))
            assert err <= tol, f"slot {s} vector {k}: {err:.3e} > {tol:.3e}"
        bits_g = g["bits"][s].astype(np.int64)
        assert np.array_equal(bits_g, fit.dp_allocate(lam_g[:r], choices, budget)), \
            f"slot {s}: allocation on the device's eigenvalues"
        if decisive:
            assert np.array_equal(bits_g, fit.dp_allocate(lam[:r], choices, budget)), \
                f"slot {s}: allocation on the oracle's eigenvalues"
        m_g = g["mean"][s].astype(np.float64)
        lo, st = fit.uniform_params(codec.project(X, m_g, V_g), bits_g)
        extra = 1e-12 * np.max(np.linalg.norm(X - m_g, axis=1))
        assert _f32_close(g["qmin"][s], lo.astype(np.float32), extra).all(), f"slot {s}: qmin"
        assert _f32_close(g["qstep"][s], st.astype(np.float32), extra).all(), f"slot {s}: qstep"
        assert np.all(g["qstep"][s][bits_g > 0] > 0)
        assert np.all(g["qmin"][s][bits_g == 0] == 0) and np.all(g["qstep"][s][bits_g == 0] == 0)


CASES = {
    # name: B, H, D, T, S_fit, r, choices, budget, dtype, alpha, outliers
    "kvtc-tiny": (1, 2, 64, 80, 64, 16, (0, 1, 2, 4, 8), 48, "f32", 0.8, 0),
    "llama-like": (2, 4, 128, 600, 512, 32, (0, 2, 4, 8), 128, "bf16", 1.0, 3),
    "full-rank-ragged-D": (1, 3, 104, 300, 300, 104, (0, 1, 2, 3, 4, 8), 300, "f16", 0.5, 0),
    "D8": (2, 1, 8, 40, 33, 5, (1, 2, 3), 11, "f32", 1.0, 0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fit_matches_oracle(kvc, name):
    B, H, D, T, S_fit, r, choices, budget, dt, alpha, outl = CASES[name]
    x = synth.kv_spectral(B, H, T, D, alpha=alpha, seed=6100, tensor=0, n_outliers=outl, dtype=dt)
    x64 = x.double().numpy()
    out = kvc.fit_uniform(x.to(_dev()), S_fit, r, choices, budget)
    torch.cuda.synchronize()
    _check_fit(out, x64, S_fit, r, choices, budget)


def test_fit_strided_input_and_unsorted_choices(kvc):
    """Rows read through strides ([B, S, H, D] memory seen as [B, H, S, D]);
    choices given unsorted and repeated; a budget beyond max(choices) * r."""
    B, H, T, D, S_fit, r = 2, 3, 200, 64, 150, 24
    x = synth.kv_spectral(B, H, T, D, alpha=0.9, seed=6200, tensor=1, dtype="bf16")
    xs = x.permute(0, 2, 1, 3).contiguous().to(_dev()).permute(0, 2, 1, 3)
    assert not xs.is_contiguous()
    choices = (8, 0, 4, 2, 4)
    out = kvc.fit_uniform(xs, S_fit, r, choices, 10_000)
    torch.cuda.synchronize()
    _check_fit(out, x.double().numpy(), S_fit, r, choices, 10_000)
    assert np.all(out["bits"].cpu().numpy() == 8)


def test_fit_two_rows_and_rank_deficient(kvc):
    """S_fit = 2 (the least the fit takes: a rank-1 covariance) and rows in a
    3-dimensional subspace: only the non-zero eigenpairs are unique."""
    D, r = 32, 8
    x2 = synth.kv_spectral(1, 2, 2, D, alpha=1.0, seed=6300, tensor=0, dtype="f32")
    out = kvc.fit_uniform(x2.to(_dev()), 2, r, (0, 1, 2, 4), 12)
    torch.cuda.synchronize()
    _check_fit(out, x2.double().numpy(), 2, r, (0, 1, 2, 4), 12, decisive=False)
    g = torch.Generator().manual_seed(6301)
    basis = torch.linalg.qr(torch.randn(D, 3, generator=g, dtype=torch.float64))[0]
    coef = torch.randn(1, 2, 100, 3, generator=g, dtype=torch.float64) * torch.tensor([3.0, 1.0, 0.3],
                                                                                        dtype=torch.float64)
    x3 = (coef @ basis.T + 0.5).to(torch.float32)
    out = kvc.fit_uniform(x3.to(_dev()), 100, r, (0, 2, 4, 8), 24)
    torch.cuda.synchronize()
    _check_fit(out, x3.double().numpy(), 100, r, (0, 2, 4, 8), 24, decisive=False)
    lam = out["lam"].cpu().numpy()
    assert np.all(np.abs(lam[:, 3:]) <= 1e-12 * lam[:, :1])


def test_fit_then_append_stores_the_oracle_codes(kvc):
    """A uniform layer built from the device fit stores, for the prefill and
    the tokens after it, the codes the oracle computes from those parameters."""
    B, H, D, T, S_fit = 2, 4, 128, 700, 512
    x = synth.kv_spectral(B, H, T, D, alpha=1.0, seed=2000, tensor=0, n_outliers=3, dtype="bf16")
    x64 = x.double().numpy()
    xd = x.to(_dev())
    from rank_quantized_kv_gb300 import calib

    params = calib.fit_uniform(xd[:, :, :S_fit], 32, (0, 2, 4, 8), 128)
    gl = kvc.KVCacheLayer("uniform", B, H, D, in_dtype="bf16", capacity=T, device=_dev(), **params)
    rl = OracleLayer("uniform", B, H, D, capacity=T, **oracle_kwargs(params))
    gl.append(xd)
    assert gl.sync_status() == 0
    rl.append(x64)
    n = mism = 0
    for s in range(rl.n_slots):
        rows, side = gl.slot_rows(s)
        c, m = compare_codes(rows.cpu().numpy(), None, rl, s, rl.slot_rows(x64, s))
        n, mism = n + c, mism + m
    assert mism <= MISMATCH_RATE * n


@pytest.mark.parametrize("bad", [
    dict(S_fit=1), dict(r=0), dict(r=65), dict(choices=(5,)), dict(choices=(2, 4), budget=10),
    dict(choices=()), dict(budget=-1),
])
def test_fit_rejects_bad_arguments(kvc, bad):
    x = torch.zeros(1, 2, 16, 64, device=_dev())
    a = dict(S_fit=16, r=8, choices=(0, 2, 4), budget=16)
    a.update(bad)
    with pytest.raises(kvc.KvcError):
        kvc.fit_uniform(x, a["S_fit"], a["r"], a["choices"], a["budget"])


def test_fit_rejects_wide_heads_and_host_rows(kvc):
    with pytest.raises(kvc.KvcError):
        kvc.fit_uniform(torch.zeros(1, 1, 8, 136, device=_dev()), 8, 8, (0, 2), 8)
    with pytest.raises(kvc.KvcError):
        kvc.fit_uniform(torch.zeros(1, 1, 8, 64), 8, 8, (0, 2), 8)
