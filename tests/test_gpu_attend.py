"""GPU parity of decode attention on the stored codes (kvc_attend) against the
float64 oracle (oracle/attend.py) applied to the oracle's decode of the GPU's
own stored codes: per (batch, query head), max-abs error <= 4e-3 max|out| and
RMS error <= 1e-3 RMS(out), the fetch's reconstruction tolerance."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle.attend import attend_rows
from oracle.layer import OracleLayer

from kvc_cases import fit_codebook, fit_uniform, oracle_kwargs

pytestmark = pytest.mark.gpu

MAX_ABS_REL = 4e-3
RMS_REL = 1e-3


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rank_quantized_kv_gb300 as kvc

    kvc.load_library()
    return kvc


def _dev():
    return torch.device("cuda:0")


def _decoded(gl, rl, slot):
    """The oracle's float64 decode of the GPU's rows of one slot [S, D]."""
    rows, side = gl.slot_rows(slot)
    sd = None
    if side is not None:
        sd = side.cpu().numpy().view(np.float16)
        if rl.mode in ("codebook", "int8"):
            sd = sd[:, 0]
    return rl.decode(slot, rows.cpu().numpy(), sd)


def _check(out, gk, rk, gv, rv, q, scale, pairs=None):
    out = out.float().cpu().numpy().astype(np.float64)
    q = q.double().cpu().numpy()
    B, Hq, D = q.shape
    H = rk.H
    rep = Hq // H
    cache = {}
    for b in range(B):
        for hq in range(Hq):
            if pairs is not None and (b, hq) not in pairs:
                continue
            s = b * H + hq // rep
            if s not in cache:
                cache[s] = (_decoded(gk, rk, s), _decoded(gv, rv, s))
            K, V = cache[s]
            ref = attend_rows(q[b, hq], K, V, scale)
            err = out[b, hq] - ref
            mx = max(np.abs(ref).max(), 1e-30)
            rms = max(math.sqrt(np.mean(ref ** 2)), 1e-30)
            assert np.abs(err).max() <= MAX_ABS_REL * mx, (b, hq, np.abs(err).max() / mx)
            assert math.sqrt(np.mean(err ** 2)) <= RMS_REL * rms, (b, hq)


def _layers(kvc, kmode, vmode, B, H, D, S, seed):
    dev = _dev()
    if kmode == "codebook":
        xk = synth.heavy_tailed_keys(B, H, S, D, seed=seed, dtype="f16")
        pk = fit_codebook(D)
        kdt = "f16"
    else:
        xk = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=seed, tensor=0, n_outliers=3,
                               dtype="bf16")
        pk = fit_uniform(xk.double().numpy(), min(S, 512), 32, [0, 2, 4, 8], 128)
        kdt = "bf16"
    xv = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=seed + 1, tensor=1,
                           dtype="f16" if vmode == "int8" else "bf16")
    if vmode == "int8":
        pv, vdt = {}, "f16"
    else:
        pv, vdt = fit_uniform(xv.double().numpy(), min(S, 512), 48, [0, 2, 4, 8], 160), "bf16"
    gk = kvc.KVCacheLayer(kmode, B, H, D, in_dtype=kdt, capacity=S, device=dev, **pk)
    gv = kvc.KVCacheLayer(vmode, B, H, D, in_dtype=vdt, capacity=S, device=dev, **pv)
    rk = OracleLayer(kmode, B, H, D, capacity=S, **oracle_kwargs(pk))
    rv = OracleLayer(vmode, B, H, D, capacity=S, **oracle_kwargs(pv))
    gk.append(xk.to(dev))
    gv.append(xv.to(dev))
    assert gk.sync_status() == 0 and gv.sync_status() == 0
    return gk, gv, rk, rv


@pytest.mark.parametrize("kmode,vmode,B,H,D,S,rep", [
    ("codebook", "int8", 2, 4, 128, 1000, 4),
    ("uniform", "uniform", 2, 2, 128, 700, 2),
    ("uniform", "int8", 1, 4, 64, 333, 1),
    ("codebook", "uniform", 1, 2, 128, 2100, 8),
])
def test_attend_matches_oracle(kvc, kmode, vmode, B, H, D, S, rep):
    gk, gv, rk, rv = _layers(kvc, kmode, vmode, B, H, D, S, 9300 + S)
    q = torch.randn(B, H * rep, D, generator=torch.Generator().manual_seed(S), dtype=torch.float32)
    out = kvc.attend(gk, gv, q.to(_dev()))
    torch.cuda.synchronize()
    _check(out, gk, rk, gv, rv, q, 1.0 / math.sqrt(D))
    # an explicit scale, and the call repeated (the workspace is reused)
    out2 = kvc.attend(gk, gv, q.to(_dev()), scale=0.3)
    torch.cuda.synchronize()
    _check(out2, gk, rk, gv, rv, q, 0.3)


def test_attend_after_decode_appends(kvc):
    """Prefill, then single-token appends: attention sees every stored token."""
    B, H, D, S = 1, 2, 128, 400
    dev = _dev()
    pk = fit_codebook(D)
    gk = kvc.KVCacheLayer("codebook", B, H, D, in_dtype="f16", capacity=S, device=dev, **pk)
    gv = kvc.KVCacheLayer("int8", B, H, D, in_dtype="f16", capacity=S, device=dev)
    xk = synth.heavy_tailed_keys(B, H, S, D, seed=9400, dtype="f16").to(dev)
    xv = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=9401, tensor=1, dtype="f16").to(dev)
    gk.append(xk[:, :, :S - 3])
    gv.append(xv[:, :, :S - 3])
    for t in range(S - 3, S):
        gk.append(xk[:, :, t:t + 1])
        gv.append(xv[:, :, t:t + 1])
    rk = OracleLayer("codebook", B, H, D, capacity=S, **oracle_kwargs(pk))
    rv = OracleLayer("int8", B, H, D, capacity=S)
    q = torch.randn(B, 4 * H, D, generator=torch.Generator().manual_seed(1))
    out = kvc.attend(gk, gv, q.to(dev))
    torch.cuda.synchronize()
    _check(out, gk, rk, gv, rv, q, 1.0 / math.sqrt(D))


def test_attend_empty_and_rejections(kvc):
    B, H, D = 1, 2, 128
    dev = _dev()
    gk = kvc.KVCacheLayer("codebook", B, H, D, in_dtype="f16", capacity=8, device=dev,
                          **fit_codebook(D))
    gv = kvc.KVCacheLayer("int8", B, H, D, in_dtype="f16", capacity=8, device=dev)
    q = torch.randn(B, 2 * H, D, device=dev)
    out = torch.full((B, 2 * H, D), 3.0, dtype=torch.float16, device=dev)
    kvc.attend(gk, gv, q, out=out)                  # no stored token: zeros
    assert bool((out == 0).all())
    gk.append(torch.randn(B, H, 2, D, device=dev).half())
    with pytest.raises(kvc.KvcError) as e:          # values hold fewer tokens
        kvc.attend(gk, gv, q)
    assert e.value.status == -1
    gv.append(torch.randn(B, H, 2, D, device=dev).half())
    with pytest.raises(kvc.KvcError):               # Hq not a multiple of H
        kvc.attend(gk, gv, torch.randn(B, 3, D, device=dev))
    with pytest.raises(kvc.KvcError):               # values as keys: int8 keys unsupported
        kvc.attend(gv, gv, q)


@pytest.mark.slow
def test_attend_turboquant_full_size_sampled(kvc):
    """The TurboQuant-style workload at full size (B 16, H_kv 8, S 16384,
    codebook keys, int8 values) with 4 query heads per key/value head; eight
    (batch, query head) pairs checked against the oracle."""
    B, H, D, S, rep = 16, 8, 128, 16384, 4
    dev = _dev()
    xk = synth.heavy_tailed_keys(B, H, S, D, seed=4000, dtype="f16", device=dev)
    xv = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=4100, tensor=1, dtype="f16", device=dev,
                           work_dtype=torch.float32)
    pk = fit_codebook(D)
    gk = kvc.KVCacheLayer("codebook", B, H, D, in_dtype="f16", capacity=S, device=dev, **pk)
    gv = kvc.KVCacheLayer("int8", B, H, D, in_dtype="f16", capacity=S, device=dev)
    gk.append(xk)
    gv.append(xv)
    del xk, xv
    rk = OracleLayer("codebook", B, H, D, capacity=S, **oracle_kwargs(pk))
    rv = OracleLayer("int8", B, H, D, capacity=S)
    q = torch.randn(B, H * rep, D, generator=torch.Generator().manual_seed(7))
    out = kvc.attend(gk, gv, q.to(dev))
    torch.cuda.synchronize()
    rng = np.random.default_rng(8)
    pairs = {(B - 1, H * rep - 1)} | {(int(rng.integers(B)), int(rng.integers(H * rep)))
                                      for _ in range(7)}
    _check(out, gk, rk, gv, rv, q, 1.0 / math.sqrt(D), pairs=pairs)
