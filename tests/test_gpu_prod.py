"""GPU parity of codebook keys with the TurboQuantProd residual sketch and the
outlier two-stream store (kvc_init_layer_prod, kvc_fit_outliers) against the
float64 oracle (oracle/prod.py).

* outlier codes and scales, fp16 norms: exact;
* centroid indices: exact, except at an oracle near-tie (|u - midpoint| <=
  1e-6) at a rate <= 1e-6;
* sign bits: exact, except where the oracle's (S r)_j is within
  1e-9 ||S_j|| ||r|| of 0 (keys whose indices differ at a near-tie are left
  out: their residual differs);
* residual norms: the GPU rounds its fp32 ||r|| to fp16: within one fp16 ulp;
* fetch: within max-abs 4e-3 max|x_hat| and RMS 1e-3 RMS(x_hat) per head of the
  oracle's decode of the GPU's own rows.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import fit, prod

pytestmark = pytest.mark.gpu

TIE_U = 1e-6
TIE_S = 1e-9
MISMATCH_RATE = 1e-6


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rank_quantized_kv_gb300 as kvc

    kvc.load_library()
    return kvc


def _dev():
    return torch.device("cuda:0")


def _keys(B, H, T, D, seed, dtype="f16", n_big=4):
    """Heavy-tailed keys with n_big channels per head scaled by 6."""
    x = synth.heavy_tailed_keys(B, H, T, D, seed=seed, dtype="f32").double()
    g = torch.Generator().manual_seed(seed + 1)
    for b in range(B):
        for h in range(H):
            ch = torch.randperm(D, generator=g)[:n_big]
            x[b, h][:, ch] *= 6.0
    return x.to(synth._DTYPES[dtype])


def _params(D, m, b_mse, seed):
    R = fit.seeded_rotation(D, seed).astype(np.float32)
    cb = fit.lloyd_max_gaussian(1 << b_mse, 1 / math.sqrt(D)).astype(np.float32)
    S = np.random.default_rng(seed).standard_normal((m, D)).astype(np.float32) if m else None
    return R, cb, S


def _x_in(X, ch, t0, split_from):
    X = X.copy()
    if ch is not None and len(ch):
        for t in range(X.shape[0]):
            if t0 + t >= split_from:
                X[t, ch] = 0.0
    return X


def _compare(gl, ol, x64, split_from):
    """Rows and side words of every slot; returns (codes, index mismatches, sign mismatches)."""
    n_codes = n_idx = n_sgn = n_sig = 0
    mids = 0.5 * (ol.centroids[:-1] + ol.centroids[1:])
    for s in range(ol.n_slots):
        b, h = divmod(s, ol.H)
        rows, side = gl.slot_rows(s)
        rows = rows.cpu().numpy()
        side = side.cpu().numpy().view(np.float16).reshape(rows.shape[0], -1)
        eg = ol.unpack(s, rows, side)
        eo = ol.enc[s]
        if ol.n_out:
            assert np.array_equal(eg["o8"], eo["o8"]), f"slot {s}: outlier codes"
            assert np.array_equal(eg["oscale16"].view(np.uint16), eo["oscale16"].view(np.uint16))
        assert np.array_equal(eg["norm16"].view(np.uint16), eo["norm16"].view(np.uint16)), \
            f"slot {s}: norms"
        ch = None if ol.channels is None else ol.channels[s]
        X = _x_in(x64[b, h], ch, 0, split_from)
        bad = np.argwhere(eg["idx"] != eo["idx"])
        if len(bad):
            n = np.sqrt(np.sum(X * X, axis=1))
            u = (X @ ol.R) / np.where(n > 0, n, 1.0)[:, None]
            for t, k in bad:
                d = np.min(np.abs(u[t, k] - mids))
                assert d <= TIE_U, f"slot {s} key {t} comp {k}: index differs {d:.3e} from a midpoint"
        n_codes += eo["idx"].size
        n_idx += len(bad)
        if ol.m:
            same_idx = np.all(eg["idx"] == eo["idx"], axis=1)
            x_mse = (eo["norm16"].astype(np.float64)[:, None] * ol.centroids[eo["idx"]]) @ ol.R.T
            r = X - x_mse
            proj = r @ ol.S.T
            scale = np.linalg.norm(ol.S, axis=1)[None, :] * np.linalg.norm(r, axis=1)[:, None]
            sb = (eg["beta"] != eo["beta"]) & same_idx[:, None]
            for t, j in np.argwhere(sb):
                assert abs(proj[t, j]) <= TIE_S * scale[t, j], \
                    f"slot {s} key {t} sign {j}: S r = {proj[t, j]:.3e}"
            n_sgn += int(sb.sum())
            n_sig += eo["beta"].size
            g = eg["gamma16"].astype(np.float64)
            o = eo["gamma16"].astype(np.float64)
            ulp = np.spacing(eo["gamma16"]).astype(np.float64)
            assert np.all(np.abs(g - o) <= ulp * (1 + 1e-9)), f"slot {s}: residual norms"
    assert n_idx <= MISMATCH_RATE * n_codes + 0.5
    assert n_sgn <= MISMATCH_RATE * max(n_sig, 1) + 0.5
    return n_codes, n_idx, n_sgn


def _check_fetch(gl, ol):
    out = gl.fetch().float().cpu().numpy().astype(np.float64)
    for s in range(ol.n_slots):
        b, h = divmod(s, ol.H)
        rows, side = gl.slot_rows(s)
        rows = rows.cpu().numpy()
        side = side.cpu().numpy().view(np.float16).reshape(rows.shape[0], -1)
        ref = ol.decode(s, ol.unpack(s, rows, side))
        err = out[b, h] - ref
        mx = max(np.abs(ref).max(), 1e-30)
        rms = max(math.sqrt(np.mean(ref ** 2)), 1e-30)
        assert np.abs(err).max() / mx <= 4e-3, f"slot {s}: max-abs"
        assert math.sqrt(np.mean(err ** 2)) / rms <= 1e-3, f"slot {s}: RMS"


def _layers(kvc, B, H, D, T, m, b_mse, n_out, split_from, x, seed, dtype, channels=None):
    R, cb, S = _params(D, m, b_mse, seed)
    if n_out and channels is None:
        x64 = x.double().numpy()
        channels = np.stack([prod.outlier_channels(x64[b, h, :split_from + 1], n_out)
                             for b in range(B) for h in range(H)])
    gl = kvc.KVCacheLayer("codebook", B, H, D, V=R, codebook=cb, in_dtype=dtype, capacity=T,
                          device=_dev(), sketch=S, outlier_channels=channels if n_out else None,
                          split_from=split_from)
    ol = prod.ProdKeyLayer(B, H, D, R=R, centroids=cb, S=S,
                           channels=channels if n_out else None, split_from=split_from)
    return gl, ol


CASES = {
    # name: B, H, D, T, m, b_mse, n_out, split_from, dtype
    "prod-outliers-d128": (2, 2, 128, 300, 128, 2, 8, 63, "f16"),
    "prod-d64-bf16": (1, 3, 64, 200, 64, 3, 0, 0, "bf16"),
    "outliers-only-d128": (1, 2, 128, 150, 0, 3, 4, 31, "f16"),
    "prod-d32-f32": (2, 1, 32, 97, 32, 1, 3, 10, "f32"),
    "prod-m16-4bit": (1, 2, 128, 70, 16, 4, 2, 0, "f16"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prod_append_and_fetch_match_the_oracle(kvc, name):
    B, H, D, T, m, b_mse, n_out, split_from, dt = CASES[name]
    x = _keys(B, H, T, D, seed=7100 + T, dtype=dt)
    gl, ol = _layers(kvc, B, H, D, T, m, b_mse, n_out, split_from, x, 7200 + D, dt)
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    x64 = x.double().numpy()
    ol.append(x64)
    n, ni, ns = _compare(gl, ol, x64, split_from)
    print(f"{name}: {n} codes, {ni} index / {ns} sign near-tie mismatches, counters {gl.counters()}")
    _check_fetch(gl, ol)
    nb = gl.nbytes()
    assert nb["payload"] + nb["side"] == prod.memory_bytes(T, D, b_mse, m, n_out, values=False) * B * H
    assert nb["fixed"] == 0


def test_prod_streaming_equals_bulk(kvc):
    """Keys appended one call at a time across the split store what one call stores."""
    B, H, D, T, m, b_mse, n_out, split_from = 1, 2, 64, 40, 32, 2, 3, 17
    x = _keys(B, H, T, D, seed=7300)
    bulk, _ = _layers(kvc, B, H, D, T, m, b_mse, n_out, split_from, x, 7301, "f16")
    step, _ = _layers(kvc, B, H, D, T, m, b_mse, n_out, split_from, x, 7301, "f16")
    xd = x.to(_dev())
    bulk.append(xd)
    for t0, t1 in ((0, 1), (1, 16), (16, 17), (17, 18), (18, 40)):
        step.append(xd[:, :, t0:t1])
    assert bulk.sync_status() == 0 and step.sync_status() == 0
    for s in range(B * H):
        rb, sb = bulk.slot_rows(s)
        rs, ss = step.slot_rows(s)
        assert torch.equal(rb, rs) and torch.equal(sb, ss)


def test_no_sketch_no_outliers_is_the_codebook_mode(kvc):
    """With m = 0 and no outlier channels the prod layer stores the codebook
    mode's rows and norms."""
    B, H, D, T = 1, 2, 128, 100
    x = _keys(B, H, T, D, seed=7400)
    R, cb, _ = _params(D, 0, 3, 7401)
    gp = kvc.KVCacheLayer("codebook", B, H, D, V=R, codebook=cb, in_dtype="f16", capacity=T,
                          device=_dev(), outlier_channels=np.zeros((B * H, 0), dtype=np.int32))
    gc = kvc.KVCacheLayer("codebook", B, H, D, V=R, codebook=cb, in_dtype="f16", capacity=T,
                          device=_dev())
    xd = x.to(_dev())
    gp.append(xd)
    gc.append(xd)
    for s in range(B * H):
        rp, sp = gp.slot_rows(s)
        rc, sc = gc.slot_rows(s)
        # indices may differ only at near-ties decided by the two kernels' own paths
        assert (rp != rc).sum().item() <= 2
        assert torch.equal(sp, sc)


def test_fit_outliers_matches_the_oracle(kvc):
    B, H, D, T, n_calib, n_out = 2, 3, 128, 90, 64, 8
    x = _keys(B, H, T, D, seed=7500, n_big=6)
    ch = kvc.fit_outliers(x.to(_dev()), n_calib, n_out).cpu().numpy()
    x64 = x.double().numpy()
    for b in range(B):
        for h in range(H):
            ref = prod.outlier_channels(x64[b, h, :n_calib], n_out)
            assert np.array_equal(ch[b * H + h], ref)


def test_prod_layer_rejects_bad_descriptors(kvc):
    D = 64
    R, cb, S = _params(D, 32, 2, 1)
    base = dict(V=R, codebook=cb, in_dtype="f16", capacity=8, device=_dev())
    with pytest.raises(kvc.KvcError):   # m not a multiple of 16
        kvc.KVCacheLayer("codebook", 1, 1, D, sketch=S[:24], **base)
    with pytest.raises(kvc.KvcError):   # channels not ascending
        kvc.KVCacheLayer("codebook", 1, 1, D, outlier_channels=[[5, 3]], **base)
    with pytest.raises(kvc.KvcError):   # D not in {32, 64, 128}
        kvc.KVCacheLayer("codebook", 1, 1, 96, V=fit.seeded_rotation(96, 1).astype(np.float32),
                         codebook=cb, in_dtype="f16", capacity=8, device=_dev(),
                         sketch=np.ones((16, 96), dtype=np.float32))
    with pytest.raises(kvc.KvcError):   # uniform mode
        kvc.KVCacheLayer("uniform", 1, 1, D, V=R[:, :8], bits=np.full(8, 2), qmin=np.zeros(8),
                         qstep=np.ones(8), in_dtype="f16", capacity=8, device=_dev(), sketch=S)


@pytest.mark.parametrize("D,m,n_out,Hq", [(128, 128, 8, 8), (64, 64, 0, 2), (128, 0, 4, 4)])
def test_prod_attend_matches_the_oracle(kvc, D, m, n_out, Hq):
    """kvc_attend over sketch / outlier keys and int8 values against the
    oracle's score estimate (plus the outlier term) over the GPU's own rows,
    softmax(scores / sqrt(D)) and the int8 decode of the values."""
    from oracle.attend import softmax

    B, H, T, split_from = 2, 2, 333, 40
    x = _keys(B, H, T, D, seed=7600 + D)
    v = synth.kv_spectral(B, H, T, D, alpha=1.0, seed=7601, tensor=1, dtype="f16")
    gl, ol = _layers(kvc, B, H, D, T, m, 2, n_out, split_from, x, 7602, "f16")
    gv = kvc.KVCacheLayer("int8", B, H, D, in_dtype="f16", capacity=T, device=_dev())
    gl.append(x.to(_dev()))
    gv.append(v.to(_dev()))
    q = torch.randn(B, Hq, D, generator=torch.Generator().manual_seed(7603)).to(_dev())
    out = kvc.attend(gl, gv, q).float().cpu().numpy().astype(np.float64)
    assert gl.sync_status() == 0
    qn = q.double().cpu().numpy()
    rep = Hq // H
    for b in range(B):
        for hq in range(Hq):
            s = b * H + hq // rep
            rows, side = gl.slot_rows(s)
            rows = rows.cpu().numpy()
            side = side.cpu().numpy().view(np.float16).reshape(rows.shape[0], -1)
            sc = ol.scores(s, qn[b, hq], ol.unpack(s, rows, side))
            p = softmax(sc / math.sqrt(D))
            vr, vs = gv.slot_rows(s)
            V = vr.cpu().numpy().view(np.int8).astype(np.float64) * \
                vs.cpu().numpy().view(np.float16).astype(np.float64)[:, :1]
            ref = p @ V
            err = out[b, hq] - ref
            assert np.abs(err).max() <= 4e-3 * np.abs(ref).max(), (b, hq)
            assert math.sqrt(np.mean(err ** 2)) <= 1e-3 * math.sqrt(np.mean(ref ** 2)), (b, hq)
