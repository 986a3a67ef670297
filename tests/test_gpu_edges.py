"""GPU parity at the method's edges, through the C ABI, against the float64 oracle.

Exact rounding ties and clamped latents decided by the tensor-core paths,
1- and 3-bit segments packed and unpacked by them, and the largest points of
the Llama-3-70B-like grid checked on seeded windows.  Where every value is
an exact tie the codes must equal the oracle's byte for byte, with no tie
allowance: the pages round half to even (numpy/mlx ``round``), and a
codebook value exactly between two centroids takes the lower one.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import codec
from oracle.layer import OracleLayer

from kvc_cases import MISMATCH_RATE, check_fetch, compare_codes, fit_uniform, oracle_kwargs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rank_quantized_kv_gb300 as kvc

    kvc.load_library()
    return kvc


def _dev():
    return torch.device("cuda:0")


def _exact_rows(gl, rl, x64):
    """Every slot's packed rows and side words equal the oracle's, byte for byte."""
    for s in range(rl.n_slots):
        rows, side = gl.slot_rows(s)
        ref_rows, ref_side = rl.encode(s, rl.slot_rows(x64, s))
        got = rows.cpu().numpy()
        if not np.array_equal(got, ref_rows):
            bits = rl.bits[rl.basis_of[s]] if rl.mode != "int8" else None
            cg, cr = codec.unpack_rows(got, bits), codec.unpack_rows(ref_rows, bits)
            bad = np.argwhere(cg != cr)
            t, k = bad[0]
            raise AssertionError(f"slot {s}: {len(bad)} codes differ, first token {t} comp {k}: "
                                 f"gpu {cg[t, k]} oracle {cr[t, k]}")
        if side is not None and ref_side.size:
            sg = side.cpu().numpy().view(np.uint16).reshape(-1)
            assert np.array_equal(sg, ref_side.view(np.uint16).reshape(-1)), f"slot {s}: side words"


def _unit_basis(d_in, r, rng):
    """V whose columns are distinct unit vectors: z_k = x_{perm(k)} exactly."""
    perm = rng.permutation(d_in)[:r]
    V = np.zeros((d_in, r), dtype=np.float32)
    V[perm, np.arange(r)] = 1.0
    return V, perm


# ------------------------------------------------------------------------- uniform ties

# widths in every segment the packer has (8, 4, 3, 2, 1), so the tensor-core
# append packs and the fetch decodes 1-bit and byte-straddling 3-bit segments
TIE_BITS = [8] * 4 + [4] * 8 + [3] * 8 + [2] * 6 + [1] * 6


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_uniform_exact_ties_and_clamps(kvc, dtype):
    """z_k = x_i exactly (unit-vector basis, zero mean), lo = 0, step = 1/4: each
    kept latent is u = 4 x_i = k + 1/2, an exact tie, rounded half to even; a
    quarter of them lie past either end of the code range and clamp."""
    B, H, D, S = 2, 2, 128, 300
    r = len(TIE_BITS)
    rng = np.random.default_rng(31)
    Vs, slots = [], B * H
    for _ in range(slots):
        Vs.append(_unit_basis(D, r, rng)[0])
    x = np.zeros((B, H, S, D))
    for b in range(B):
        for h in range(H):
            for k, w in enumerate(TIE_BITS):
                qmax = (1 << w) - 1
                # 2k+1 < 256 keeps (k + 1/2)/4 exact in bf16 (8 significant bits)
                hi = min(qmax + 2, 126)
                kk = rng.integers(-3, hi + 1, size=S)
                i = int(np.argmax(Vs[b * H + h][:, k]))
                x[b, h, :, i] = (kk + 0.5) / 4.0
    # components outside the basis carry other values (they do not enter z)
    free = rng.standard_normal(x.shape) * (np.abs(x) == 0)
    x = x + free
    xt = torch.from_numpy(x).to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    x64 = xt.double().numpy()
    params = dict(V=np.stack(Vs), mean=np.zeros((slots, D), np.float32),
                  bits=np.tile(np.array(TIE_BITS, np.uint8), (slots, 1)),
                  qmin=np.zeros((slots, r), np.float32), qstep=np.full((slots, r), 0.25, np.float32),
                  basis_of=np.arange(slots))
    gl = kvc.KVCacheLayer("uniform", B, H, D, in_dtype=dtype, capacity=S, device=_dev(), **params)
    rl = OracleLayer("uniform", B, H, D, capacity=S, **oracle_kwargs(params))
    gl.append(xt.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _exact_rows(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)
    assert gl.counters()["refined_codes"] > 0


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_uniform_one_and_three_bit_segments(kvc, dtype):
    """A fitted PCA basis at D = 128 whose widths include 1 and 3 bits: the
    tensor-core append packs every segment width and the fetch decodes them."""
    B, H, D, S = 2, 4, 128, 530
    x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=9100, tensor=0, n_outliers=3, dtype=dtype)
    x64 = x.double().numpy()
    p = fit_uniform(x64, 256, 48, [0, 1, 2, 3, 4, 8], 80)
    assert all(np.any(p["bits"] == w) for w in (1, 3)), p["bits"]
    gl = kvc.KVCacheLayer("uniform", B, H, D, in_dtype=dtype, capacity=S, device=_dev(), **p)
    rl = OracleLayer("uniform", B, H, D, capacity=S, **oracle_kwargs(p))
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    n = mism = 0
    for s in range(rl.n_slots):
        rows, _ = gl.slot_rows(s)
        c, m = compare_codes(rows.cpu().numpy(), None, rl, s, rl.slot_rows(x64, s))
        n, mism = n + c, mism + m
    assert mism <= MISMATCH_RATE * n
    check_fetch(gl.fetch(), gl, rl)


# ------------------------------------------------------------------------- codebook ties

def test_codebook_values_on_midpoints(kvc):
    """Identity rotation and a codebook with exact midpoints; every row has norm 8
    and entries in {0, +-1/2, +-1, +-3/2}, so each u = x_k / 8 is exactly a
    midpoint (0, +-1/16, +-1/8, +-3/16): the lower centroid wins every one."""
    B, H, D, S = 1, 4, 128, 260
    cb = (np.array([-1.75, -1.25, -0.75, -0.25, 0.25, 0.75, 1.25, 1.75]) / 8).astype(np.float32)
    rng = np.random.default_rng(32)
    x = np.zeros((B, H, S, D))
    for h in range(H):
        for t in range(S):
            mags = np.array([1.5] * 16 + [0.5] * 16 + [1.0] * 24 + [0.0] * 72)  # sum of squares 64
            row = mags * rng.choice([-1.0, 1.0], size=D)
            x[0, h, t] = rng.permutation(row)
    xt = torch.from_numpy(x).to(torch.float16)
    x64 = xt.double().numpy()
    params = dict(V=np.eye(D, dtype=np.float32), codebook=cb)
    gl = kvc.KVCacheLayer("codebook", B, H, D, in_dtype="f16", capacity=S, device=_dev(), **params)
    rl = OracleLayer("codebook", B, H, D, capacity=S, **oracle_kwargs(params))
    gl.append(xt.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _exact_rows(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)


# ------------------------------------------------------------------------- group ties

def test_group_exact_ties_and_zero_group(kvc):
    """Group mode (2 heads of D = 64, unit-vector basis, r = 96): a 4-bit group
    whose largest |z| is 7 (s = 1, z = k + 1/2 ties), a 2-bit group with |z|/s
    = 1/2 ties, and a 2-bit group that is all zero (s = 1e-8, fp16 0)."""
    B, H, D, S, hpg = 2, 4, 64, 200, 2
    d_in, r = hpg * D, 96
    bits = np.array([4] * 32 + [2] * 64, np.uint8)
    rng = np.random.default_rng(33)
    Hg = H // hpg
    Vs, perms = [], []
    for _ in range(Hg):
        V, perm = _unit_basis(d_in, r, rng)
        Vs.append(V)
        perms.append(perm)
    x = rng.standard_normal((B, H, S, D)) * 0.1
    for b in range(B):
        for g in range(Hg):
            rows = np.zeros((S, d_in))
            rows[:] = np.concatenate([x[b, g * hpg + j] for j in range(hpg)], axis=1)
            z = np.zeros((S, r))
            z[:, 0] = 7.0 * rng.choice([-1.0, 1.0], size=S)
            z[:, 1:32] = rng.integers(-7, 7, size=(S, 31)) + 0.5            # 4-bit ties
            z[:, 32] = 4.0 * rng.choice([-1.0, 1.0], size=S)
            z[:, 33:64] = 2.0 * rng.choice([-1.0, 0.0, 1.0], size=(S, 31))  # |z|/s = 1/2
            z[:, 64:96] = 0.0                                                # all-zero group
            rows[:, perms[g]] = z
            for j in range(hpg):
                x[b, g * hpg + j] = rows[:, j * D:(j + 1) * D]
    xt = torch.from_numpy(x).to(torch.bfloat16)
    x64 = xt.double().numpy()
    params = dict(V=np.stack(Vs), mean=np.zeros((Hg, d_in), np.float32),
                  bits=np.tile(bits, (Hg, 1)), basis_of=np.array([g for _ in range(B)
                                                                   for g in range(Hg)]),
                  heads_per_group=hpg, group_size=32)
    gl = kvc.KVCacheLayer("group", B, H, D, in_dtype="bf16", capacity=S, device=_dev(), **params)
    rl = OracleLayer("group", B, H, D, capacity=S, **oracle_kwargs(params))
    gl.append(xt.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _exact_rows(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)


# ------------------------------------------------------------------------- bounded waits

def test_wait_limit_times_out_and_recovers(kvc):
    """A wait limit far below a tile's load time makes the tensor-core append
    give up at its first wait: it drains its copies and MMAs, frees TMEM and
    returns; kvc_sync_status reports KVC_ETIMEOUT.  With the default limit
    restored the same layer appends correctly (the rows of the timed-out call
    are dropped first)."""
    B, H, D, S = 2, 4, 128, 700
    x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=9200, tensor=0, n_outliers=3, dtype="bf16")
    x64 = x.double().numpy()
    p = fit_uniform(x64, 512, 32, [0, 2, 4, 8], 128)
    gl = kvc.KVCacheLayer("uniform", B, H, D, in_dtype="bf16", capacity=S, device=_dev(), **p)
    with pytest.raises(kvc.KvcError) as e:
        gl.set_wait_limit(-1)
    assert e.value.status == -1
    xd = x.to(_dev())
    gl.set_wait_limit(1)
    gl.append(xd)
    assert gl.sync_status() == -5                  # KVC_ETIMEOUT, read once
    assert gl.sync_status() == 0                   # the error word was cleared
    assert gl.trim(S) == S
    gl.set_wait_limit(0)
    gl.append(xd)
    assert gl.sync_status() == 0
    rl = OracleLayer("uniform", B, H, D, capacity=S, **oracle_kwargs(p))
    rl.append(x64)
    n = mism = 0
    for s in range(rl.n_slots):
        rows, _ = gl.slot_rows(s)
        c, m = compare_codes(rows.cpu().numpy(), None, rl, s, rl.slot_rows(x64, s))
        n, mism = n + c, mism + m
    assert mism <= MISMATCH_RATE * n
    check_fetch(gl.fetch(), gl, rl)


# ------------------------------------------------------------------------- accounting

def test_fixed_bytes_match_the_golden_values(kvc):
    """kvc_nbytes' fixed bytes equal the values worked by hand from the pages'
    byte accounting (tests/golden/fixed_bytes.json, first case)."""
    import json
    from pathlib import Path

    case = json.loads((Path(__file__).parent / "golden" / "fixed_bytes.json").read_text())["cases"][0]
    nb, d_in, r = case["n_bases"], case["d_in"], case["r"]
    rng = np.random.default_rng(1)
    gl = kvc.KVCacheLayer("uniform", 1, nb, d_in, r=r, V=rng.standard_normal((nb, d_in, r)),
                          mean=np.zeros((nb, d_in)), bits=np.array(case["bits"], np.uint8),
                          qmin=np.zeros((nb, r)), qstep=np.ones((nb, r)), basis_of=np.arange(nb),
                          in_dtype="f32", capacity=4, device=_dev())
    assert gl.nbytes()["fixed"] == case["fixed"]


# ------------------------------------------------------------------------- grid windows

@pytest.mark.parametrize("r,bits", [(32, 2), (64, 4)])
def test_grid_largest_point_windows(kvc, r, bits):
    """The Llama-3-70B-like grid at its largest point (B = 64, H_kv = 8, D = 128,
    S = 128k: 8.4 M token-heads, 17 GB of bf16 input and of fp16 output, so
    element offsets pass 2^32), appended in 8192-token chunks and fetched in one
    call; the oracle checks four seeded (b, h) x 4096-token windows."""
    B, H, D, S, chunk = 64, 8, 128, 131072, 8192
    dev = _dev()
    src = synth.kv_spectral(1, H, chunk, D, alpha=1.0, seed=5000, tensor=0, dtype="f32",
                            device=dev, work_dtype=torch.float32)
    from rank_quantized_kv_gb300 import calib

    params = calib.fit_uniform_shared(src[:, :, :4096], r, bits)
    params["basis_of"] = np.array([h for _ in range(B) for h in range(H)], dtype=np.int32)
    gl = kvc.KVCacheLayer("uniform", B, H, D, in_dtype="bf16", capacity=S, device=dev, **params)
    x = torch.empty(B, H, S, D, dtype=torch.bfloat16, device=dev)
    gen = torch.Generator(device=dev)
    for c in range(S // chunk):
        gen.manual_seed(5100 + c)               # every batch entry and chunk its own rows
        xc = (src + 0.05 * torch.randn(B, H, chunk, D, generator=gen, device=dev)).to(torch.bfloat16)
        x[:, :, c * chunk:(c + 1) * chunk] = xc
        gl.append(xc)
        del xc
    assert gl.sync_status() == 0
    out = gl.fetch()
    torch.cuda.synchronize()
    rl = OracleLayer("uniform", B, H, D, capacity=S, **oracle_kwargs(params))
    rng = np.random.default_rng(77 + r)
    for _ in range(4):
        b, h = int(rng.integers(B)), int(rng.integers(H))
        if _ == 0:
            b, h = B - 1, H - 1                 # the last slot: the largest offsets
        t0 = int(rng.integers(0, S - 4096 + 1))
        s = b * H + h
        X = x[b, h, t0:t0 + 4096].double().cpu().numpy()
        rows, _side = gl.slot_rows(s)
        n, mism = compare_codes(rows[t0:t0 + 4096].cpu().numpy(), None, rl, s, X)
        assert mism <= MISMATCH_RATE * n
        ref = rl.decode(s, rows[t0:t0 + 4096].cpu().numpy(), None)
        o = out[b, h, t0:t0 + 4096].double().cpu().numpy()
        err = o - ref
        assert np.abs(err).max() <= 4e-3 * np.abs(ref).max()
        assert math.sqrt(np.mean(err ** 2)) <= 1e-3 * math.sqrt(np.mean(ref ** 2))
    del out, x
    gl.close()
    torch.cuda.empty_cache()
