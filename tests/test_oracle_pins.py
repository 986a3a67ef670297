"""Pins of the float64 oracle to things other than itself.

Each test ties an oracle function to the pages' printed layouts, a hand
worked example under tests/golden/, a closed form, a textbook table, a
library routine or brute force -- chosen so that a dropped term, a wrong
sign, index or bit order fails one of them.
"""
import itertools
import json
import math
from pathlib import Path

import numpy as np
import pytest

from oracle import codec, fit
from oracle.layer import OracleLayer

GOLDEN = Path(__file__).parent / "golden"


def _golden(name):
    return json.loads((GOLDEN / name).read_text())


# ---------------------------------------------------------------- bit packing

def test_pack_golden_rows():
    for case in _golden("bitpack.json")["cases"]:
        row = codec.pack_rows(np.array([case["codes"]]), case["bits"])[0]
        assert row.tolist() == case["row"], case["why"]
        back = codec.unpack_rows(row[None, :], case["bits"])[0]
        kept = np.array(case["bits"]) > 0
        assert np.array_equal(back[kept], np.array(case["codes"])[kept])


@pytest.mark.parametrize("d", [8, 37, 128])
def test_pack_matches_printed_1bit_unpack(d):
    # turboquant_cache page, _unpack_indices_block, b == 1 branch
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 2, size=(50, d))
    rows = codec.pack_rows(codes, [1] * d)
    bits = np.unpackbits(rows, axis=1, bitorder="little")
    assert np.array_equal(bits[:, :d], codes)


@pytest.mark.parametrize("d", [4, 30, 128])
def test_pack_matches_printed_2bit_unpack(d):
    # turboquant_cache page, _unpack_indices_block, b == 2 branch
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 4, size=(50, d))
    rows = codec.pack_rows(codes, [2] * d)
    shifts = np.array([0, 2, 4, 6], dtype=np.uint8)
    vals = ((rows[:, :, None] >> shifts[None, None, :]) & 0x3).reshape(50, -1)
    assert np.array_equal(vals[:, :d], codes)


@pytest.mark.parametrize("d", [2, 33, 128])
def test_pack_matches_printed_4bit_unpack(d):
    # turboquant_cache page, _unpack_indices_block, b == 4 branch
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, size=(50, d))
    rows = codec.pack_rows(codes, [4] * d)
    shifts = np.array([0, 4], dtype=np.uint8)
    vals = ((rows[:, :, None] >> shifts[None, None, :]) & 0xF).reshape(50, -1)
    assert np.array_equal(vals[:, :d], codes)


def test_pack_3bit_every_stream_bit():
    # A 3-bit code straddling bytes: check each stored bit against the
    # little-endian stream position it must occupy, for every code value in
    # every one of the 8 alignments.
    d = 8
    for v in range(8):
        for m in range(d):
            codes = np.zeros((1, d), dtype=np.int64)
            codes[0, m] = v
            row = codec.pack_rows(codes, [3] * d)[0]
            assert row.shape[0] == 3
            for i in range(24):
                expect = (v >> (i - 3 * m)) & 1 if 3 * m <= i < 3 * m + 3 else 0
                assert (row[i // 8] >> (i % 8)) & 1 == expect


@pytest.mark.parametrize("d,b", [(128, 3), (128, 1), (128, 2), (128, 4), (64, 3), (10, 3), (7, 1)])
def test_packed_length_formula(d, b):
    # turboquant_cache page: _idx_packed_len = ceil(d * b_mse / 8); 128 x 3 bits = 48 bytes
    assert codec.row_bytes([b] * d) == math.ceil(d * b / 8)


def test_roundtrip_mixed_widths():
    rng = np.random.default_rng(4)
    bits = rng.choice([0, 1, 2, 3, 4, 8], size=41)
    codes = np.stack([rng.integers(0, 1 << int(b), size=200) if b else np.zeros(200, int)
                      for b in bits], axis=1)
    rows = codec.pack_rows(codes, bits)
    assert rows.shape[1] == sum(math.ceil(int(np.sum(bits == w)) * w / 8) for w in (1, 2, 3, 4, 8))
    assert np.array_equal(codec.unpack_rows(rows, bits), codes)


# ---------------------------------------------------------------- PCA

def test_pca_recovers_known_covariance():
    # Rows built so that their covariance is exactly U diag(a^2) U^T.
    rng = np.random.default_rng(5)
    S, D = 64, 6
    M = rng.standard_normal((S, D))
    M -= M.mean(axis=0)
    Hq, _ = np.linalg.qr(M)                      # orthonormal, zero-mean columns
    U, _ = np.linalg.qr(rng.standard_normal((D, D)))
    a = np.array([3.0, 2.0, 1.5, 1.0, 0.5, 0.25])
    mu = rng.standard_normal(D)
    X = mu + math.sqrt(S) * Hq @ np.diag(a) @ U.T
    mean, lam, V = fit.pca_fit(X)
    assert np.allclose(mean, mu, atol=1e-12)
    assert np.allclose(lam, a ** 2, rtol=1e-10)
    # columns equal up to sign, and the sign rule holds
    assert np.allclose(np.abs(V.T @ U), np.eye(D), atol=1e-9)
    piv = np.argmax(np.abs(V), axis=0)
    assert np.all(V[piv, np.arange(D)] > 0)


def test_pca_matches_svd():
    rng = np.random.default_rng(6)
    X = rng.standard_normal((300, 12)) @ rng.standard_normal((12, 12)) + 3.0
    mean, lam, V = fit.pca_fit(X)
    _, sv, Vt = np.linalg.svd(X - X.mean(axis=0), full_matrices=False)
    assert np.allclose(lam, sv ** 2 / X.shape[0], rtol=1e-10)
    assert np.allclose(np.abs(V.T @ Vt.T), np.eye(12), atol=1e-8)


def test_pca_needs_two_rows():
    with pytest.raises(ValueError):
        fit.pca_fit(np.ones((1, 4)))


# ---------------------------------------------------------------- DP allocation

def test_dp_golden():
    for case in _golden("dp_allocation.json")["cases"]:
        bits = fit.dp_allocate(case["lam"], case["choices"], case["budget"])
        assert sum(bits) <= case["budget"]
        assert fit.allocation_distortion(case["lam"], bits) == pytest.approx(case["min"], rel=1e-12)
        assert list(bits) in [list(m) for m in case["minimisers"]]
        best, arg = fit.brute_force_allocate(case["lam"], case["choices"], case["budget"])
        assert best == pytest.approx(case["min"], rel=1e-12)
        assert sorted(map(list, arg)) == sorted(case["minimisers"])


@pytest.mark.parametrize("seed", range(25))
def test_dp_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    r = int(rng.integers(1, 9))
    choices = sorted(set(rng.choice([0, 1, 2, 3, 4, 8], size=int(rng.integers(2, 5)))) | {0})
    lam = np.sort(rng.exponential(size=r) ** 2)[::-1] if seed % 2 else rng.exponential(size=r)
    budget = int(rng.integers(0, 4 * r + 1))
    bits = fit.dp_allocate(lam, choices, budget)
    best, arg = fit.brute_force_allocate(lam, choices, budget)
    assert sum(bits) <= budget and all(b in choices for b in bits)
    assert fit.allocation_distortion(lam, bits) == pytest.approx(best, rel=1e-12, abs=1e-300)
    assert tuple(int(b) for b in bits) in arg


def test_dp_monotone_in_lambda():
    # exchange argument: a larger eigenvalue never gets fewer bits
    rng = np.random.default_rng(7)
    for _ in range(20):
        lam = np.sort(rng.exponential(size=32))[::-1]
        bits = fit.dp_allocate(lam, [0, 2, 4, 8], 128)
        assert np.all(np.diff(bits) <= 0)


def test_dp_scale_invariant():
    rng = np.random.default_rng(8)
    lam = rng.exponential(size=16)
    b1 = fit.dp_allocate(lam, [0, 1, 2, 4, 8], 48)
    b2 = fit.dp_allocate(lam * 1024.0, [0, 1, 2, 4, 8], 48)
    assert np.array_equal(b1, b2)


def test_dp_rejects_negative_budget():
    # kvtc_cache page: KVTCKVCache raises on kvtc_bit_budget < 0
    with pytest.raises(ValueError):
        fit.dp_allocate([1.0], [0, 1], -1)


# ---------------------------------------------------------------- Lloyd-Max

def test_lloyd_max_matches_max_table():
    table = _golden("lloyd_max_gaussian.json")["levels"]
    for levels, row in table.items():
        c = fit.lloyd_max_gaussian(int(levels))
        half = c[int(levels) // 2:]
        assert np.allclose(half, row["outputs"], atol=6e-4)
        assert np.allclose(c, -c[::-1], atol=1e-12)          # symmetric
        # mean squared error of the fixed point, by numerical integration
        t = np.concatenate(([-12.0], 0.5 * (c[:-1] + c[1:]), [12.0]))
        mse = 0.0
        for j in range(len(c)):
            xs = np.linspace(t[j], t[j + 1], 20001)
            f = np.exp(-xs ** 2 / 2) / math.sqrt(2 * math.pi) * (xs - c[j]) ** 2
            mse += np.trapezoid(f, xs)
        assert mse == pytest.approx(row["mse"], rel=2e-3)


def test_lloyd_max_two_levels_closed_form():
    # two levels: +-E|X| = +-sqrt(2/pi) sigma
    c = fit.lloyd_max_gaussian(2, sigma=0.3)
    assert c[1] == pytest.approx(0.3 * math.sqrt(2 / math.pi), rel=1e-10)


def test_lloyd_max_scales_with_sigma():
    c1 = fit.lloyd_max_gaussian(8)
    c2 = fit.lloyd_max_gaussian(8, sigma=1 / math.sqrt(128))
    assert np.allclose(c2, c1 / math.sqrt(128), rtol=1e-12)


# ---------------------------------------------------------------- rotation

def test_rotation_orthogonal_and_qr_unique():
    R = fit.seeded_rotation(64, 1234)
    assert np.allclose(R @ R.T, np.eye(64), atol=1e-12)
    G = np.random.default_rng(1234).standard_normal((64, 64))
    Rt = R.T @ G                                       # the triangular factor
    assert np.allclose(np.tril(Rt, -1), 0, atol=1e-10)
    assert np.all(np.diag(Rt) > 0)
    assert np.array_equal(R, fit.seeded_rotation(64, 1234))
    assert not np.allclose(R, fit.seeded_rotation(64, 1235))


# ---------------------------------------------------------------- quantisers

def test_uniform_params_hand_worked():
    """Frozen minimum and step of the fit rows (kvtc_cache page,
    ``_TensorKVTC._requantize``: ``quantize_component`` gives each surviving
    component a minimum and a scale).  Worked by hand: the minimum of each
    column, and (max - min) / (2^b - 1) as the step; a constant column takes
    the 1e-8 floor; a dropped column takes nothing."""
    Z = np.array([[1.0, -2.0, 5.0, 7.0],
                  [3.0, 0.0, 5.0, 1.0],
                  [2.0, 4.0, 5.0, -3.0]])
    lo, step = fit.uniform_params(Z, [2, 1, 3, 0])
    assert lo.tolist() == [1.0, -2.0, 5.0, 0.0]
    assert step[0] == 2.0 / 3.0           # (3 - 1) / (2^2 - 1)
    assert step[1] == 6.0                 # (4 - (-2)) / (2^1 - 1)
    assert step[2] == 1e-8                # constant column: the floor
    assert step[3] == 0.0                 # 0 bits: not stored
    lo8, step8 = fit.uniform_params(Z[:, :1], [8])
    assert lo8[0] == 1.0 and step8[0] == 2.0 / 255.0


@pytest.mark.parametrize("b", [1, 2, 3, 4, 8])
def test_uniform_params_span_the_code_range(b):
    """On its own fit rows the frozen quantiser uses every end of the code
    range: the row holding a column's minimum gets code 0, the row holding its
    maximum gets 2^b - 1, and every fit row decodes within half a step.  A step
    of (max - min) / 2^b, or a minimum off by a row, fails one of these."""
    rng = np.random.default_rng(40 + b)
    Z = rng.standard_normal((300, 5)) * np.array([3.0, 1.0, 0.2, 7.0, 0.01]) + 2.0
    bits = [b] * 5
    lo, step = fit.uniform_params(Z, bits)
    codes = codec.quantize_uniform(Z, lo, step, bits)
    qmax = (1 << b) - 1
    for k in range(5):
        assert codes[np.argmin(Z[:, k]), k] == 0
        assert codes[np.argmax(Z[:, k]), k] == qmax
        assert codes[:, k].min() == 0 and codes[:, k].max() == qmax
    zhat = codec.dequantize_uniform(codes, lo, step, bits)
    assert np.all(np.abs(zhat - Z) <= step / 2 * (1 + 1e-12))


def test_fixed_bytes_golden():
    """The frozen-parameter bytes the stored size carries, against values worked
    by hand from the pages' byte accounting (tests/golden/fixed_bytes.json)."""
    rng = np.random.default_rng(5)
    for case in _golden("fixed_bytes.json")["cases"]:
        mode, d_in = case["mode"], case["d_in"]
        if mode == "int8":
            L = OracleLayer("int8", 1, 2, d_in)
        elif mode == "codebook":
            L = OracleLayer("codebook", 1, 2, d_in, V=np.eye(d_in),
                            codebook=[-1.0, -0.3, 0.3, 1.0])
        elif mode == "group":
            hpg = case["hpg"]
            nb, r = case["n_bases"], case["r"]
            D = d_in // hpg
            L = OracleLayer("group", 1, nb * hpg, D, heads_per_group=hpg,
                            V=np.zeros((nb, d_in, r)), mean=np.zeros((nb, d_in)),
                            bits=[[4] * (r // 4) + [2] * (r - r // 4)] * nb, group_size=32,
                            basis_of=np.arange(nb))
        else:
            nb, r = case["n_bases"], case["r"]
            bits = np.array(case["bits"])
            L = OracleLayer("uniform", 1, nb, d_in, V=rng.standard_normal((nb, d_in, r)),
                            mean=rng.standard_normal((nb, d_in)), bits=bits,
                            qmin=np.zeros((nb, r)), qstep=np.ones((nb, r)),
                            basis_of=np.arange(nb))
        assert L.param_bytes() == case["fixed"], case["why"]
        assert L.nbytes()["fixed"] == case["fixed"]


def test_uniform_ties_round_half_to_even():
    lo, step = np.array([0.0]), np.array([0.25])         # exact binary fractions
    z = (np.arange(16) + 0.5)[:, None] * 0.25
    codes = codec.quantize_uniform(z, lo, step, [4])[:, 0]
    expect = [k if k % 2 == 0 else k + 1 for k in range(16)]
    assert codes.tolist() == [min(e, 15) for e in expect]


def test_uniform_clamps_out_of_range():
    codes = codec.quantize_uniform(np.array([[-5.0], [0.1], [99.0]]), [0.0], [1.0], [2])[:, 0]
    assert codes.tolist() == [0, 0, 3]


def test_uniform_code_error_within_half_step():
    rng = np.random.default_rng(9)
    z = rng.uniform(-1, 3, size=(500, 3))
    lo, step = np.array([-1.0, -1.0, -1.0]), np.array([4 / 255, 4 / 15, 4 / 3])
    bits = [8, 4, 2]
    zhat = codec.dequantize_uniform(codec.quantize_uniform(z, lo, step, bits), lo, step, bits)
    assert np.all(np.abs(zhat - z) <= step / 2 + 1e-12)


def test_all_dropped_reconstructs_mean():
    rng = np.random.default_rng(10)
    D, r = 16, 4
    V, _ = np.linalg.qr(rng.standard_normal((D, D)))
    mean = rng.standard_normal(D)
    L = OracleLayer("uniform", 1, 2, D, V=V[:, :r], mean=mean, bits=[0] * r,
                    qmin=[0.0] * r, qstep=[0.0] * r)
    L.append(rng.standard_normal((1, 2, 5, D)))
    assert L.nbytes()["payload"] == 0
    assert np.array_equal(L.fetch(), np.broadcast_to(mean, (1, 2, 5, D)))


def test_full_rank_8bit_near_lossless():
    # r = D at 8 bits: the error vector is sum_k e_k V_k with |e_k| <= step_k/2
    rng = np.random.default_rng(11)
    D, S = 16, 400
    X = rng.standard_normal((S, D)) @ np.diag(np.linspace(2, 0.2, D)) + 1.0
    mean, lam, V = fit.pca_fit(X)
    bits = np.full(D, 8)
    lo, step = fit.uniform_params(codec.project(X, mean, V), bits)
    L = OracleLayer("uniform", 1, 1, D, V=V, mean=mean, bits=bits, qmin=lo, qstep=step)
    L.append(X[None, None])
    err = np.linalg.norm(L.fetch()[0, 0] - X, axis=1)
    assert np.all(err <= math.sqrt(np.sum((step / 2) ** 2)) * (1 + 1e-9))
    assert np.max(err) / np.max(np.linalg.norm(X, axis=1)) < 2e-2


def test_group_dominant_entry_and_zero_group():
    bits = [4] * 4 + [2] * 4
    z = np.array([[10.0, 0.5, -0.2, 0.0, 0.0, 0.0, 0.0, 0.0],
                  [0.0, 0.0, 0.0, 0.0, -3.0, 1.6, 1.4, 0.0]])
    codes, scales = codec.quantize_group(z, bits, 4)
    # row 0: 4-bit group absmax 10 -> s = 10/7, 10 -> +7 -> code 15; zero 2-bit group
    assert codes[0, 0] == 15 and float(scales[0, 0]) == pytest.approx(10 / 7, rel=1e-3)
    assert codes[0, 1] == 8 + int(np.rint(0.5 / (10 / 7)))
    assert np.all(codes[0, 4:] == 2) and float(scales[0, 1]) == 0.0   # fp16(1e-8) == 0
    # row 1: 2-bit group absmax 3 -> s = 3: -3 -> -1 -> 1; 1.6/3 = 0.53 -> 1 -> 3; 1.4/3 -> 0 -> 2
    assert codes[1, 4:].tolist() == [1, 3, 2, 2]
    assert np.all(codes[1, :4] == 8)
    zhat = codec.dequantize_group(codes, scales, bits, 4)
    assert zhat[1, 4] == -float(scales[1, 1]) and zhat[0, 0] == 7 * float(scales[0, 0])


def test_group_codes_symmetric_and_within_half_scale():
    """Random latents at mixed widths: every code lies in [1, 2^b - 1] (symmetric
    around 2^(b-1)); each group's largest |z| takes the extreme code; and the
    decode is within half a scale of z plus the fp16 rounding of the scale,
    |zhat - z| <= s/2 + qmax |fp16(s) - s| (q is taken with the unrounded s)."""
    rng = np.random.default_rng(13)
    bits = [4] * 12 + [2] * 36
    z = rng.standard_normal((300, 48)) * np.linspace(3.0, 0.05, 48)
    codes, scales = codec.quantize_group(z, bits, 16)
    zhat = codec.dequantize_group(codes, scales, bits, 16)
    for g, (w, comps) in enumerate(codec.group_ranges(bits, 16)):
        qmax, off = (1 << (w - 1)) - 1, 1 << (w - 1)
        c = codes[:, comps].astype(np.int64)
        assert c.min() >= off - qmax and c.max() <= off + qmax
        zg = z[:, comps]
        s = np.maximum(np.abs(zg).max(axis=1) / qmax, 1e-8)
        s16 = np.asarray(scales[:, g], dtype=np.float64)
        assert np.array_equal(s16, s.astype(np.float16).astype(np.float64))
        top = np.argmax(np.abs(zg), axis=1)
        q_top = c[np.arange(len(top)), top] - off
        assert np.array_equal(q_top, np.sign(zg[np.arange(len(top)), top]).astype(np.int64) * qmax)
        bound = s / 2 + qmax * np.abs(s16 - s)
        assert np.all(np.abs(zhat[:, comps] - zg) <= bound[:, None] * (1 + 1e-12))


def test_group_ranges_cfg3_split():
    bits = fit.palu_bits(256, 4, 2, 0.25)
    g = codec.group_ranges(bits, 32)
    assert [w for w, _ in g] == [4, 4, 2, 2, 2, 2, 2, 2]
    assert all(len(c) == 32 for _, c in g)
    # effective bits (palu_cache page, "Byte accounting"): (r / D_in) * avg bits
    assert codec.row_bytes(bits) * 8 / 1024 == pytest.approx((256 / 1024) * 2.5)


def test_codebook_zero_and_fine_grid():
    rng = np.random.default_rng(12)
    d = 32
    R = fit.seeded_rotation(d, 5)
    c8 = fit.lloyd_max_gaussian(64, sigma=1 / math.sqrt(d))
    idx, n16 = codec.quantize_codebook(np.zeros((1, d)), R, c8)
    assert float(n16[0]) == 0.0
    assert np.all(codec.reconstruct(codec.dequantize_codebook(idx, n16, c8), R, np.zeros(d)) == 0)
    x = rng.standard_normal((200, d))
    idx, n16 = codec.quantize_codebook(x, R, c8)
    xh = codec.reconstruct(codec.dequantize_codebook(idx, n16, c8), R, np.zeros(d))
    rel = np.linalg.norm(xh - x, axis=1) / np.linalg.norm(x, axis=1)
    assert np.max(rel) < 0.08 and np.sqrt(np.mean(rel ** 2)) < 0.04
    # nearest centroid: no other centroid is strictly closer
    u = (x @ R) / np.linalg.norm(x, axis=1, keepdims=True)
    dist = np.abs(u[:, :, None] - c8[None, None, :])
    assert np.all(np.take_along_axis(dist, idx[:, :, None], 2)[..., 0] <= dist.min(axis=2))


def test_int8_golden():
    for case in _golden("int8_values.json")["cases"]:
        q, s = codec.int8_quantize(np.array([case["v"]]))
        assert q[0].tolist() == case["q"], case["why"]
        assert float(s[0]) == case["scale"]


def test_int8_bounds():
    rng = np.random.default_rng(13)
    v = rng.standard_normal((300, 64)) * rng.exponential(size=(300, 1))
    q, s16 = codec.int8_quantize(v)
    a = np.max(np.abs(v), axis=1)
    s = a / 127
    assert np.all(np.abs(q).max(axis=1) == 127)
    assert np.all(np.abs(v - q * s[:, None]) <= s[:, None] / 2 * (1 + 1e-12))
    assert np.array_equal(codec.int8_dequantize(q, s16), q * s16.astype(np.float64)[:, None])


# ---------------------------------------------------------------- layer invariants

def _small_layer(mode, rng, B=2, H=4, D=16):
    if mode == "int8":
        return OracleLayer("int8", B, H, D)
    if mode == "codebook":
        return OracleLayer("codebook", B, H, D, V=fit.seeded_rotation(D, 3),
                           codebook=fit.lloyd_max_gaussian(8, 1 / math.sqrt(D)))
    hpg = 2 if mode == "group" else 1
    d_in = hpg * D
    r = 8
    nb = 3
    V = np.stack([np.linalg.qr(rng.standard_normal((d_in, d_in)))[0][:, :r] for _ in range(nb)])
    mean = rng.standard_normal((nb, d_in))
    basis_of = rng.integers(0, nb, size=B * H // hpg)
    if mode == "group":
        return OracleLayer("group", B, H, D, heads_per_group=hpg, basis_of=basis_of, V=V,
                           mean=mean, bits=np.tile([4, 4, 2, 2, 2, 2, 2, 2], (nb, 1)),
                           group_size=4)
    bits = rng.choice([0, 1, 2, 3, 4, 8], size=(nb, r))
    return OracleLayer("uniform", B, H, D, basis_of=basis_of, V=V, mean=mean, bits=bits,
                       qmin=-2 * np.ones((nb, r)), qstep=0.05 * np.ones((nb, r)))


@pytest.mark.parametrize("mode", ["uniform", "group", "codebook", "int8"])
def test_streaming_equals_bulk(mode):
    # kvtc_cache page, "NOT PATH-DEPENDENT": one token at a time after
    # prefill == all at once (identical codes and reconstruction)
    rng = np.random.default_rng(14)
    a = _small_layer(mode, np.random.default_rng(15))
    b = _small_layer(mode, np.random.default_rng(15))
    x = rng.standard_normal((a.B, a.H, 12, a.D))
    a.append(x)
    b.append(x[:, :, :8])
    for t in range(8, 12):
        b.append(x[:, :, t:t + 1])
    for s in range(a.n_slots):
        assert np.array_equal(a.rows[s], b.rows[s])
        assert np.array_equal(a.side[s], b.side[s])
    assert np.array_equal(a.fetch(), b.fetch())


def test_trim_semantics():
    rng = np.random.default_rng(16)
    L = _small_layer("uniform", rng)
    x = rng.standard_normal((L.B, L.H, 10, L.D))
    L.append(x)
    full = L.fetch()
    assert L.trim(0) == 0 and L.trim(-3) == 0
    assert L.trim(4) == 4 and L.len == 6
    assert np.array_equal(L.fetch(), full[:, :, :6])
    assert L.trim(100) == 6 and L.len == 0
    L.append(x[:, :, :3])                          # basis kept after trimming to 0
    assert np.array_equal(L.fetch(), full[:, :, :3])


def test_nbytes_accounting():
    rng = np.random.default_rng(17)
    L = _small_layer("group", rng)
    L.append(rng.standard_normal((L.B, L.H, 7, L.D)))
    nb = L.nbytes()
    # 2 comps at 4 bits + 6 at 2 bits: 8 + 12 bits -> 1 + 2 bytes
    assert L.row_bytes(0) == 1 + 2
    assert nb["payload"] == L.n_slots * 7 * 3
    assert nb["side"] == L.n_slots * 7 * 2 * 3            # groups of 4: [4,4] [2,2,2,2] [2,2]
    assert nb["fp16_equiv"] == L.B * L.H * 7 * L.D * 2
    with pytest.raises(OverflowError):
        OracleLayer("int8", 1, 1, 4, capacity=2).append(np.zeros((1, 1, 3, 4)))
