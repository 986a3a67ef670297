"""Pins of the TurboQuantProd residual sketch and the outlier two-stream oracle
(oracle/prod.py) against hand-worked values, closed forms, Monte Carlo
expectations and special cases that reduce to the codebook mode."""
import math

import numpy as np
import pytest

from oracle import codec, fit, prod
from oracle.layer import OracleLayer


def test_sign_bits_hand_worked():
    S = np.array([[1.0, 0.0], [0.0, -1.0], [1.0, 1.0]])
    # S r = (2, 0, 2): a zero projection stores bit 0; S r' = (0, -3, 3)
    assert prod.sign_bits([[2.0, 0.0], [0.0, 3.0]], S).tolist() == [[1, 0, 1], [0, 0, 1]]


def test_qjl_inner_one_row_closed_form():
    """m = 1 with the sketch row along r: the sign is +1 and the estimate is
    sqrt(pi/2) gamma <r, q> / ||r||, i.e. 11 sqrt(pi/2) for r = (3, 4), q = (1, 2)."""
    S = np.array([[0.6, 0.8]])
    beta = prod.sign_bits([[3.0, 4.0]], S)
    assert beta.tolist() == [[1]]
    est = prod.qjl_inner([1.0, 2.0], beta, np.array([5.0], dtype=np.float16), S)
    assert est[0] == pytest.approx(11.0 * 1.2533141373155003, rel=1e-15)


def _sketches(n, m, d, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, m, d))


def test_qjl_inner_is_unbiased():
    """E over Gaussian sketches of the residual term is <q, r> (QJL); a missing
    sqrt(pi/2), a missing 1/m or a flipped sign moves the mean by many sigma."""
    rng = np.random.default_rng(7)
    d, m, N = 16, 4, 6000
    r, q = rng.standard_normal(d), rng.standard_normal(d)
    g = np.array([np.linalg.norm(r)])
    ests = np.array([prod.qjl_inner(q, prod.sign_bits(r[None], S), g, S)[0]
                     for S in _sketches(N, m, d, 8)])
    se = ests.std() / math.sqrt(N)
    assert abs(ests.mean() - q @ r) < 5 * se
    assert abs(ests.mean() - q @ r) < 0.05 * abs(q @ r) + 5 * se


def test_qjl_decode_is_unbiased_and_matches_the_inner_product():
    rng = np.random.default_rng(9)
    d, m, N = 8, 8, 6000
    r = rng.standard_normal(d)
    g = np.array([np.linalg.norm(r)])
    dec = np.array([prod.qjl_decode(prod.sign_bits(r[None], S), g, S)[0]
                    for S in _sketches(N, m, d, 10)])
    se = dec.std(axis=0) / math.sqrt(N)
    assert np.all(np.abs(dec.mean(axis=0) - r) < 5 * se)
    S = _sketches(1, m, d, 11)[0]
    q = rng.standard_normal(d)
    beta = prod.sign_bits(r[None], S)
    assert (prod.qjl_decode(beta, g, S)[0] @ q
            == pytest.approx(prod.qjl_inner(q, beta, g, S)[0], rel=1e-12))


def test_prod_encode_hand_worked():
    """D 2, identity rotation, centroids {-1, 1}, x = (3, -4), S = [[1, 1], [1, -1]]:
    norm 5, u = (0.6, -0.8) -> indices (1, 0), x_mse = (5, -5), r = (-2, 1),
    S r = (-1, -3) -> bits (0, 0), gamma = fp16(sqrt 5) = 1145 / 512;
    x_hat = x_mse + sqrt(pi/2)/2 gamma S^T (-1, -1) = (5 - sqrt(pi/2) 1145/512, -5)."""
    S = np.array([[1.0, 1.0], [1.0, -1.0]])
    e = prod.encode_keys([[3.0, -4.0]], np.eye(2), [-1.0, 1.0], S=S)
    assert e["idx"].tolist() == [[1, 0]]
    assert float(e["norm16"][0]) == 5.0
    assert e["beta"].tolist() == [[0, 0]]
    assert float(e["gamma16"][0]) == 1145 / 512
    x = prod.decode_keys(e, np.eye(2), [-1.0, 1.0], S=S)
    assert x[0, 0] == pytest.approx(5.0 - 1.2533141373155003 * 1145 / 512, rel=1e-15)
    assert x[0, 1] == -5.0


def test_outlier_channels_hand_worked():
    K = np.array([[1.0, -5.0, 0.5, 2.0], [-1.0, 3.0, 0.5, -2.0], [1.0, -4.0, 0.5, 2.0]])
    # mean |k| = (1, 4, 0.5, 2)
    assert prod.outlier_channels(K, 2).tolist() == [1, 3]
    assert prod.outlier_channels(K, 1).tolist() == [1]
    # equal scores (2, 1, 2, 1): the lower channel first
    T = np.array([[2.0, 1.0, -2.0, 1.0]])
    assert prod.outlier_channels(T, 1).tolist() == [0]
    assert prod.outlier_channels(T, 3).tolist() == [0, 1, 2]


def test_outlier_split_starts_at_the_calibrating_key():
    """n_calib = 3: keys 0 and 1 are encoded whole with no outlier part; key 2
    (the one completing the calibration) and later keys are split: o = (-5, 2)
    is stored as s = 5/127, codes rint(o / s) = (-127, rint(50.8) = 51)."""
    R = fit.seeded_rotation(4, 3)
    cb = fit.lloyd_max_gaussian(4, 0.5)
    X = np.array([[1.0, -5.0, 0.5, 2.0], [-1.0, 3.0, 0.5, -2.0], [1.0, -5.0, 0.5, 2.0],
                  [0.3, 1.0, -0.2, 0.0]])
    ch = np.array([1, 3])
    e = prod.encode_keys(X, R, cb, channels=ch, split_from=2)
    assert e["oscale16"][:2].tolist() == [0.0, 0.0] and not e["o8"][:2].any()
    assert e["o8"][2].tolist() == [-127, 51]
    assert float(e["oscale16"][2]) == float(np.float16(5 / 127))
    whole_idx, whole_n = codec.quantize_codebook(X[:2], R, cb)
    assert np.array_equal(e["idx"][:2], whole_idx) and np.array_equal(e["norm16"][:2], whole_n)
    Xz = X[2:].copy()
    Xz[:, ch] = 0.0
    split_idx, split_n = codec.quantize_codebook(Xz, R, cb)
    assert np.array_equal(e["idx"][2:], split_idx) and np.array_equal(e["norm16"][2:], split_n)
    # the same keys appended from index 5 on are all split
    e5 = prod.encode_keys(X, R, cb, channels=ch, split_from=2, t0=5)
    assert np.all(e5["oscale16"] > 0)


def test_outlier_scores_are_masked_before_the_split():
    R = fit.seeded_rotation(4, 3)
    cb = fit.lloyd_max_gaussian(4, 0.5)
    X = np.array([[1.0, -5.0, 0.5, 2.0], [1.0, -5.0, 0.5, 2.0]])
    ch = np.array([1, 3])
    e = prod.encode_keys(X, R, cb, channels=ch, split_from=1)
    q = np.array([0.5, 1.0, -1.0, 2.0])
    s = prod.key_scores(q, e, R, cb, channels=ch)
    base = prod.key_scores(q, {"idx": e["idx"], "norm16": e["norm16"]}, R, cb)
    assert s[0] == base[0]
    sc = float(e["oscale16"][1])
    assert s[1] == pytest.approx(base[1] + sc * (-127 * 1.0 + 51 * 2.0), rel=1e-12)


def test_mse_only_layer_is_the_codebook_mode():
    """Without a sketch and without outliers the layer stores what the
    codebook mode stores (rows and norms)."""
    rng = np.random.default_rng(3)
    B, H, D, T = 1, 2, 16, 9
    R = fit.seeded_rotation(D, 5)
    cb = fit.lloyd_max_gaussian(8, 1 / math.sqrt(D))
    x = rng.standard_normal((B, H, T, D))
    pl = prod.ProdKeyLayer(B, H, D, R=R, centroids=cb)
    ol = OracleLayer("codebook", B, H, D, V=R, codebook=cb)
    pl.append(x)
    ol.append(x)
    for s in range(B * H):
        rows, side = pl.rows(s)
        assert np.array_equal(rows, ol.rows[s])
        assert np.array_equal(side[:, 0].view(np.uint16), ol.side[s].view(np.uint16))
    assert np.allclose(pl.fetch(), ol.fetch(), rtol=0, atol=0)


def test_streaming_equals_bulk_across_the_split():
    rng = np.random.default_rng(4)
    B, H, D, T, m = 1, 2, 16, 12, 24
    R = fit.seeded_rotation(D, 6)
    cb = fit.lloyd_max_gaussian(4, 1 / math.sqrt(D))
    S = rng.standard_normal((m, D))
    x = rng.standard_normal((B, H, T, D))
    ch = np.stack([prod.outlier_channels(x[0, h, :5], 3) for h in range(H)])
    bulk = prod.ProdKeyLayer(B, H, D, R=R, centroids=cb, S=S, channels=ch, split_from=4)
    step = prod.ProdKeyLayer(B, H, D, R=R, centroids=cb, S=S, channels=ch, split_from=4)
    bulk.append(x)
    for t in range(T):
        step.append(x[:, :, t:t + 1])
    for s in range(B * H):
        rb, sb = bulk.rows(s)
        rs, ss = step.rows(s)
        assert np.array_equal(rb, rs) and np.array_equal(sb.view(np.uint16), ss.view(np.uint16))
        e = bulk.unpack(s, rb, sb)
        for k, v in bulk.enc[s].items():
            assert np.array_equal(np.asarray(e[k]), np.asarray(v)), k
    assert bulk.row_bytes() == math.ceil(D * 2 / 8) + 3 + 3


def test_memory_bytes_hand_worked():
    """n 10, d 128, b_mse 2, m 128, 8 outlier channels: indices 10 * 32,
    signs 10 * 16, residual norms 10 * 2, values 10 * 130, outliers 10 * 10,
    plus this build's fp16 norms 10 * 2 = 1920 bytes."""
    assert prod.memory_bytes(10, 128, 2, 128, 8) == 1920
    assert prod.memory_bytes(0, 128, 2, 128, 8) == 0
    # the key rows of the layer account for everything but the values
    lay = prod.ProdKeyLayer(1, 1, 128, R=np.eye(128), centroids=[-1, -0.3, 0.3, 1],
                            S=np.ones((128, 128)), channels=np.zeros((1, 8), dtype=int))
    assert 10 * (lay.row_bytes() + 2 * lay.side_words()) == 1920 - 10 * 130


def test_prod_residual_term_lowers_the_inner_product_bias():
    """Averaged over sketches, <q, x_hat> of the prod encoding is an unbiased
    estimate of <q, x>, while the MSE part alone shrinks it (Lloyd-Max decodes
    toward 0)."""
    rng = np.random.default_rng(12)
    D, n, m, n_sk = 32, 300, 32, 30
    R = fit.seeded_rotation(D, 13)
    cb = fit.lloyd_max_gaussian(2, 1 / math.sqrt(D))
    X = rng.standard_normal((n, D))
    q = rng.standard_normal(D)
    true = X @ q
    slopes = []
    for S in _sketches(n_sk, m, D, 14):
        e = prod.encode_keys(X, R, cb, S=S)
        full = prod.key_scores(q, e, R, cb, S=S)
        slopes.append((full @ true) / (true @ true))
    e = prod.encode_keys(X, R, cb)
    slope_mse = (prod.key_scores(q, e, R, cb) @ true) / (true @ true)
    slopes = np.array(slopes)
    assert abs(slopes.mean() - 1.0) < 5 * slopes.std() / math.sqrt(n_sk) + 0.01
    assert slope_mse < 0.85


def test_attend_scores_equal_the_decoded_keys():
    """The score estimate (P2 plus the outlier term) is the inner product with
    the reconstruction (P3 plus the outlier decode), so attention through the
    estimator equals softmax attention over the decoded keys."""
    from oracle.attend import attend_rows

    rng = np.random.default_rng(21)
    B, H, D, T, m, Hq = 2, 2, 16, 10, 16, 4
    R = fit.seeded_rotation(D, 22)
    cb = fit.lloyd_max_gaussian(4, 1 / math.sqrt(D))
    S = rng.standard_normal((m, D))
    x = rng.standard_normal((B, H, T, D))
    ch = np.stack([prod.outlier_channels(x[b, h, :4], 2) for b in range(B) for h in range(H)])
    kl = prod.ProdKeyLayer(B, H, D, R=R, centroids=cb, S=S, channels=ch, split_from=3)
    kl.append(x)
    vl = OracleLayer("int8", B, H, D)
    vl.append(rng.standard_normal((B, H, T, D)))
    q = rng.standard_normal((B, Hq, D))
    out = prod.attend(kl, vl, q)
    K, V = kl.fetch(), vl.fetch()
    for b in range(B):
        for hq in range(Hq):
            h = hq // (Hq // H)
            assert np.allclose(kl.scores(b * H + h, q[b, hq]), K[b, h] @ q[b, hq], rtol=1e-12,
                               atol=1e-12)
            ref = attend_rows(q[b, hq], K[b, h], V[b, h], 1 / math.sqrt(D))
            assert np.allclose(out[b, hq], ref, rtol=1e-12, atol=1e-12)


def test_trim_then_append_equals_appending_the_kept_keys():
    rng = np.random.default_rng(31)
    B, H, D, m = 1, 1, 16, 16
    R = fit.seeded_rotation(D, 32)
    cb = fit.lloyd_max_gaussian(4, 1 / math.sqrt(D))
    S = rng.standard_normal((m, D))
    x = rng.standard_normal((B, H, 12, D))
    ch = np.array([prod.outlier_channels(x[0, 0, :4], 2)])
    a = prod.ProdKeyLayer(B, H, D, R=R, centroids=cb, S=S, channels=ch, split_from=3)
    b = prod.ProdKeyLayer(B, H, D, R=R, centroids=cb, S=S, channels=ch, split_from=3)
    a.append(x)
    assert a.trim(5) == 5 and a.len == 7 and a.trim(-1) == 0
    a.append(x[:, :, 7:])
    b.append(x)
    ra, sa = a.rows(0)
    rb, sb = b.rows(0)
    assert np.array_equal(ra, rb) and np.array_equal(sa.view(np.uint16), sb.view(np.uint16))
    assert a.trim(100) == 12 and a.len == 0
