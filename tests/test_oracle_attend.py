"""Pins of the decode-attention oracle (oracle/attend.py): hand-worked
values, closed forms and invariants, no GPU."""
import math

import numpy as np
import pytest

from oracle import attend as at
from oracle.layer import OracleLayer


def test_softmax_hand_worked_and_shift_invariant():
    p = at.softmax([0.0, math.log(3.0)])
    assert np.allclose(p, [0.25, 0.75], rtol=0, atol=1e-15)
    assert np.allclose(at.softmax([5.0, 5.0, 5.0, 5.0]), 0.25, atol=1e-15)
    s = np.array([0.3, -1.2, 2.0])
    assert np.allclose(at.softmax(s), at.softmax(s + 123.0), atol=1e-15)
    # huge scores do not overflow (the maximum is subtracted first)
    p = at.softmax([1000.0, 0.0])
    assert np.isfinite(p).all() and p[0] == 1.0


def test_attend_rows_hand_worked():
    """scale 1/2, scores 1/2 * (0, 2 ln 3) = (0, ln 3): weights (1/4, 3/4);
    values (4, 0) and (0, 8) give (1, 6)."""
    q = np.array([1.0, 0.0])
    K = np.array([[0.0, 5.0], [2.0 * math.log(3.0), -1.0]])
    V = np.array([[4.0, 0.0], [0.0, 8.0]])
    out = at.attend_rows(q, K, V, 0.5)
    assert np.allclose(out, [1.0, 6.0], rtol=0, atol=1e-14)


def _int8_layer(vals):
    """An int8 layer holding rows whose int8 encoding is exact (absmax 127, integers)."""
    B, H, S, D = vals.shape
    L = OracleLayer("int8", B, H, D)
    L.append(vals)
    return L


def test_one_token_returns_its_value_row():
    rng = np.random.default_rng(3)
    v = np.round(rng.uniform(-127, 127, size=(1, 2, 1, 8)))
    v[..., 0] = 127.0
    K = _int8_layer(np.round(rng.uniform(-127, 127, size=(1, 2, 1, 8))))
    Vl = _int8_layer(v)
    out = at.attend(K, Vl, rng.standard_normal((1, 2, 8)))
    assert np.array_equal(out, v[:, :, 0, :])


def test_query_heads_read_their_kv_head():
    """Hq = 2 H: query head hq reads kv head hq // 2.  Keys equal within a head
    give equal weights, so the output is that head's mean value row."""
    B, H, S, D = 2, 3, 5, 4
    rng = np.random.default_rng(4)
    kv = np.zeros((B, H, S, D))
    kv[..., 0] = 127.0                              # every key row the same
    vals = np.round(rng.uniform(-100, 100, size=(B, H, S, D)))
    vals[..., 1] = 127.0 * (1 + np.arange(H))[None, :, None] / H
    vals = np.round(vals)
    vals[..., 2] = 127.0
    K, Vl = _int8_layer(kv), _int8_layer(vals)
    q = rng.standard_normal((B, 2 * H, D))
    out = at.attend(K, Vl, q)
    dec = Vl.fetch()
    for b in range(B):
        for hq in range(2 * H):
            assert np.allclose(out[b, hq], dec[b, hq // 2].mean(axis=0), atol=1e-12)
    assert not np.allclose(out[:, 0], out[:, 2])    # different kv heads differ


def test_a_dominant_score_takes_all_the_weight():
    B, H, S, D = 1, 1, 6, 4
    keys = np.zeros((B, H, S, D))
    keys[0, 0, :, 0] = 1.0
    keys[0, 0, 3, 0] = 127.0
    vals = np.zeros((B, H, S, D))
    vals[0, 0, :, 1] = 127.0
    vals[0, 0, 3] = [127.0, 0.0, -64.0, 5.0]
    K, Vl = _int8_layer(keys), _int8_layer(vals)
    q = np.array([[[1000.0, 0.0, 0.0, 0.0]]])
    out = at.attend(K, Vl, q, scale=1.0)
    assert np.allclose(out[0, 0], Vl.fetch()[0, 0, 3], atol=1e-12)


def test_mismatched_layers_are_rejected():
    K = _int8_layer(np.ones((1, 2, 3, 4)) * 127)
    V = _int8_layer(np.ones((1, 2, 2, 4)) * 127)
    with pytest.raises(ValueError):
        at.attend(K, V, np.zeros((1, 2, 4)))
    with pytest.raises(ValueError):
        at.attend(K, K, np.zeros((1, 3, 4)))
