"""Pins of the order-0 Huffman accounting (oracle/entropy.py): a hand-worked
code, Kraft's equality, brute-force optimality, the entropy bounds and the
fixed-width fallback."""
import itertools
import math

import numpy as np
import pytest

from oracle import entropy as en
from oracle.layer import OracleLayer


def test_hand_worked_code():
    # merge c+d (2), then b with cd (4), then a with bcd (9): lengths 1, 2, 3, 3
    assert en.huffman_lengths([5, 2, 1, 1]) == [1, 2, 3, 3]
    assert en.component_bits([0] * 5 + [1] * 2 + [2, 3]) == 15
    assert en.huffman_lengths([0, 7, 0]) == [0, 1, 0]          # one symbol: one bit
    assert en.component_bits([2] * 9) == 9


@pytest.mark.parametrize("seed", range(10))
def test_kraft_equality_and_entropy_bounds(seed):
    rng = np.random.default_rng(seed)
    counts = rng.integers(1, 50, size=int(rng.integers(2, 12)))
    lengths = en.huffman_lengths(counts)
    assert sum(2.0 ** -l for l in lengths) == pytest.approx(1.0, abs=1e-12)
    n = counts.sum()
    p = counts / n
    H = -np.sum(p * np.log2(p))
    bits = sum(int(c) * l for c, l in zip(counts, lengths))
    assert H * n - 1e-9 <= bits < (H + 1) * n


@pytest.mark.parametrize("seed", range(6))
def test_optimal_against_every_prefix_code(seed):
    """Brute force over every length assignment that satisfies Kraft's
    inequality (a prefix code exists for each): Huffman's cost is the minimum."""
    rng = np.random.default_rng(100 + seed)
    counts = rng.integers(1, 30, size=int(rng.integers(2, 6)))
    best = math.inf
    for ls in itertools.product(range(1, len(counts) + 1), repeat=len(counts)):
        if sum(2.0 ** -l for l in ls) <= 1.0 + 1e-12:
            best = min(best, sum(int(c) * l for c, l in zip(counts, ls)))
    lengths = en.huffman_lengths(counts)
    assert sum(int(c) * l for c, l in zip(counts, lengths)) == best


def test_slot_bytes_hand_worked_and_fallback():
    # 2 components at 2 bits: a row is 1 byte
    codes = np.stack([np.zeros(8, int), np.tile([0, 1, 2, 3], 2)], axis=1)
    # payload 8 + 16 = 24 bits = 3 bytes, tables 4 + 4 -> 11 > fixed 8: fixed width
    assert en.slot_bytes(codes, [2, 2]) == (8, 11, 8)
    codes = np.stack([np.zeros(64, int), np.tile([0, 1, 2, 3], 16)], axis=1)
    # payload 64 + 128 = 192 bits = 24 bytes, + 8 = 32 < 64
    assert en.slot_bytes(codes, [2, 2]) == (64, 32, 32)
    # a dropped component costs nothing
    codes = np.stack([np.zeros(64, int), np.zeros(64, int)], axis=1)
    # (one 2-bit component: 1 byte per row; one value: 1 bit per token + a 4-byte table)
    assert en.slot_bytes(codes, [0, 2]) == (64, 8 + 4, 12)


def test_layer_gain_reads_below_one_when_the_basis_dominates():
    rng = np.random.default_rng(3)
    D, r = 16, 4
    V = np.linalg.qr(rng.standard_normal((D, D)))[0][:, :r]
    L = OracleLayer("uniform", 1, 1, D, V=V, mean=np.zeros(D), bits=[2] * r,
                    qmin=[-1.0] * r, qstep=[0.5] * r)
    L.append(rng.standard_normal((1, 1, 4, D)) * 0.01)     # few tokens: the basis dominates
    acc = en.layer_bytes(L)
    assert acc["stored_payload"] <= acc["pre_entropy"]
    assert acc["gain"] < 1.0
    assert acc["params"] == L.param_bytes()
