"""Decode attention over the stored codes (float64, CPU).

Test infrastructure only -- see ``oracle/__init__.py``.

turboquant_cache page, ``TurboQuantKVCache.attend``: unpack the stored keys,
estimate the query's inner product with every key, turn the scores into
weights with ``softmax(scores / sqrt(d))``, decode the values and return the
weighted sum of the decoded values.  palu_cache page, module docstring: the
latents are reconstructed only at attend time.  Here the keys and values are
those of two ``OracleLayer`` objects (any coded mode for the keys, any mode
for the values), decoded exactly as ``OracleLayer.fetch`` decodes them, and
one query vector per (batch, query head) attends over every stored token.
With Hq query heads over the layers' H key/value heads (Hq a multiple of H),
query head hq reads key/value head hq // (Hq / H).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["softmax", "attend_rows", "attend"]


def softmax(s):
    """exp(s - max s) / sum exp(s - max s) over the last axis (float64)."""
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def attend_rows(q, K, V, scale):
    """One query q [D] over decoded keys K [S, D] and values V [S, D]:
    softmax(scale * K q) V."""
    p = softmax(scale * (np.asarray(K, dtype=np.float64) @ np.asarray(q, dtype=np.float64)))
    return p @ np.asarray(V, dtype=np.float64)


def attend(klayer, vlayer, q, scale=None):
    """Queries q [B, Hq, D] over every stored token of the key layer ``klayer``
    and the value layer ``vlayer``; returns [B, Hq, D] float64.  ``scale``
    defaults to 1 / sqrt(D), the pages' score scale."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    H = klayer.H
    if vlayer.H != H or vlayer.B != B or klayer.B != B or Hq % H:
        raise ValueError("query heads must be a multiple of the key/value heads")
    if klayer.len != vlayer.len:
        raise ValueError("keys and values hold different lengths")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    K = klayer.fetch()          # [B, H, S, D] decoded keys
    V = vlayer.fetch()          # [B, H, S, D] decoded values
    rep = Hq // H
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for hq in range(Hq):
            h = hq // rep
            out[b, hq] = attend_rows(q[b, hq], K[b, h], V[b, h], scale)
    return out
