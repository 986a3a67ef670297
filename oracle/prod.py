"""TurboQuantProd residual sketch and the outlier two-stream key store (float64, CPU).

Test infrastructure only -- see ``oracle/__init__.py``.

turboquant_cache page:
* module and class docstrings: keys are stored bit-packed, codebook indices at
  ``b_mse`` bits per coordinate and QJL sign bits at one bit each; an optional
  set of calibrated outlier channels is kept at higher precision beside the
  quantised inlier stream;
* ``TurboQuantKVCache.__init__``: with the prod quantiser ``b_mse = max(b - 1, 1)``;
  ``m`` sketch dimensions (``jl_dim``), ``ceil(m / 8)`` sign bytes per key; an
  fp16 residual norm per key; the outlier detector takes ``n_outliers``
  channels after ``n_calib`` keys; an int8 outlier row and an fp16 scale per key;
* ``append_key``: the detector observes the key, the key that completes the
  calibration and every later one is split, its outlier channels quantised as
  ``append_value`` quantises a value row and zeroed before the key quantiser
  sees it; a sign is stored as bit 1 when positive; the residual norm as fp16;
* ``_unpack_signs_block``: bit b -> 2 b - 1;
* ``attend``: ``estimate_inner_product`` plus the outlier inner product
  ``sum_c q_c o8_c s`` masked by ``s > 0``, then ``softmax(scores / sqrt(d))``
  and the weighted sum of the decoded values;
* ``memory_bytes``: index, sign, residual-norm, value and outlier bytes.

The pages print neither ``TurboQuantProd`` nor ``OutlierDetector``.  Readings:

P1 encode: the MSE stage is ``codec.quantize_codebook`` at ``b_mse`` bits
   (rotation R, fp16 norm n); its decode is x_mse = fp16(n) R c[idx]; the
   residual is r = x - x_mse; sign bit j is [(S r)_j > 0] (a zero projection
   gives bit 0, i.e. -1), S the m x d sketch whose seeded N(0, 1) entries are
   an input; the residual norm gamma = ||r||_2 is stored as fp16.  This is the
   published TurboQuant_prod (Zandieh et al., 2025): the MSE quantiser at one
   bit less plus the one-bit QJL transform of its residual (Zandieh et al.,
   2024).
P2 inner product: <q, x_mse> + sqrt(pi/2) / m * fp16(gamma) * <S q, 2 beta - 1>,
   QJL's unbiased estimator of <q, r> added to the MSE part.
P3 reconstruction (what fetch returns): x_mse + sqrt(pi/2) / m * fp16(gamma)
   * S^T (2 beta - 1), QJL's dequantiser; <q, x_hat> equals P2.
P4 outlier channels: the n_outliers channels of largest mean |k_c| over the
   first n_calib keys (the lower channel first among equals), listed in
   ascending channel order.
P5 outlier stream: keys with index >= n_calib - 1 are split: o = k[channels]
   is stored as ``codec.int8_quantize`` stores a value row, and the inlier
   stream encodes k with those channels set to 0.  Earlier keys are encoded
   whole and carry outlier codes 0 with scale 0.
P6 the stored row of a key is [indices (b_mse bits each, LSB-first) | sign
   bits (LSB-first, ceil(m / 8) bytes) | outlier int8 codes], its side words
   [fp16 norm, fp16 residual norm (prod only), fp16 outlier scale (outliers
   only)].
"""
from __future__ import annotations

import math

import numpy as np

from . import codec

__all__ = ["QJL_COEF", "sign_bits", "qjl_decode", "qjl_inner", "outlier_channels",
           "encode_keys", "decode_keys", "key_scores", "ProdKeyLayer", "memory_bytes", "attend"]

# sqrt(pi / 2): E[sign(<s, r>) <s, q>] = sqrt(2 / pi) <q, r> / ||r|| for s ~ N(0, I).
QJL_COEF = math.sqrt(math.pi / 2.0)


def sign_bits(r, S) -> np.ndarray:
    """beta [n, m] uint8: 1 where (S r_t)_j > 0, else 0 (P1)."""
    proj = np.asarray(r, dtype=np.float64) @ np.asarray(S, dtype=np.float64).T
    return (proj > 0).astype(np.uint8)


def qjl_decode(beta, gamma16, S) -> np.ndarray:
    """sqrt(pi/2) / m * gamma * S^T (2 beta - 1), per row (P3)."""
    S = np.asarray(S, dtype=np.float64)
    m = S.shape[0]
    pm = 2.0 * np.asarray(beta, dtype=np.float64) - 1.0
    g = np.asarray(gamma16, dtype=np.float64)
    return (QJL_COEF / m) * g[:, None] * (pm @ S)


def qjl_inner(q, beta, gamma16, S) -> np.ndarray:
    """sqrt(pi/2) / m * gamma * <S q, 2 beta - 1>, per row (P2's residual term)."""
    S = np.asarray(S, dtype=np.float64)
    m = S.shape[0]
    sq = S @ np.asarray(q, dtype=np.float64)
    pm = 2.0 * np.asarray(beta, dtype=np.float64) - 1.0
    return (QJL_COEF / m) * np.asarray(gamma16, dtype=np.float64) * (pm @ sq)


def outlier_channels(K_calib, n_out: int) -> np.ndarray:
    """P4: the n_out channels of largest mean |k| over the calibration keys, ascending."""
    K = np.asarray(K_calib, dtype=np.float64)
    score = np.mean(np.abs(K), axis=0)
    order = np.argsort(-score, kind="stable")   # larger first; equal scores by index
    return np.sort(order[:n_out]).astype(np.int64)


def encode_keys(X, R, centroids, *, S=None, channels=None, split_from=0, t0=0):
    """Encode keys X [n, d] with global indices t0 .. t0 + n - 1 (P1, P5).

    Returns a dict: idx [n, d], norm16 [n], beta [n, m] (prod), gamma16 [n]
    (prod), o8 [n, n_out] and oscale16 [n] (outliers).
    """
    X = np.array(X, dtype=np.float64)
    n, d = X.shape
    out = {}
    if channels is not None and len(channels):
        ch = np.asarray(channels, dtype=np.int64)
        split = (t0 + np.arange(n)) >= split_from
        o8 = np.zeros((n, len(ch)), dtype=np.int8)
        os16 = np.zeros(n, dtype=np.float16)
        if split.any():
            q, s = codec.int8_quantize(X[split][:, ch])
            o8[split], os16[split] = q, s
            Xs = X[split]
            Xs[:, ch] = 0.0
            X[split] = Xs
        out["o8"], out["oscale16"] = o8, os16
    idx, norm16 = codec.quantize_codebook(X, R, centroids)
    out["idx"], out["norm16"] = idx, norm16
    if S is not None:
        x_mse = codec.reconstruct(codec.dequantize_codebook(idx, norm16, centroids), R,
                                  np.zeros(d))
        r = X - x_mse
        out["beta"] = sign_bits(r, S)
        out["gamma16"] = np.sqrt(np.sum(r * r, axis=1)).astype(np.float16)
    return out


def decode_keys(enc, R, centroids, *, S=None, channels=None) -> np.ndarray:
    """Reconstructed keys [n, d] (P3, plus the outlier channels' int8 decode)."""
    x = codec.reconstruct(codec.dequantize_codebook(enc["idx"], enc["norm16"], centroids), R,
                          np.zeros(np.asarray(R).shape[0]))
    if S is not None:
        x = x + qjl_decode(enc["beta"], enc["gamma16"], S)
    if channels is not None and len(channels):
        x[:, np.asarray(channels)] += codec.int8_dequantize(enc["o8"], enc["oscale16"])
    return x


def key_scores(q, enc, R, centroids, *, S=None, channels=None) -> np.ndarray:
    """Raw scores [n] of query q against the stored keys (P2 plus the outlier term)."""
    q = np.asarray(q, dtype=np.float64)
    x_mse = codec.reconstruct(codec.dequantize_codebook(enc["idx"], enc["norm16"], centroids), R,
                              np.zeros(q.shape[0]))
    s = x_mse @ q
    if S is not None:
        s = s + qjl_inner(q, enc["beta"], enc["gamma16"], S)
    if channels is not None and len(channels):
        ch = np.asarray(channels)
        sc = np.asarray(enc["oscale16"], dtype=np.float64)
        s = s + (enc["o8"].astype(np.float64) @ q[ch]) * sc * (sc > 0)
    return s


def memory_bytes(n, d, b_mse, m, n_out, values=True) -> int:
    """turboquant_cache page ``memory_bytes`` for n stored tokens (outlier bytes
    counted when the outlier stream is on), plus the fp16 norm per key this
    build stores (the codebook mode's norm reading)."""
    if n == 0:
        return 0
    b = n * math.ceil(d * b_mse / 8)
    if m:
        b += n * math.ceil(m / 8) + 2 * n
    if values:
        b += n * (d + 2)
    if n_out:
        b += n * (n_out + 2)
    return b + 2 * n


class ProdKeyLayer:
    """Key layer of the TurboQuant cache with the residual sketch and/or the
    outlier stream, one slot per (b, h), rows laid out as P6.

    R [d, d] and centroids (2^b_mse levels) as the codebook mode takes them; S
    [m, d] or None; channels [n_slots, n_out] or None; split_from = n_calib - 1.
    """

    def __init__(self, B, H, D, *, R, centroids, S=None, channels=None, split_from=0):
        self.B, self.H, self.D = B, H, D
        self.n_slots = B * H
        self.R = np.asarray(R, dtype=np.float64)
        self.centroids = np.asarray(centroids, dtype=np.float64)
        self.b_mse = int(round(math.log2(self.centroids.shape[0])))
        self.S = None if S is None else np.asarray(S, dtype=np.float64)
        self.m = 0 if S is None else self.S.shape[0]
        self.channels = None if channels is None else np.asarray(channels, dtype=np.int64)
        self.n_out = 0 if channels is None else self.channels.shape[1]
        self.split_from = int(split_from)
        self.len = 0
        self.enc = [None] * self.n_slots

    def _slot_kw(self, s):
        return dict(S=self.S, channels=None if self.channels is None else self.channels[s])

    def row_bytes(self) -> int:
        return math.ceil(self.D * self.b_mse / 8) + math.ceil(self.m / 8) + self.n_out

    def side_words(self) -> int:
        return 1 + (1 if self.m else 0) + (1 if self.n_out else 0)

    def append(self, x):
        """Append T keys of x [B, H, T, D] to every slot."""
        x = np.asarray(x, dtype=np.float64)
        for s in range(self.n_slots):
            b, h = divmod(s, self.H)
            e = encode_keys(x[b, h], self.R, self.centroids, split_from=self.split_from,
                            t0=self.len, **self._slot_kw(s))
            if self.enc[s] is None:
                self.enc[s] = e
            else:
                self.enc[s] = {k: np.concatenate([self.enc[s][k], e[k]], axis=0) for k in e}
        self.len += x.shape[2]
        return self.len

    def trim(self, n: int) -> int:
        """Drop the n most recent keys (clamped to the length); the sketch,
        channels and split point stay, as ``OracleLayer.trim`` keeps its fit."""
        n = min(self.len, int(n))
        if n <= 0:
            return 0
        self.len -= n
        self.enc = [None if e is None or self.len == 0 else {k: v[: self.len] for k, v in e.items()}
                    for e in self.enc]
        return n

    def rows(self, s):
        """Packed rows [len, row_bytes] uint8 and side words [len, k] fp16 of slot s (P6)."""
        e = self.enc[s]
        parts = [codec.pack_rows(e["idx"], np.full(self.D, self.b_mse))]
        side = [e["norm16"]]
        if self.m:
            parts.append(codec.pack_rows(e["beta"].astype(np.int64), np.ones(self.m, dtype=np.int64)))
            side.append(e["gamma16"])
        if self.n_out:
            parts.append(e["o8"].view(np.uint8))
            side.append(e["oscale16"])
        return np.concatenate(parts, axis=1), np.stack(side, axis=1)

    def unpack(self, s, rows, side):
        """The inverse of rows(): the encoding dict of one slot from its bytes."""
        rows = np.asarray(rows, dtype=np.uint8)
        side = np.asarray(side, dtype=np.float16)
        pc = math.ceil(self.D * self.b_mse / 8)
        e = {"idx": codec.unpack_rows(rows[:, :pc], np.full(self.D, self.b_mse)),
             "norm16": side[:, 0]}
        off, w = pc, 1
        if self.m:
            nb = math.ceil(self.m / 8)
            e["beta"] = codec.unpack_rows(rows[:, off:off + nb], np.ones(self.m, dtype=np.int64))
            e["gamma16"] = side[:, w]
            off, w = off + nb, w + 1
        if self.n_out:
            e["o8"] = rows[:, off:off + self.n_out].view(np.int8)
            e["oscale16"] = side[:, w]
        return e

    def decode(self, s, enc=None):
        return decode_keys(self.enc[s] if enc is None else enc, self.R, self.centroids,
                           **self._slot_kw(s))

    def scores(self, s, q, enc=None):
        return key_scores(q, self.enc[s] if enc is None else enc, self.R, self.centroids,
                          **self._slot_kw(s))

    def fetch(self):
        out = np.zeros((self.B, self.H, self.len, self.D))
        for s in range(self.n_slots):
            b, h = divmod(s, self.H)
            out[b, h] = self.decode(s)
        return out


def attend(klayer: "ProdKeyLayer", vlayer, q, scale=None):
    """turboquant_cache page ``attend`` with these keys: per (batch, query head)
    the raw scores of P2 plus the outlier term, softmax(scale * scores) (scale
    1 / sqrt(D) by default) and the weighted sum of the value layer's decoded
    rows; query head hq reads key/value head hq // (Hq / H)."""
    from .attend import softmax

    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    H = klayer.H
    if Hq % H or klayer.len != vlayer.len:
        raise ValueError("query heads must be a multiple of the key/value heads")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    V = vlayer.fetch()
    rep = Hq // H
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for hq in range(Hq):
            s = b * H + hq // rep
            p = softmax(scale * klayer.scores(s, q[b, hq]))
            out[b, hq] = p @ V[b, hq // rep]
    return out
