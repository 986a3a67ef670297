"""A cache layer with the append / fetch / trim / nbytes semantics of the C ABI.

Test infrastructure only -- see ``oracle/__init__.py``.

Slots: the layer holds B * (H / heads_per_group) slots; slot (b, g) stores the
token rows of head group g of batch entry b (one head per group outside the
PALU-style group mode).  A token row of a slot is the concatenation of the
group's heads, D_in = heads_per_group * D values.  Slot (b, g) uses basis
``basis_of[b * (H / heads_per_group) + g]``.

Parameters are the frozen fit (kvtc_cache page, "NOT PATH-DEPENDENT": basis
and allocation fit once, reused unchanged); the minimum/step of the uniform
mode are frozen as well (the plainest per-token reading of "frozen per
component min and step").  Appending T tokens one call at a time or in one
call therefore gives the same rows.
"""
from __future__ import annotations

import numpy as np

from . import codec

MODES = ("uniform", "group", "codebook", "int8")


class OracleLayer:
    def __init__(self, mode, B, H, D, *, heads_per_group=1, basis_of=None, V=None, mean=None,
                 bits=None, qmin=None, qstep=None, group_size=32, codebook=None,
                 capacity=1 << 30):
        if mode not in MODES:
            raise ValueError(mode)
        if H % heads_per_group:
            raise ValueError("heads_per_group must divide H")
        if mode != "group" and heads_per_group != 1:
            raise ValueError("head groups only in group mode")
        self.mode, self.B, self.H, self.D = mode, B, H, D
        self.hpg = heads_per_group
        self.Hg = H // heads_per_group
        self.d_in = heads_per_group * D
        self.n_slots = B * self.Hg
        self.capacity = int(capacity)
        self.group_size = group_size
        self.len = 0
        if mode == "int8":
            self.n_bases = 0
            self.basis_of = np.zeros(self.n_slots, dtype=np.int64)
        else:
            V = np.asarray(V, dtype=np.float64)
            if V.ndim == 2:
                V = V[None]
            self.V = V
            self.n_bases, _, self.r = V.shape
            self.mean = (np.zeros((self.n_bases, self.d_in)) if mean is None
                         else np.asarray(mean, dtype=np.float64).reshape(self.n_bases, self.d_in))
            if mode == "codebook":
                self.codebook = np.asarray(codebook, dtype=np.float64)
                cb_bits = int(round(np.log2(self.codebook.shape[0])))
                self.bits = np.full((self.n_bases, self.r), cb_bits, dtype=np.int64)
            else:
                self.bits = np.asarray(bits, dtype=np.int64).reshape(self.n_bases, self.r)
            if mode == "uniform":
                self.qmin = np.asarray(qmin, dtype=np.float64).reshape(self.n_bases, self.r)
                self.qstep = np.asarray(qstep, dtype=np.float64).reshape(self.n_bases, self.r)
            self.basis_of = (np.zeros(self.n_slots, dtype=np.int64) if basis_of is None
                             else np.asarray(basis_of, dtype=np.int64))
        self.rows = [np.zeros((0, self.row_bytes(s)), dtype=np.uint8) for s in range(self.n_slots)]
        self.side = [np.zeros((0,) + self._side_shape(s), dtype=np.float16)
                     for s in range(self.n_slots)]

    # ---- geometry -----------------------------------------------------------------
    def row_bytes(self, slot) -> int:
        if self.mode == "int8":
            return self.D
        return codec.row_bytes(self.bits[self.basis_of[slot]])

    def _side_shape(self, slot):
        if self.mode == "group":
            return (len(codec.group_ranges(self.bits[self.basis_of[slot]], self.group_size)),)
        if self.mode in ("codebook", "int8"):
            return ()
        return (0,)

    def slot_rows(self, x, slot):
        """Token rows [T, D_in] of slot ``slot`` from x [B, H, T, D]."""
        b, g = divmod(slot, self.Hg)
        heads = x[b, g * self.hpg:(g + 1) * self.hpg]          # [hpg, T, D]
        return np.concatenate(list(heads), axis=1) if self.hpg > 1 else heads[0]

    # ---- append ---------------------------------------------------------------------
    def encode(self, slot, X):
        """Rows [T, D_in] -> (packed rows [T, P] uint8, side data)."""
        X = np.asarray(X, dtype=np.float64)
        if self.mode == "int8":
            q, s = codec.int8_quantize(X)
            return q.view(np.uint8), s
        bsel = self.basis_of[slot]
        bits = self.bits[bsel]
        if self.mode == "uniform":
            z = codec.project(X, self.mean[bsel], self.V[bsel])
            codes = codec.quantize_uniform(z, self.qmin[bsel], self.qstep[bsel], bits)
            side = np.zeros((X.shape[0], 0), dtype=np.float16)
        elif self.mode == "group":
            z = codec.project(X, self.mean[bsel], self.V[bsel])
            codes, side = codec.quantize_group(z, bits, self.group_size)
        else:
            codes, side = codec.quantize_codebook(X, self.V[bsel], self.codebook)
        return codec.pack_rows(codes, bits), side

    def append(self, x):
        """Append T tokens of x [B, H, T, D] to every slot; returns the new length."""
        x = np.asarray(x, dtype=np.float64)
        if x.shape[:2] != (self.B, self.H) or x.shape[3] != self.D:
            raise ValueError("x must be [B, H, T, D]")
        T = x.shape[2]
        if self.len + T > self.capacity:
            raise OverflowError("capacity exceeded")
        for s in range(self.n_slots):
            rows, side = self.encode(s, self.slot_rows(x, s))
            self.rows[s] = np.concatenate([self.rows[s], rows], axis=0)
            self.side[s] = np.concatenate([self.side[s], side], axis=0)
        self.len += T
        return self.len

    # ---- fetch ----------------------------------------------------------------------
    def decode(self, slot, rows, side):
        """Packed rows (+ side data) -> reconstructed rows [T, D_in], float64."""
        if self.mode == "int8":
            return codec.int8_dequantize(np.asarray(rows, dtype=np.uint8).view(np.int8), side)
        bsel = self.basis_of[slot]
        bits = self.bits[bsel]
        codes = codec.unpack_rows(rows, bits)
        if self.mode == "uniform":
            zhat = codec.dequantize_uniform(codes, self.qmin[bsel], self.qstep[bsel], bits)
            return codec.reconstruct(zhat, self.V[bsel], self.mean[bsel])
        if self.mode == "group":
            zhat = codec.dequantize_group(codes, side, bits, self.group_size)
            return codec.reconstruct(zhat, self.V[bsel], self.mean[bsel])
        zhat = codec.dequantize_codebook(codes, side, self.codebook)
        return codec.reconstruct(zhat, self.V[bsel], np.zeros(self.d_in))

    def fetch(self):
        """Reconstructed [B, H, S, D] float64 of everything stored."""
        out = np.zeros((self.B, self.H, self.len, self.D))
        for s in range(self.n_slots):
            b, g = divmod(s, self.Hg)
            xr = self.decode(s, self.rows[s], self.side[s])
            for j in range(self.hpg):
                out[b, g * self.hpg + j] = xr[:, j * self.D:(j + 1) * self.D]
        return out

    # ---- trim / accounting --------------------------------------------------------------
    def trim(self, n: int) -> int:
        """Drop the n most recent tokens; returns the number dropped.

        kvtc_cache page, ``KVTCKVCache.trim`` (n clamped to the offset; n <= 0
        drops nothing) and palu_cache page, ``trim``.  The fitted parameters
        stay (as ``TurboQuantKVCache.reset`` keeps its quantiser).
        """
        n = min(self.len, int(n))
        if n <= 0:
            return 0
        self.len -= n
        for s in range(self.n_slots):
            self.rows[s] = self.rows[s][: self.len]
            self.side[s] = self.side[s][: self.len]
        return n

    def param_bytes(self) -> int:
        """Bytes of the frozen parameters the stored bytes carry beside the codes.

        uniform: kvtc_cache page, "Byte accounting" (the stored size carries
        the projection basis) and ``_TensorKVTC._requantize`` (a minimum and a
        scale for each surviving component, with the per-component bit
        allocation): per basis V and mean in fp32, one width byte per
        component, and an fp32 minimum and step per kept component.
        group: palu_cache page, ``projection_bytes`` (V_g and mu_g in fp32 per
        head group); the widths are the cache's configuration, not stored.
        codebook and int8: turboquant_cache page, ``memory_bytes`` counts only
        per-token bytes (the rotation and codebook follow from the seed and
        the width).
        """
        if self.mode in ("int8", "codebook"):
            return 0
        per = 4 * self.d_in * self.r + 4 * self.d_in
        if self.mode == "group":
            return self.n_bases * per
        kept = int(np.sum(self.bits > 0))
        return self.n_bases * (per + self.r) + 8 * kept

    def nbytes(self) -> dict:
        """Stored-byte accounting (kvtc_cache page "Byte accounting"; turboquant_cache
        page ``memory_bytes``; palu_cache page "Byte accounting")."""
        payload = sum(self.len * self.row_bytes(s) for s in range(self.n_slots))
        side = sum(self.len * 2 * int(np.prod(self._side_shape(s), dtype=np.int64))
                   for s in range(self.n_slots))
        return {
            "payload": int(payload),
            "side": int(side),
            "fixed": int(self.param_bytes()),
            "fp16_equiv": int(self.B * self.H * self.len * self.D * 2),
        }
