"""Per-token append and fetch arithmetic, float64 (CPU).

Test infrastructure only -- see ``oracle/__init__.py``.

Append: project, quantise, bit-pack.  Fetch: unpack, dequantise,
reconstruct.  All rounding is NumPy's ``rint`` (round half to even, the
semantics of the pages' ``round``).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "segments",
    "row_bytes",
    "pack_rows",
    "unpack_rows",
    "project",
    "quantize_uniform",
    "dequantize_uniform",
    "group_ranges",
    "quantize_group",
    "dequantize_group",
    "quantize_codebook",
    "dequantize_codebook",
    "reconstruct",
    "int8_quantize",
    "int8_dequantize",
    "INT8_MAX",
]

# turboquant_cache page: INT8_MAX, used symmetrically (clip to [-127, 127]).
INT8_MAX = 127


# --------------------------------------------------------------------------
# Bit packing
# --------------------------------------------------------------------------

def segments(bits):
    """The packed row's segments: [(width, components), ...].

    One segment per distinct non-zero width, widest first; inside a segment
    the components keep ascending index order.  0-bit components are not
    stored at all (kvtc_cache page, ``_TensorKVTC._requantize``: only
    ``survived_idx`` components are quantised and encoded).
    """
    bits = np.asarray(bits)
    out = []
    for w in sorted(set(int(b) for b in bits if b > 0), reverse=True):
        out.append((w, np.nonzero(bits == w)[0]))
    return out


def row_bytes(bits) -> int:
    """Packed bytes per token: sum over segments of ceil(r_b * b / 8).

    turboquant_cache page, ``TurboQuantKVCache.__init__``
    (``_idx_packed_len = ceil(d * b_mse / 8)``) and ``memory_bytes``, applied
    per segment.
    """
    return int(sum((len(c) * w + 7) // 8 for w, c in segments(bits)))


def pack_rows(codes, bits) -> np.ndarray:
    """Pack codes [n, r] into rows [n, P] of bytes.

    turboquant_cache page, ``BitPackBuffer`` as read back by
    ``_unpack_indices_block``: little-endian bit order (``unpackbits(...,
    bitorder="little")`` for 1 bit, shifts 0, 2, 4, 6 for 2 bits, 0 and 4 for
    4 bits), which is the LSB-first bit stream: code m of a segment occupies
    stream bits [m*b, m*b + b), code bit 0 lowest, stream bit i in byte
    i // 8 at position i % 8.  A 3-bit code may straddle two bytes.  Pad
    bits are zero.  Segments follow each other byte-aligned.
    """
    codes = np.asarray(codes, dtype=np.int64)
    n = codes.shape[0]
    parts = []
    for w, comps in segments(bits):
        sub = codes[:, comps]
        if np.any(sub < 0) or np.any(sub >= (1 << w)):
            raise ValueError("code out of range for its width")
        # stream bit (m * w + j) = bit j of code m
        bitmat = ((sub[:, :, None] >> np.arange(w)[None, None, :]) & 1).astype(np.uint8)
        parts.append(np.packbits(bitmat.reshape(n, -1), axis=1, bitorder="little"))
    if not parts:
        return np.zeros((n, 0), dtype=np.uint8)
    return np.concatenate(parts, axis=1)


def unpack_rows(rows, bits) -> np.ndarray:
    """Inverse of ``pack_rows``: rows [n, P] -> codes [n, r] (0 for dropped)."""
    rows = np.asarray(rows, dtype=np.uint8)
    bits = np.asarray(bits)
    n = rows.shape[0]
    codes = np.zeros((n, bits.shape[0]), dtype=np.int64)
    off = 0
    for w, comps in segments(bits):
        nb = (len(comps) * w + 7) // 8
        stream = np.unpackbits(rows[:, off:off + nb], axis=1, bitorder="little")
        stream = stream[:, : len(comps) * w].reshape(n, len(comps), w).astype(np.int64)
        codes[:, comps] = np.sum(stream << np.arange(w)[None, None, :], axis=2)
        off += nb
    return codes


# --------------------------------------------------------------------------
# Projection and reconstruction
# --------------------------------------------------------------------------

def project(x, mean, V):
    """z = (x - mean) @ V.

    kvtc_cache page, module docstring "Design", decode step 1 (project into
    the already-fitted basis) and ``_TensorKVTC._requantize``
    (``x_centered = raw - mean``; ``L = x_centered @ V``).
    """
    return (np.asarray(x, dtype=np.float64) - np.asarray(mean, dtype=np.float64)) @ np.asarray(
        V, dtype=np.float64)


def reconstruct(zhat, V, mean):
    """x_hat = zhat @ V^T + mean (kvtc_cache page, module docstring: every call
    returns reconstructed ``[B, H, S_total, D]`` for SDPA; palu_cache page,
    "Design": latent -> dequant -> reconstruct)."""
    return np.asarray(zhat, dtype=np.float64) @ np.asarray(V, dtype=np.float64).T + np.asarray(
        mean, dtype=np.float64)


# --------------------------------------------------------------------------
# Uniform (KVTC-style) quantiser with frozen min / step
# --------------------------------------------------------------------------

def quantize_uniform(z, lo, step, bits) -> np.ndarray:
    """code_k = clip(rint((z_k - lo_k) / step_k), 0, 2^b_k - 1); 0-bit -> 0 (not stored).

    kvtc_cache page, ``_TensorKVTC._requantize`` (``quantize_component`` per
    surviving component at its allocated width), with the minimum and step
    frozen at fit time.
    """
    z = np.asarray(z, dtype=np.float64)
    bits = np.asarray(bits)
    codes = np.zeros(z.shape, dtype=np.int64)
    for k, b in enumerate(bits):
        if b == 0:
            continue
        u = (z[:, k] - float(lo[k])) / float(step[k])
        codes[:, k] = np.clip(np.rint(u), 0, (1 << int(b)) - 1).astype(np.int64)
    return codes


def dequantize_uniform(codes, lo, step, bits) -> np.ndarray:
    """zhat_k = lo_k + code_k * step_k; a dropped component contributes 0."""
    codes = np.asarray(codes, dtype=np.float64)
    bits = np.asarray(bits)
    lo = np.asarray(lo, dtype=np.float64)
    step = np.asarray(step, dtype=np.float64)
    zhat = lo[None, :] + codes * step[None, :]
    zhat[:, bits == 0] = 0.0
    return zhat


# --------------------------------------------------------------------------
# Group-scale (PALU-style) mixed-bit quantiser
# --------------------------------------------------------------------------

def group_ranges(bits, group_size: int):
    """Scale groups: [(width, components), ...] in segment order.

    palu_cache page, ``palu_group_size`` (default 32): each segment's
    components, in order, are cut into runs of ``group_size`` (the last run
    of a segment may be shorter), so a group never mixes widths.
    """
    out = []
    for w, comps in segments(bits):
        for s in range(0, len(comps), group_size):
            out.append((w, comps[s:s + group_size]))
    return out


def quantize_group(z, bits, group_size: int):
    """Per token and group g of width b: s = max(absmax_g / qmax_b, 1e-8) with
    qmax_b = 2^(b-1) - 1; q = clip(rint(z / s), -qmax, qmax); the stored code
    is q + 2^(b-1) and the stored scale is fp16(s).

    palu_cache page ("Design", mixed-bit quantisation of the latents,
    ``palu_group_size``), with the symmetric per-token absmax convention of
    the turboquant_cache page's ``append_value`` (scale floor 1e-8; codes
    taken with the unrounded scale, the scale then stored as fp16).
    Returns (codes [n, r], scales fp16 [n, n_groups]).
    """
    z = np.asarray(z, dtype=np.float64)
    n = z.shape[0]
    groups = group_ranges(bits, group_size)
    codes = np.zeros(z.shape, dtype=np.int64)
    scales = np.zeros((n, len(groups)), dtype=np.float16)
    for g, (w, comps) in enumerate(groups):
        if w < 2:
            raise ValueError("group mode needs widths >= 2")
        qmax = (1 << (w - 1)) - 1
        sub = z[:, comps]
        s = np.maximum(np.max(np.abs(sub), axis=1) / qmax, 1e-8)
        q = np.clip(np.rint(sub / s[:, None]), -qmax, qmax)
        codes[:, comps] = q.astype(np.int64) + (1 << (w - 1))
        scales[:, g] = s.astype(np.float16)
    return codes, scales


def dequantize_group(codes, scales16, bits, group_size: int) -> np.ndarray:
    """zhat = (code - 2^(b-1)) * fp16 scale of the component's group."""
    codes = np.asarray(codes, dtype=np.int64)
    zhat = np.zeros(codes.shape, dtype=np.float64)
    for g, (w, comps) in enumerate(group_ranges(bits, group_size)):
        s = np.asarray(scales16[:, g], dtype=np.float64)
        zhat[:, comps] = (codes[:, comps] - (1 << (w - 1))).astype(np.float64) * s[:, None]
    return zhat


# --------------------------------------------------------------------------
# Rotation + scalar codebook (TurboQuant-MSE-style)
# --------------------------------------------------------------------------

def quantize_codebook(x, R, centroids):
    """n = ||x||_2; u = (x @ R) / n; idx_k = argmin_j |u_k - c_j| (first on ties).

    turboquant_cache page, ``append_key`` (``key_quantizer.encode`` -> codebook
    indices, packed at ``b_mse`` bits) for ``TurboQuantMSE``; the per-token
    norm is stored as fp16 (as the page stores its per-token fp16 norms).
    A zero vector gives u = 0.  Returns (idx [n, d], norm fp16 [n]).
    """
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(centroids, dtype=np.float64)
    nrm = np.sqrt(np.sum(x * x, axis=1))
    z = x @ np.asarray(R, dtype=np.float64)
    u = np.zeros_like(z)
    nz = nrm > 0
    u[nz] = z[nz] / nrm[nz, None]
    idx = np.argmin(np.abs(u[:, :, None] - c[None, None, :]), axis=2)
    return idx.astype(np.int64), nrm.astype(np.float16)


def dequantize_codebook(idx, norm16, centroids) -> np.ndarray:
    """zhat_k = fp16(n) * c[idx_k]."""
    c = np.asarray(centroids, dtype=np.float64)
    return np.asarray(norm16, dtype=np.float64)[:, None] * c[np.asarray(idx)]


# --------------------------------------------------------------------------
# Per-token int8 values
# --------------------------------------------------------------------------

def int8_quantize(v):
    """s = max(absmax / 127, 1e-8); q = clip(rint(v / s), -127, 127); store fp16(s).

    turboquant_cache page, ``TurboQuantKVCache.append_value``.
    Returns (q int8 [n, d], s fp16 [n]).
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.max(np.abs(v), axis=1)
    s = np.maximum(a / INT8_MAX, 1e-8)
    q = np.clip(np.rint(v / s[:, None]), -INT8_MAX, INT8_MAX).astype(np.int8)
    return q, s.astype(np.float16)


def int8_dequantize(q, s16) -> np.ndarray:
    """v_hat = q * fp16(s) (turboquant_cache page, ``attend``: value decode)."""
    return np.asarray(q, dtype=np.float64) * np.asarray(s16, dtype=np.float64)[:, None]
