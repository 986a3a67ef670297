"""Workloads and comparisons shared by the GPU parity tests.

Inputs come from ``synth`` (seeded), the frozen parameters from the float64
oracle's fit rounded to fp32; the GPU and the oracle consume the same fp32
numbers.  The GPU's packed rows are compared with the oracle's byte for
byte; the GPU's reconstruction is compared with the oracle's float64
reconstruction of the GPU's own codes.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import synth
from oracle import codec, fit
from oracle.layer import OracleLayer

# Tolerances of the reconstruction (per head): max-abs and RMS relative to x_hat.
MAX_ABS_REL = 4e-3
RMS_REL = 1e-3
# Codes may differ from the oracle only at ties this close to a boundary,
# at a rate of at most this many per code.
TIE_WINDOW = 1e-6
MISMATCH_RATE = 1e-6


# ---------------------------------------------------------------------------- fits

def fit_uniform(x64, fit_len, r, choices, budget):
    """Per-(b, h) local PCA + DP allocation + frozen min/step (fp32)."""
    B, H = x64.shape[:2]
    Vs, ms, bs, los, sts = [], [], [], [], []
    for b in range(B):
        for h in range(H):
            X = x64[b, h, :fit_len]
            mean, lam, U = fit.pca_fit(X)
            V32 = U[:, :r].astype(np.float32)
            m32 = mean.astype(np.float32)
            bits = fit.dp_allocate(lam[:r], choices, budget)
            lo, st = fit.uniform_params(codec.project(X, m32, V32), bits)
            Vs.append(V32), ms.append(m32), bs.append(bits)
            los.append(lo.astype(np.float32)), sts.append(st.astype(np.float32))
    return dict(V=np.stack(Vs), mean=np.stack(ms), bits=np.stack(bs).astype(np.uint8),
                qmin=np.stack(los), qstep=np.stack(sts), basis_of=np.arange(B * H))


def group_rows(x64, hpg, g):
    """Rows [B*S, hpg*D] of head group g, pooled over the batch."""
    B, H, S, D = x64.shape
    return np.concatenate([np.concatenate(list(x64[b, g * hpg:(g + 1) * hpg]), axis=1)
                           for b in range(B)], axis=0)


def fit_group(x64, hpg, r, hi=4, lo=2, frac=0.25):
    B, H = x64.shape[:2]
    Hg = H // hpg
    Vs, ms = [], []
    for g in range(Hg):
        mean, lam, U = fit.pca_fit(group_rows(x64, hpg, g))
        Vs.append(U[:, :r].astype(np.float32)), ms.append(mean.astype(np.float32))
    bits = np.tile(fit.palu_bits(r, hi, lo, frac), (Hg, 1)).astype(np.uint8)
    basis_of = np.array([g for b in range(B) for g in range(Hg)])
    return dict(V=np.stack(Vs), mean=np.stack(ms), bits=bits, basis_of=basis_of,
                heads_per_group=hpg, group_size=32)


def fit_codebook(D, bits=3, seed=1234):
    return dict(V=fit.seeded_rotation(D, seed).astype(np.float32),
                codebook=fit.lloyd_max_gaussian(1 << bits, 1 / math.sqrt(D)).astype(np.float32))


def oracle_kwargs(params):
    kw = dict(params)
    for k in ("qmin", "qstep", "V", "mean", "codebook"):
        if k in kw and kw[k] is not None:
            kw[k] = np.asarray(kw[k], dtype=np.float64)
    return kw


# ---------------------------------------------------------------------------- comparisons

def _u_values(rl: OracleLayer, slot: int, X: np.ndarray):
    """Oracle's pre-rounding quantities [T, r] (distance to boundaries is taken on these)."""
    bsel = rl.basis_of[slot]
    if rl.mode == "uniform":
        z = codec.project(X, rl.mean[bsel], rl.V[bsel])
        return (z - rl.qmin[bsel]) / np.where(rl.qstep[bsel] > 0, rl.qstep[bsel], 1.0)
    if rl.mode == "group":
        z = codec.project(X, rl.mean[bsel], rl.V[bsel])
        u = np.zeros_like(z)
        for w, comps in codec.group_ranges(rl.bits[bsel], rl.group_size):
            qmax = (1 << (w - 1)) - 1
            s = np.maximum(np.max(np.abs(z[:, comps]), axis=1) / qmax, 1e-8)
            u[:, comps] = z[:, comps] / s[:, None]
        return u
    nrm = np.sqrt(np.sum(X * X, axis=1))
    z = X @ rl.V[bsel]
    return np.where(nrm[:, None] > 0, z / np.where(nrm > 0, nrm, 1)[:, None], 0.0)


def _boundary_distance(rl: OracleLayer, u):
    if rl.mode == "codebook":
        c = rl.codebook
        mids = 0.5 * (c[:-1] + c[1:])
        return np.min(np.abs(u[..., None] - mids), axis=-1)
    if rl.mode == "group":
        au = np.abs(u)
        return np.abs(au - np.floor(au) - 0.5)
    return np.abs(u - np.floor(u) - 0.5)


def compare_codes(gpu_rows, gpu_side, rl: OracleLayer, slot: int, X: np.ndarray,
                  t_index=None):
    """Compare one slot's GPU rows with the oracle's encoding of X (rows [T, D_in]).

    Returns (n_codes, n_mismatch); asserts every mismatch is an oracle near-tie.
    """
    ref_rows, ref_side = rl.encode(slot, X)
    gpu_rows = np.asarray(gpu_rows)
    if rl.mode == "int8":
        q_g = gpu_rows.view(np.int8).astype(np.int64)
        q_r = ref_rows.view(np.int8).astype(np.int64)
        s_g = np.asarray(gpu_side).view(np.float16)[:, 0]
        assert np.array_equal(s_g.view(np.uint16), ref_side.view(np.uint16)), "int8 scales differ"
        bad = q_g != q_r
        assert not bad.any(), f"int8 codes differ at {np.argwhere(bad)[:5]}"
        return q_g.size, 0
    bits = rl.bits[rl.basis_of[slot]]
    n_codes = int(np.sum(bits > 0)) * X.shape[0]
    mism = 0
    if not np.array_equal(gpu_rows, ref_rows):
        cg = codec.unpack_rows(gpu_rows, bits)
        cr = codec.unpack_rows(ref_rows, bits)
        diff = np.argwhere(cg != cr)
        u = _u_values(rl, slot, X)
        dist = _boundary_distance(rl, u)
        for t, k in diff:
            assert dist[t, k] <= TIE_WINDOW, (
                f"slot {slot} token {t} comp {k}: gpu {cg[t, k]} oracle {cr[t, k]}, "
                f"oracle distance to boundary {dist[t, k]:.3e}")
        mism = len(diff)
    if gpu_side is not None and ref_side.size:
        sg = np.asarray(gpu_side).view(np.float16).reshape(ref_side.shape)
        if not np.array_equal(sg.view(np.uint16), ref_side.view(np.uint16)):
            bad = np.argwhere(sg.view(np.uint16) != ref_side.view(np.uint16))
            raise AssertionError(f"slot {slot}: side words differ at {bad[:5].tolist()}")
    return n_codes, mism


def check_fetch(out_gpu, gpu_layer, rl: OracleLayer, slots=None, t_slice=None):
    """Fetched fp16 vs the oracle's float64 decode of the GPU's own codes, per head."""
    out = out_gpu.float().cpu().numpy().astype(np.float64)
    worst = (0.0, 0.0)
    for s in (range(rl.n_slots) if slots is None else slots):
        rows, side = gpu_layer.slot_rows(s)
        rows = rows.cpu().numpy()
        sd = None
        if side is not None:
            sd = side.cpu().numpy().view(np.float16)
            if rl.mode in ("codebook", "int8"):
                sd = sd[:, 0]
        if t_slice is not None:
            rows = rows[t_slice]
            sd = sd[t_slice] if sd is not None else None
        ref = rl.decode(s, rows, sd)
        b, g = divmod(s, rl.Hg)
        for j in range(rl.hpg):
            h = g * rl.hpg + j
            o = out[b, h] if t_slice is None else out[b, h][t_slice]
            rh = ref[:, j * rl.D:(j + 1) * rl.D]
            err = o - rh
            mx = max(np.abs(rh).max(), 1e-30)
            rms = max(math.sqrt(np.mean(rh ** 2)), 1e-30)
            ma, re = np.abs(err).max() / mx, math.sqrt(np.mean(err ** 2)) / rms
            assert ma <= MAX_ABS_REL, f"slot {s} head {h}: max-abs error {ma:.2e} of max|x_hat|"
            assert re <= RMS_REL, f"slot {s} head {h}: RMS error {re:.2e} of RMS(x_hat)"
            worst = (max(worst[0], ma), max(worst[1], re))
    return worst


def to_device(x: torch.Tensor, dev):
    return x.to(dev).contiguous()
