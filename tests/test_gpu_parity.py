"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Packed codes must match the oracle byte for byte (a mismatch is tolerated
only at an oracle near-tie, at most 1e-6 of the codes); fp16 side words
exactly; the fetched reconstruction within max-abs 4e-3 max|x_hat| and RMS
1e-3 RMS(x_hat) per head of the oracle's float64 decode of the GPU's codes.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import codec, fit
from oracle.layer import OracleLayer

from kvc_cases import (MISMATCH_RATE, check_fetch, compare_codes, fit_codebook, fit_group,
                       fit_uniform, oracle_kwargs)

pytestmark = pytest.mark.gpu

PATHS = ["auto", "generic"]


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rank_quantized_kv_gb300 as kvc

    kvc.load_library()
    return kvc


def _dev():
    return torch.device("cuda:0")


def _all_slots_match(gl, rl, x64):
    n, mism = 0, 0
    for s in range(rl.n_slots):
        rows, side = gl.slot_rows(s)
        X = rl.slot_rows(x64, s)
        c, m = compare_codes(rows.cpu().numpy(), None if side is None else side.cpu().numpy(),
                             rl, s, X)
        n, mism = n + c, mism + m
    assert mism <= MISMATCH_RATE * n, f"{mism} code mismatches out of {n}"
    return n, mism


def _make(kvc, mode, B, H, D, params, in_dtype, capacity, path):
    gl = kvc.KVCacheLayer(mode, B, H, D, in_dtype=in_dtype, capacity=capacity, device=_dev(),
                          path=path, **params)
    rl = OracleLayer(mode, B, H, D, capacity=capacity, **oracle_kwargs(params))
    return gl, rl


# ------------------------------------------------------------------------- config 1

@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("tensor", [0, 1])
def test_cfg1_kvtc_tiny(kvc, path, tensor):
    """B=1, H=2, D=64, fp32; fit on a 64-token prefill (r=16, {0,1,2,4,8}, 48 bits);
    then 16 tokens appended one at a time."""
    B, H, D = 1, 2, 64
    x = synth.kv_spectral(B, H, 80, D, alpha=0.8, seed=1000, tensor=tensor, dtype="f32")
    x64 = x.double().numpy()
    params = fit_uniform(x64, 64, 16, [0, 1, 2, 4, 8], 48)
    gl, rl = _make(kvc, "uniform", B, H, D, params, "f32", 80, path)
    xd = x.to(_dev())
    gl.append(xd[:, :, :64].contiguous())
    for t in range(64, 80):
        gl.append(xd[:, :, t:t + 1])
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    out = gl.fetch()
    check_fetch(out, gl, rl)
    assert gl.nbytes() == rl.nbytes()


# ------------------------------------------------------------------------- config 2

def _cfg2_inputs(B, H, S, tensor):
    x = synth.kv_spectral(B, H, S, 128, alpha=1.0, seed=2000, tensor=tensor, n_outliers=3,
                          dtype="bf16")
    return x, x.double().numpy()


@pytest.mark.parametrize("path", PATHS)
def test_cfg2_scaled(kvc, path):
    """Llama-3-8B-like head shape (D=128, bf16, 2 % outlier channels), fewer heads
    and tokens: fit on 512, r=32, {0,2,4,8}, 128 bits; 700 tokens (ragged tail)."""
    B, H, S = 2, 4, 700
    x, x64 = _cfg2_inputs(B, H, S, 0)
    params = fit_uniform(x64, 512, 32, [0, 2, 4, 8], 128)
    gl, rl = _make(kvc, "uniform", B, H, 128, params, "bf16", S + 8, path)
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)


@pytest.mark.parametrize("tensor", [0, 1])
def test_cfg2_full(kvc, tensor):
    """B=8, H_kv=8, D=128, S=4096 appended in one call, then one decode token."""
    B, H, S = 8, 8, 4097
    x, x64 = _cfg2_inputs(B, H, S, tensor)
    params = fit_uniform(x64, 512, 32, [0, 2, 4, 8], 128)
    gl, rl = _make(kvc, "uniform", B, H, 128, params, "bf16", S, "auto")
    xd = x.to(_dev())
    gl.append(xd[:, :, :4096])
    gl.append(xd[:, :, 4096:])
    assert gl.sync_status() == 0
    rl.append(x64)
    n, mism = _all_slots_match(gl, rl, x64)
    c = gl.counters()
    print(f"cfg2 full: {n} codes, {mism} tie mismatches, counters {c}")
    # the fast path's error stays well inside the bound it is flagged against
    assert c["max_error_ratio"] < 0.5
    check_fetch(gl.fetch(), gl, rl)


# ------------------------------------------------------------------------- config 3

def _cfg3_inputs(B, H, S, hpg, tensor):
    x = synth.group_spectral(B, H, S, 128, hpg, alpha=1.0, seed=3000, tensor=tensor,
                             n_outliers=20, dtype="bf16")
    return x, x.double().numpy()


@pytest.mark.parametrize("path", PATHS)
def test_cfg3_scaled(kvc, path):
    """PALU group mode: groups of 8 heads (D_in = 1024 -> r = 256), 25 % of the
    components at 4 bits, the rest at 2, fp16 scale per 32 components."""
    B, H, S, hpg = 2, 16, 300, 8
    x, x64 = _cfg3_inputs(B, H, S, hpg, 0)
    params = fit_group(x64, hpg, 256)
    gl, rl = _make(kvc, "group", B, H, 128, params, "bf16", S, path)
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)
    nb = gl.nbytes()
    assert nb == rl.nbytes()
    # effective bits (palu_cache page "Byte accounting"): (r / D_in) * average bits
    assert nb["payload"] * 8 / (B * H * S * 128) == pytest.approx(256 / 1024 * 2.5)


@pytest.mark.slow
def test_cfg3_full_sampled(kvc):
    """32 KV heads, 4 groups of 8, B=4, S=8192 on the GPU; the oracle checks two
    slots in full and the fetch on sampled token ranges of every slot."""
    B, H, S, hpg = 4, 32, 8192, 8
    x, x64 = _cfg3_inputs(B, H, S, hpg, 1)
    params = fit_group(x64, hpg, 256)
    gl, rl = _make(kvc, "group", B, H, 128, params, "bf16", S, "auto")
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    n = mism = 0
    for s in (0, rl.n_slots - 1):
        rows, side = gl.slot_rows(s)
        c, m = compare_codes(rows.cpu().numpy(), side.cpu().numpy(), rl, s, rl.slot_rows(x64, s))
        n, mism = n + c, mism + m
    assert mism <= MISMATCH_RATE * n
    out = gl.fetch()
    check_fetch(out, gl, rl, t_slice=slice(4000, 4400))
    print(f"cfg3 full: counters {gl.counters()}")


def _same_store(ga, gb, n_slots):
    for s in range(n_slots):
        ra, sa = ga.slot_rows(s)
        rb, sb = gb.slot_rows(s)
        assert torch.equal(ra, rb), f"slot {s}: packed rows differ"
        assert torch.equal(sa, sb), f"slot {s}: side words differ"


def test_group_tensor_core_projection_chunks(kvc):
    """Group mode with the tensor-core projection in two chunks (16 slots, r = 256:
    2048 tokens per chunk, then a ragged 452).  Codes against the oracle on two
    slots; the whole store equal to the CUDA-core projection's (both decide every
    code exactly)."""
    B, H, S, hpg = 8, 16, 2500, 8
    x, x64 = _cfg3_inputs(B, H, S, hpg, 0)
    params = fit_group(x64[:, :, :512], hpg, 256)
    ga, rl = _make(kvc, "group", B, H, 128, params, "bf16", S, "auto")
    gg, _ = _make(kvc, "group", B, H, 128, params, "bf16", S, "generic")
    xd = x.to(_dev())
    ga.append(xd)
    gg.append(xd)
    assert ga.sync_status() == 0 and gg.sync_status() == 0
    c = ga.counters()
    assert c["launches"] == 4, c  # per chunk: the projection, then the quantiser
    assert c["max_error_ratio"] < 1.0, c
    _same_store(ga, gg, rl.n_slots)
    n = mism = 0
    for s in (0, rl.n_slots - 1):
        rows, side = ga.slot_rows(s)
        cc, m = compare_codes(rows.cpu().numpy(), side.cpu().numpy(), rl, s, rl.slot_rows(x64, s))
        n, mism = n + cc, mism + m
    assert mism <= MISMATCH_RATE * n
    print(f"group tensor-core projection: counters {c}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_group_tile_beyond_split_range(kvc, dtype):
    """Tokens with |x - mean| in the thousands, beyond the fp16 split the
    tensor-core projection uses: their 128-token tiles are projected on the CUDA
    cores instead, and every code still matches the oracle (bf16 and fp16 x)."""
    B, H, S, hpg = 1, 16, 300, 8
    x, x64 = _cfg3_inputs(B, H, S, hpg, 1)
    params = fit_group(x64, hpg, 256)
    x[0, 3, 150, 5] = 3000.0
    x[0, 9, 20, 100] = -2500.0
    if dtype == "f16":
        x = x.to(torch.float16)
    x64 = x.double().numpy()
    gl, rl = _make(kvc, "group", B, H, 128, params, dtype, S, "auto")
    gg, _ = _make(kvc, "group", B, H, 128, params, dtype, S, "generic")
    gl.append(x.to(_dev()))
    gg.append(x.to(_dev()))
    assert gl.sync_status() == 0 and gg.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    _same_store(gl, gg, rl.n_slots)
    check_fetch(gl.fetch(), gl, rl)


@pytest.mark.parametrize("dtype, path", [("f32", "generic"), ("f16", "auto"), ("f16", "generic"),
                                         ("bf16", "auto")])
def test_group_tiny_group_latents(kvc, dtype, path):
    """Rows whose latents in one 32-component group are tiny against
    ||x - mean|| (log-spread from 0 to 1e-2 of it): the group's maximum is at
    or below a few times the projection's error bound, where the fp32 scale,
    the maximum's own code and the codes next to the outer boundaries can all
    be wrong.  Every code and fp16 scale against the oracle; the tensor-core
    and CUDA-core projections store the same bytes."""
    B, H, D, hpg, r, S = 1, 16, 128, 8, 64, 256
    base = synth.group_spectral(B, H, 400, D, hpg, alpha=1.0, seed=7700, tensor=0, dtype="f32")
    params = fit_group(base.double().numpy(), hpg, r)
    rng = np.random.default_rng(7701)
    d_in = hpg * D
    x64 = np.zeros((B, H, S, D))
    for g in range(H // hpg):
        V = params["V"][g].astype(np.float64)
        m = params["mean"][g].astype(np.float64)
        c = rng.standard_normal((S, r)) * 0.3
        qg = rng.integers(0, r // 32, size=S)  # the tiny group of each row
        eps = np.concatenate([[0.0], 10.0 ** rng.uniform(-8, -2, size=S - 1)])
        for t in range(S):
            c[t, 32 * qg[t]:32 * qg[t] + 32] = eps[t] * rng.standard_normal(32)
        w = rng.standard_normal((S, d_in))
        w -= (w @ V) @ np.linalg.pinv(V)  # no component in the basis's span
        w *= 1.0 / np.linalg.norm(w, axis=1, keepdims=True)
        rows = m + c @ V.T + w
        for hh in range(hpg):
            x64[0, g * hpg + hh] = rows[:, hh * D:(hh + 1) * D]
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    x = torch.from_numpy(x64).to(tdt)
    x64 = x.double().numpy()
    gl, rl = _make(kvc, "group", B, H, D, params, dtype, S, path)
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    if dtype != "f32":
        gg, _ = _make(kvc, "group", B, H, D, params, dtype, S, "generic" if path == "auto" else "auto")
        gg.append(x.to(_dev()))
        assert gg.sync_status() == 0
        _same_store(gl, gg, rl.n_slots)
    print(f"tiny group latents {dtype}/{path}: counters {gl.counters()}")


@pytest.mark.parametrize("hpg, r, dtype", [(2, 20, "bf16"), (4, 128, "f16")])
def test_group_tensor_core_ranks(kvc, hpg, r, dtype):
    """The tensor-core group projection at other ranks: r = 20 (N padded to 32,
    the padding columns never written) and r = 128 (32 components per epilogue
    thread); D = 64, 200 tokens.  Codes against the oracle, and the same store as
    the CUDA-core projection."""
    B, S, D = 2, 200, 64
    H = 2 * hpg
    x = synth.group_spectral(B, H, S, D, hpg, alpha=1.0, seed=7300 + r, tensor=0, dtype=dtype)
    x64 = x.double().numpy()
    params = fit_group(x64, hpg, r)
    ga, rl = _make(kvc, "group", B, H, D, params, dtype, S, "auto")
    gg, _ = _make(kvc, "group", B, H, D, params, dtype, S, "generic")
    xd = x.to(_dev())
    ga.append(xd)
    gg.append(xd)
    assert ga.sync_status() == 0 and gg.sync_status() == 0
    assert ga.counters()["launches"] == 2  # the projection, then the quantiser
    rl.append(x64)
    _all_slots_match(ga, rl, x64)
    _same_store(ga, gg, rl.n_slots)
    check_fetch(ga.fetch(), ga, rl)


@pytest.mark.parametrize("D, dtype", [(80, "bf16"), (36, "f16")])
def test_uniform_odd_shapes(kvc, D, dtype):
    """Head sizes that are not multiples of 64 (the CUDA-core kernels; D = 36 is
    not a multiple of 8 either, so x loads one value at a time), 3 heads, r = 20,
    widths {0,1,2,3,4,8} with 3-bit codes straddling bytes, a ragged 77 tokens."""
    B, H, S = 2, 3, 77
    x = synth.kv_spectral(B, H, S, D, alpha=0.9, seed=7100, tensor=0, dtype=dtype)
    x64 = x.double().numpy()
    params = fit_uniform(x64, S, 20, [0, 1, 2, 3, 4, 8], 53)
    gl, rl = _make(kvc, "uniform", B, H, D, params, dtype, S, "auto")
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)


def test_group_odd_shapes(kvc):
    """Group mode with 3 heads of D = 40 per group (D_in = 120, not a power of
    two), r = 48 (a full and a half 32-component group), fp16 input, 150 tokens."""
    B, H, S, D, hpg = 2, 6, 150, 40, 3
    x = synth.group_spectral(B, H, S, D, hpg, alpha=1.0, seed=7200, tensor=0, dtype="f16")
    x64 = x.double().numpy()
    params = fit_group(x64, hpg, 48)
    gl, rl = _make(kvc, "group", B, H, D, params, "f16", S, "auto")
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)


# ------------------------------------------------------------------------- config 4

@pytest.mark.parametrize("path", PATHS)
def test_cfg4_keys_scaled(kvc, path):
    """Rotation + 3-bit Lloyd-Max codebook for N(0, 1/128), fp16 norm; keys with
    1 % Student-t (nu = 3) coordinates."""
    B, H, S, D = 2, 4, 520, 128
    x = synth.heavy_tailed_keys(B, H, S, D, seed=4000, dtype="f16")
    x64 = x.double().numpy()
    params = fit_codebook(D)
    gl, rl = _make(kvc, "codebook", B, H, D, params, "f16", S, path)
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    assert gl.counters()["max_error_ratio"] < 0.5
    check_fetch(gl.fetch(), gl, rl)
    assert gl.nbytes()["payload"] == B * H * S * 48        # ceil(128 * 3 / 8)


@pytest.mark.parametrize("D, bits", [(128, 1), (128, 2), (128, 4), (64, 3), (256, 3), (256, 2)])
@pytest.mark.parametrize("path", PATHS)
def test_codebook_widths_and_heads(kvc, D, bits, path):
    """Codebook keys at 1, 2, 3 and 4 bits and head sizes 64, 128 and 256 (the
    fetch decodes widths up to 3 four codes per lookup, 4 bits by pairs), with
    a ragged last tile: codes and norms against the oracle, the fetch within
    its tolerance of the oracle's decode of the GPU's rows."""
    B, H, S = 2, 2, 300
    x = synth.heavy_tailed_keys(B, H, S, D, seed=4200 + D + bits, dtype="f16")
    x64 = x.double().numpy()
    params = fit_codebook(D, bits=bits, seed=77 + bits)
    gl, rl = _make(kvc, "codebook", B, H, D, params, "f16", S, path)
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)
    assert gl.nbytes()["payload"] == B * H * S * (D * bits // 8)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_cfg4_values_int8(kvc, dtype):
    B, H, S, D = 2, 8, 1000, 128
    x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=4100, tensor=1, dtype=dtype)
    x[0, 0, 5] = 0                                         # a zero row: scale 1e-8 -> fp16 0
    x[0, 1, 7, :4] = torch.tensor([127.0, 63.5, -0.5, 2.5])  # exact ties
    x[0, 1, 7, 4:] = 0
    x64 = x.double().numpy()
    gl, rl = _make(kvc, "int8", B, H, D, {}, dtype, S, "auto")
    gl.append(x.to(_dev()))
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    out = gl.fetch().float().cpu().numpy()
    assert np.array_equal(out, rl.fetch().astype(np.float16).astype(np.float32))
    assert gl.nbytes()["payload"] + gl.nbytes()["side"] == B * H * S * (D + 2)


@pytest.mark.slow
def test_cfg4_full(kvc):
    """B=16, H_kv=8, S=16384: keys in codebook mode, values int8; sampled oracle."""
    B, H, S, D = 16, 8, 16384, 128
    dev = _dev()
    keys = synth.heavy_tailed_keys(B, H, S, D, seed=4000, dtype="f16")
    params = fit_codebook(D)
    gk = kvc.KVCacheLayer("codebook", B, H, D, in_dtype="f16", capacity=S, device=dev, **params)
    rk = OracleLayer("codebook", B, H, D, **oracle_kwargs(params))
    gk.append(keys.to(dev))
    assert gk.sync_status() == 0
    k64 = keys.double().numpy()
    n = mism = 0
    for s in (0, 77, B * H - 1):
        rows, side = gk.slot_rows(s)
        c, m = compare_codes(rows.cpu().numpy(), side.cpu().numpy(), rk, s, rk.slot_rows(k64, s))
        n, mism = n + c, mism + m
    assert mism <= MISMATCH_RATE * max(n, 1)
    check_fetch(gk.fetch(), gk, rk, slots=(0, 77, B * H - 1), t_slice=slice(9000, 9500))
    print(f"cfg4 keys full: counters {gk.counters()}")
    del gk
    vals = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=4100, tensor=1, dtype="f16")
    gv = kvc.KVCacheLayer("int8", B, H, D, in_dtype="f16", capacity=S, device=dev)
    rv = OracleLayer("int8", B, H, D)
    gv.append(vals.to(dev))
    v64 = vals.double().numpy()
    for s in (3, 100):
        rows, side = gv.slot_rows(s)
        compare_codes(rows.cpu().numpy(), side.cpu().numpy(), rv, s, rv.slot_rows(v64, s))


# ------------------------------------------------------------------------- config 5

@pytest.mark.parametrize("B,S,r,bits", [(1, 1024, 32, 2), (8, 1024, 64, 4), (1, 8192, 64, 2)])
def test_cfg5_points(kvc, B, S, r, bits):
    """Llama-3-70B-like KV shape (H_kv=8, D=128), uniform all-b allocation,
    frozen min/step from the first min(S, 4096) tokens; full oracle check."""
    H, D = 8, 128
    x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=5000 + S, tensor=0, dtype="bf16")
    x64 = x.double().numpy()
    fl = min(S, 4096)
    p = fit_uniform(x64, fl, r, [bits], bits * r)
    assert np.all(p["bits"] == bits)
    gl, rl = _make(kvc, "uniform", B, H, D, p, "bf16", S, "auto")
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)


@pytest.mark.parametrize("r, bits", [(32, 1), (64, 2), (32, 4), (64, 8), (40, 4), (36, 2)])
@pytest.mark.parametrize("path", PATHS)
def test_uniform_one_width(kvc, r, bits, path):
    """Every kept component at one width (the fetch decodes such rows chunk by
    chunk from aligned loads when the rank is a multiple of 8; r = 36 keeps a
    partial chunk and takes the chunk table), a ragged last tile; codes against
    the oracle and the fetch within its tolerance."""
    B, H, D, S = 2, 2, 128, 300
    x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=5100 + r + bits, tensor=0, dtype="bf16")
    x64 = x.double().numpy()
    p = fit_uniform(x64, S, r, [bits], bits * r)
    assert np.all(p["bits"] == bits)
    gl, rl = _make(kvc, "uniform", B, H, D, p, "bf16", S, path)
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)


@pytest.mark.parametrize("r,choices,budget", [(128, [0, 2, 4, 8], 384), (96, [0, 4, 8], 384)])
def test_uniform_wide_rank_bf16(kvc, r, choices, budget):
    """bf16 input, one basis per (b, h), rank above 64: the basis' three 16-bit
    pieces no longer stack along one MMA N (3 r > 256), so the append takes
    its one-tile-per-CTA tensor-core kernel.  Several tiles and a ragged tail."""
    B, H, D, S = 1, 2, 128, 300
    x = synth.kv_spectral(B, H, S, D, alpha=0.7, seed=7100 + r, tensor=0, dtype="bf16")
    x64 = x.double().numpy()
    p = fit_uniform(x64, 256, r, choices, budget)
    gl, rl = _make(kvc, "uniform", B, H, D, p, "bf16", S, "auto")
    gl.append(x.to(_dev()))
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    check_fetch(gl.fetch(), gl, rl)


# ------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("mode", ["uniform", "group", "codebook", "int8"])
def test_streaming_equals_bulk_on_gpu(kvc, mode):
    """kvtc_cache page, "NOT PATH-DEPENDENT": prefill then one token at a time
    stores exactly what one bulk append stores."""
    B, H, D, S = 2, 8, 128, 160
    if mode == "group":
        x = synth.group_spectral(B, H, S, D, 4, alpha=1.0, seed=6000, tensor=0, dtype="bf16")
        params = fit_group(x.double().numpy()[:, :, :100], 4, 64)
        dt = "bf16"
    elif mode == "codebook":
        x = synth.heavy_tailed_keys(B, H, S, D, seed=6001, dtype="f16")
        params, dt = fit_codebook(D), "f16"
    elif mode == "int8":
        x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=6002, tensor=1, dtype="f16")
        params, dt = {}, "f16"
    else:
        x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=6003, tensor=0, dtype="bf16")
        params = fit_uniform(x.double().numpy(), 100, 32, [0, 2, 4, 8], 128)
        dt = "bf16"
    dev = _dev()
    a = kvc.KVCacheLayer(mode, B, H, D, in_dtype=dt, capacity=S, device=dev, **params)
    b = kvc.KVCacheLayer(mode, B, H, D, in_dtype=dt, capacity=S, device=dev, **params)
    xd = x.to(dev)
    a.append(xd)
    b.append(xd[:, :, :130])
    for t in range(130, S):
        b.append(xd[:, :, t:t + 1])
    assert torch.equal(a.store, b.store)
    assert torch.equal(a.fetch(), b.fetch())


def test_all_dropped_fetches_the_mean_exactly(kvc):
    B, H, D, r = 1, 4, 128, 16
    rng = np.random.default_rng(7)
    V = np.linalg.qr(rng.standard_normal((D, D)))[0][:, :r].astype(np.float32)
    mean = rng.standard_normal((1, D)).astype(np.float32)
    gl = kvc.KVCacheLayer("uniform", B, H, D, V=V, mean=mean, bits=np.zeros(r), qmin=np.zeros(r),
                          qstep=np.ones(r), in_dtype="bf16", capacity=300, device=_dev())
    x = torch.randn(B, H, 300, D, device=_dev()).to(torch.bfloat16)
    gl.append(x)
    out = gl.fetch()
    want = torch.from_numpy(mean[0]).to(torch.float16).to(_dev()).expand(B, H, 300, D)
    assert torch.equal(out, want)
    assert gl.nbytes()["payload"] == 0


def test_full_rank_8bit_near_lossless(kvc):
    B, H, D, S = 1, 2, 64, 500
    x = synth.kv_spectral(B, H, S, D, alpha=0.5, seed=7000, tensor=0, dtype="f32")
    x64 = x.double().numpy()
    params = fit_uniform(x64, S, D, [8], 8 * D)
    gl = kvc.KVCacheLayer("uniform", B, H, D, in_dtype="f32", capacity=S, device=_dev(), **params)
    gl.append(x.to(_dev()))
    out = gl.fetch().double().cpu().numpy()
    for h in range(H):
        bound = math.sqrt(np.sum((params["qstep"][h].astype(np.float64) / 2) ** 2))
        err = np.linalg.norm(out[0, h] - x64[0, h], axis=1)
        # quantisation bound plus the fp16 output rounding
        assert np.all(err <= bound + 2 ** -11 * np.linalg.norm(x64[0, h], axis=1) + 1e-6)


def test_trim_capacity_and_ld_s(kvc):
    B, H, D, S = 2, 4, 128, 200
    x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=8000, tensor=0, dtype="bf16")
    params = fit_uniform(x.double().numpy(), 128, 32, [0, 2, 4, 8], 128)
    dev = _dev()
    gl = kvc.KVCacheLayer("uniform", B, H, D, in_dtype="bf16", capacity=S, device=dev, **params)
    xd = x.to(dev)
    gl.append(xd)
    full = gl.fetch()
    with pytest.raises(kvc.KvcError) as e:
        gl.append(xd[:, :, :1])
    assert e.value.status == -3 and len(gl) == S
    assert gl.trim(0) == 0 and gl.trim(-5) == 0
    assert gl.trim(50) == 50 and len(gl) == 150
    assert torch.equal(gl.fetch(), full[:, :, :150])
    gl.append(xd[:, :, 150:])
    assert torch.equal(gl.fetch(), full)
    # rows beyond the length are left untouched in a taller output
    out = torch.full((B, H, S + 37, D), 7.0, dtype=torch.float16, device=dev)
    gl.fetch(out=out)
    assert torch.equal(out[:, :, :S], full) and bool((out[:, :, S:] == 7).all())
    assert gl.trim(10**9) == S and len(gl) == 0
    assert gl.fetch().shape == (B, H, 0, D)
    gl.append(xd[:, :, :3])                          # the basis survives trimming to zero
    assert torch.equal(gl.fetch(), full[:, :, :3])


def test_host_pointer_is_rejected(kvc):
    B, H, D = 1, 1, 128
    gl = kvc.KVCacheLayer("int8", B, H, D, in_dtype="f16", capacity=4, device=_dev())
    with pytest.raises(kvc.KvcError) as e:
        gl.append(torch.zeros(B, H, 2, D, dtype=torch.float16))     # CPU tensor
    assert e.value.status == -1 and len(gl) == 0


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_int8_values_pipelined_many_steps(kvc, dtype):
    """Enough rows (4 x 8 x 3001, ragged) that every block of the persistent,
    pipelined int8 append walks several steps; rows read through strides."""
    B, H, S, D = 4, 8, 3001, 128
    x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=4200, tensor=1, dtype=dtype)
    x64 = x.double().numpy()
    gl, rl = _make(kvc, "int8", B, H, D, {}, dtype, S, "auto")
    xs = x.permute(0, 2, 1, 3).contiguous().to(_dev()).permute(0, 2, 1, 3)
    gl.append(xs)
    assert gl.sync_status() == 0
    rl.append(x64)
    _all_slots_match(gl, rl, x64)
    assert gl.counters()["appended"] == S
