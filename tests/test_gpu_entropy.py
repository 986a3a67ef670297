"""GPU parity of the code histogram (kvc_code_histogram, exact counts) and of
the Huffman byte accounting (kvc_entropy_bytes) against the oracle
(oracle/entropy.py) applied to the GPU's own stored codes."""
import numpy as np
import pytest
import torch

import synth
from oracle import codec
from oracle import entropy as en
from oracle.layer import OracleLayer

from kvc_cases import fit_codebook, fit_group, fit_uniform, oracle_kwargs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rank_quantized_kv_gb300 as kvc

    kvc.load_library()
    return kvc


def _positions(bits):
    """Packed (chunk-aligned) position of each kept component, in order."""
    pos, nch = {}, 0
    for w, comps in codec.segments(bits):
        for m, k in enumerate(comps):
            pos[k] = nch * 8 + m
        nch += (len(comps) + 7) // 8
    return pos


@pytest.mark.parametrize("mode", ["uniform", "codebook", "group"])
def test_histogram_and_entropy_bytes(kvc, mode):
    dev = torch.device("cuda:0")
    B, H, D, S = 2, 4, 128, 1500
    if mode == "uniform":
        x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=9500, tensor=0, n_outliers=3,
                              dtype="bf16")
        params = fit_uniform(x.double().numpy(), 512, 32, [0, 1, 2, 3, 4, 8], 96)
        dt = "bf16"
    elif mode == "codebook":
        x = synth.heavy_tailed_keys(B, H, S, D, seed=9501, dtype="f16")
        params, dt = fit_codebook(D), "f16"
    else:
        x = synth.group_spectral(B, H, S, D, 2, alpha=1.0, seed=9502, tensor=0, dtype="bf16")
        params, dt = fit_group(x.double().numpy(), 2, 64), "bf16"
    gl = kvc.KVCacheLayer(mode, B, H, D, in_dtype=dt, capacity=S, device=dev, **params)
    gl.append(x.to(dev))
    assert gl.sync_status() == 0
    rl = OracleLayer(mode, B, H, D, capacity=S, **oracle_kwargs(params))
    # the oracle accounts for the GPU's own codes
    rl.len = S
    for s in range(rl.n_slots):
        rows, _ = gl.slot_rows(s)
        rl.rows[s] = rows.cpu().numpy()
    counts = gl.code_histogram().cpu().numpy().astype(np.int64)
    for s in range(rl.n_slots):
        bits = rl.bits[rl.basis_of[s]]
        codes = codec.unpack_rows(rl.rows[s], bits)
        pos = _positions(bits)
        for k, j in pos.items():
            want = np.bincount(codes[:, k], minlength=256)
            assert np.array_equal(counts[s, j], want), (s, k, j)
    got = gl.entropy_bytes()
    ref = en.layer_bytes(rl)
    assert got["pre_entropy"] == ref["pre_entropy"]
    assert got["stored_payload"] == ref["stored_payload"]
    assert got["params"] == ref["params"]
    assert got["gain"] == pytest.approx(ref["gain"], rel=1e-12)
    assert got["stored_payload"] <= got["pre_entropy"]
