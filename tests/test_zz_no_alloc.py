"""kvc_append_noalloc: the append for callers that may not allocate device memory.

A plugin or custom operator run inside another inference engine's execution
step is handed its buffers and must not call cudaMalloc there, and a server
whose device memory is all reserved by its own pool has none left for it.
Such a caller passes the descriptor, its store and its input on every call;
the library keeps the kernel's tables in one static device array instead of
allocating a parameter block.

This file is collected last (its name sorts after the other test files), so
a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from kvc_cases import fit_group, fit_uniform

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rank_quantized_kv_gb300 as kvc

    kvc.load_library()
    return kvc


def _noalloc(kvc, desc, length, x):
    """One kvc_append_noalloc call through the C ABI on the current stream."""
    lib = kvc.load_library()
    sb, sh, st, _ = x.stride()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = lib.kvc_append_noalloc(ctypes.byref(desc), length, ctypes.c_void_p(x.data_ptr()),
                                    x.shape[2], sb, sh, st, stream)
    assert status == 0, lib.kvc_last_error().decode()


@pytest.mark.parametrize("mode", ["uniform", "group", "int8"])
def test_noalloc_matches_kvc_append_on_two_calls(kvc, mode):
    dev = torch.device("cuda:0")
    B, H, D = 2, 8, 128
    if mode == "group":
        x = synth.group_spectral(B, H, 300, D, 4, alpha=1.0, seed=9100, tensor=0, dtype="bf16")
        params = fit_group(x.double().numpy()[:, :, :200], 4, 64)
    elif mode == "int8":
        x = synth.kv_spectral(B, H, 300, D, alpha=1.0, seed=9200, tensor=1, dtype="bf16")
        params = {}
    else:
        x = synth.kv_spectral(B, H, 300, D, alpha=1.0, seed=9300, tensor=0, n_outliers=3,
                              dtype="bf16")
        params = fit_uniform(x.double().numpy(), 256, 32, [0, 2, 4, 8], 128)
    xd = x.to(dev)
    T1, T2 = 171, 129                       # two calls, ragged against 8-token tiles
    ref = kvc.KVCacheLayer(mode, B, H, D, in_dtype="bf16", capacity=T1 + T2, device=dev,
                           path="generic", **params)
    desc, keep = kvc._build_desc(mode, B, H, D, None, params.get("V"), params.get("mean"),
                                 params.get("bits"), params.get("qmin"), params.get("qstep"),
                                 params.get("basis_of"), params.get("heads_per_group", 1),
                                 params.get("group_size", 32), None, "bf16", "f16", T1 + T2)
    store = torch.zeros_like(ref.store)     # the caller's own buffer
    desc.store = ctypes.c_void_p(store.data_ptr())
    desc.store_bytes = store.numel()

    ref.append(xd[:, :, :T1])
    _noalloc(kvc, desc, 0, xd[:, :, :T1])
    torch.cuda.synchronize()
    assert torch.equal(store, ref.store), "first call differs from kvc_append"

    ref.append(xd[:, :, T1:])
    _noalloc(kvc, desc, T1, xd[:, :, T1:])
    torch.cuda.synchronize()
    assert torch.equal(store, ref.store), "second call differs from kvc_append"


def test_noalloc_rejects_tables_beyond_its_limit(kvc):
    # 8 bases of 1024 x 256 need 2 x 8 MiB of basis tables alone.
    rng = np.random.default_rng(0)
    nb, d_in, r = 8, 1024, 256
    V = rng.standard_normal((nb, d_in, r)).astype(np.float32)
    bits = np.full((nb, r), 2, dtype=np.uint8)
    desc, keep = kvc._build_desc("uniform", 1, 8, d_in, None, V, None, bits, np.zeros((nb, r)),
                                 np.ones((nb, r)), np.arange(8), 1, 32, None, "bf16", "f16", 16)
    n = kvc.store_bytes("uniform", 1, 8, d_in, capacity=16, V=V, bits=bits,
                        qmin=np.zeros((nb, r)), qstep=np.ones((nb, r)), basis_of=np.arange(8))
    store = torch.zeros(n, dtype=torch.uint8, device="cuda:0")
    desc.store = ctypes.c_void_p(store.data_ptr())
    desc.store_bytes = n
    x = torch.zeros(1, 8, 4, d_in, dtype=torch.bfloat16, device="cuda:0")
    lib = kvc.load_library()
    st = lib.kvc_append_noalloc(ctypes.byref(desc), 0, ctypes.c_void_p(x.data_ptr()), 4,
                                *x.stride()[:3], None)
    assert st == -1 and b"8 MiB" in lib.kvc_last_error()
    torch.cuda.synchronize()
    assert int(store.count_nonzero()) == 0


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_noalloc_refuses_stream_capture(kvc):
    # The tables are uploaded from a host buffer freed on return, so a captured
    # call would replay a stale upload: the call must refuse and enqueue nothing.
    B, H, D = 1, 8, 128
    x = synth.kv_spectral(B, H, 40, D, alpha=1.0, seed=9400, tensor=0, dtype="bf16")
    params = fit_uniform(x.double().numpy(), 256, 32, [0, 2, 4, 8], 128)
    desc, keep = kvc._build_desc("uniform", B, H, D, None, params["V"], params["mean"],
                                 params["bits"], params["qmin"], params["qstep"],
                                 params.get("basis_of"), 1, 32, None, "bf16", "f16", 64)
    n = kvc.store_bytes("uniform", B, H, D, capacity=64, V=params["V"], bits=params["bits"],
                        qmin=params["qmin"], qstep=params["qstep"],
                        basis_of=params.get("basis_of"))
    store = torch.zeros(n, dtype=torch.uint8, device="cuda:0")
    desc.store = ctypes.c_void_p(store.data_ptr())
    desc.store_bytes = n
    xd = x.to("cuda:0")
    lib = kvc.load_library()
    sb, sh, st_, _ = xd.stride()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        cur = torch.cuda.current_stream().cuda_stream
        status = lib.kvc_append_noalloc(ctypes.byref(desc), 0, ctypes.c_void_p(xd.data_ptr()),
                                        xd.shape[2], sb, sh, st_, ctypes.c_void_p(cur))
    assert status == -1 and b"capture" in lib.kvc_last_error()
    torch.cuda.synchronize()
    assert int(store.count_nonzero()) == 0
    # Outside the capture the same call succeeds.
    _noalloc(kvc, desc, 0, xd)
    torch.cuda.synchronize()
    assert int(store.count_nonzero()) > 0
