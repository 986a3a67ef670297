"""The C-ABI library: it loads, exports every symbol include/kvc.h declares,
and validates descriptors on the host (no GPU needed, no compute calls)."""
import ctypes
import math
import re
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def kvc():
    import rank_quantized_kv_gb300 as kvc

    try:
        kvc.load_library()
    except ImportError:
        import __graft_entry__

        __graft_entry__.build()
        kvc.load_library()
    return kvc


def _declared():
    text = (ROOT / "include" / "kvc.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(kvc_\w+)\s*\(", text))


def test_exports_every_declared_symbol(kvc):
    declared = _declared()
    assert declared == set(kvc.EXPORTED_SYMBOLS)
    lib = ctypes.CDLL(kvc.library_path())
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.kvc_abi_version() == 1


def _uniform_args(rng, nb=3, B=2, H=4, D=32, r=8):
    V = rng.standard_normal((nb, D, r)).astype(np.float32)
    bits = rng.choice([0, 1, 2, 3, 4, 8], size=(nb, r)).astype(np.uint8)
    return dict(V=V, mean=rng.standard_normal((nb, D)), bits=bits,
                qmin=-np.ones((nb, r)), qstep=np.full((nb, r), 0.1),
                basis_of=rng.integers(0, nb, size=B * H))


def test_store_bytes_covers_every_slot(kvc):
    rng = np.random.default_rng(0)
    a = _uniform_args(rng)
    P = [sum(math.ceil(int(np.sum(bb == w)) * w / 8) for w in (8, 4, 3, 2, 1)) for bb in a["bits"]]
    need = sum(100 * P[b] for b in a["basis_of"])
    n100 = kvc.store_bytes("uniform", 2, 4, 32, capacity=100, **a)
    n200 = kvc.store_bytes("uniform", 2, 4, 32, capacity=200, **a)
    assert n100 >= need and n100 % 256 == 0
    assert n200 >= 2 * need and n200 > n100
    # int8: D bytes + a 2-byte scale per token
    n = kvc.store_bytes("int8", 2, 4, 32, capacity=10)
    assert n >= 8 * 10 * (32 + 2)


@pytest.mark.parametrize("bad", [
    dict(mode="uniform", change=lambda a: a.update(bits=np.full_like(a["bits"], 5))),
    dict(mode="uniform", change=lambda a: a.update(qstep=np.zeros_like(a["qstep"]))),
    dict(mode="uniform", change=lambda a: a.update(basis_of=np.full(8, 7))),
    dict(mode="uniform", change=lambda a: a.update(V=np.full_like(a["V"], np.nan))),
    dict(mode="uniform", change=lambda a: a.update(capacity=0)),
    dict(mode="uniform", change=lambda a: a.update(heads_per_group=2, mean=None)),
    dict(mode="group", change=lambda a: a.update(bits=np.tile([2, 4, 4, 4, 2, 2, 2, 2], (3, 1)),
                                                 qmin=None, qstep=None)),
    dict(mode="group", change=lambda a: a.update(bits=np.tile([4, 4, 1, 1, 0, 0, 0, 0], (3, 1)),
                                                 qmin=None, qstep=None)),
    dict(mode="codebook", change=lambda a: a.update(codebook=[0.3, 0.1], mean=None, qmin=None,
                                                    qstep=None, bits=None)),
])
def test_bad_descriptors_are_rejected(kvc, bad):
    rng = np.random.default_rng(1)
    a = _uniform_args(rng)
    a["capacity"] = 16
    bad["change"](a)
    with pytest.raises(kvc.KvcError) as e:
        kvc.store_bytes(bad["mode"], 2, 4, 32, **a)
    assert e.value.status == -1


def test_null_layer_calls_fail_cleanly(kvc):
    lib = kvc.load_library()
    n = ctypes.c_int64()
    assert lib.kvc_trim(None, 3, ctypes.byref(n)) == -2
    assert lib.kvc_length(None, ctypes.byref(n)) == -2
    assert lib.kvc_append(None, None, 1, None) == -2
    assert lib.kvc_fetch(None, None, 1, None, None) == -2
    assert lib.kvc_set_wait_limit(None, 1000) == -2
    lib.kvc_destroy(None)
    assert b"NULL" in lib.kvc_last_error()


def test_init_without_device_memory_is_an_error(kvc):
    # A host buffer is never accepted as the store (CPU-only machines report a
    # CUDA error; machines with a GPU reject the host pointer).
    rng = np.random.default_rng(2)
    a = _uniform_args(rng)
    desc, keep = kvc._build_desc("uniform", 2, 4, 32, None, a["V"], a["mean"], a["bits"],
                                 a["qmin"], a["qstep"], a["basis_of"], 1, 32, None, "bf16",
                                 "f16", 16)
    n = ctypes.c_size_t()
    lib = kvc.load_library()
    assert lib.kvc_store_bytes(ctypes.byref(desc), ctypes.byref(n)) == 0
    host = (ctypes.c_uint8 * (n.value + 256))()
    addr = (ctypes.addressof(host) + 255) // 256 * 256
    desc.store = ctypes.c_void_p(addr)
    desc.store_bytes = n.value
    h = ctypes.c_void_p()
    st = lib.kvc_init_layer(ctypes.byref(desc), ctypes.byref(h))
    assert st in (-1, -4) and not h.value


def _fit_desc(kvc, **kw):
    a = dict(in_dtype=0, B=2, H=3, D=64, S_fit=16, stride_b=3 * 16 * 64, stride_h=16 * 64,
             stride_t=64, r=8, choices=(0, 2, 4), bit_budget=16)
    a.update(kw)
    ch = a.pop("choices")
    arr = (ctypes.c_int32 * max(len(ch), 1))(*ch)
    d = kvc._FitDesc(**a, bit_choices=arr, n_choices=len(ch))
    return d, arr


def test_fit_workspace_bytes_and_host_validation(kvc):
    """kvc_fit_uniform_workspace_bytes validates the descriptor on the host:
    float64 mean, two eigenvalue arrays, covariance and eigenvectors per slot,
    plus the DP table of (r + 1) x (budget + 1) entries (the budget clamped at
    max(choices) * r, beyond which the allocation no longer changes)."""
    lib = kvc.load_library()
    n = ctypes.c_size_t()
    d, keep = _fit_desc(kvc)
    assert lib.kvc_fit_uniform_workspace_bytes(ctypes.byref(d), ctypes.byref(n)) == 0
    al = lambda v: (v + 255) // 256 * 256  # noqa: E731
    ns, D, r, W = 6, 64, 8, 17
    assert n.value == 3 * al(ns * D * 8) + 2 * al(ns * D * D * 8) + al(ns * (r + 1) * W * 8)
    d, keep = _fit_desc(kvc, bit_budget=10_000)
    assert lib.kvc_fit_uniform_workspace_bytes(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value == 3 * al(ns * D * 8) + 2 * al(ns * D * D * 8) + al(ns * (r + 1) * 33 * 8)
    for bad in (dict(S_fit=1), dict(D=136), dict(D=60), dict(r=0), dict(r=65), dict(in_dtype=3),
                dict(choices=(5,)), dict(choices=()), dict(choices=(2, 4), bit_budget=15),
                dict(bit_budget=-1), dict(B=0)):
        d, keep = _fit_desc(kvc, **bad)
        assert lib.kvc_fit_uniform_workspace_bytes(ctypes.byref(d), ctypes.byref(n)) == -1, bad
    assert lib.kvc_fit_uniform_workspace_bytes(None, ctypes.byref(n)) == -1


def test_prod_descriptor_host_validation(kvc):
    """kvc_store_bytes_prod sizes rows [indices | sign bytes | outlier codes]
    and fp16 side words [norm, residual norm, outlier scale], and rejects bad
    sketch or outlier fields before anything touches a device."""
    lib = kvc.load_library()
    rng = np.random.default_rng(5)
    D, B, H, cap = 64, 1, 2, 10
    R = np.linalg.qr(rng.standard_normal((D, D)))[0].astype(np.float32)
    cb = np.array([-0.2, -0.05, 0.05, 0.2], dtype=np.float32)
    desc, keep = kvc._build_desc("codebook", B, H, D, None, R, None, None, None, None, None, 1,
                                 32, cb, "f16", "f16", cap)
    S = rng.standard_normal((32, D)).astype(np.float32)
    ch = np.array([[3, 9, 40], [0, 1, 63]], dtype=np.int32)

    def prod_desc(m=32, S=S, n_out=3, ch=ch, split=0):
        pd = kvc._ProdDesc()
        pd.m, pd.n_outliers, pd.split_from = m, n_out, split
        pd.S = S.ctypes.data_as(ctypes.POINTER(ctypes.c_float)) if S is not None else None
        pd.channels = ch.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if ch is not None else None
        return pd

    n = ctypes.c_size_t()
    pd = prod_desc()
    assert lib.kvc_store_bytes_prod(ctypes.byref(desc), ctypes.byref(pd), ctypes.byref(n)) == 0
    P = D * 2 // 8 + 32 // 8 + 3
    al = lambda v: (v + 255) // 256 * 256  # noqa: E731
    per_slot = al(cap * P + 16) + al(cap * 6 + 16)
    assert n.value == B * H * per_slot
    bad = [prod_desc(m=24), prod_desc(m=144), prod_desc(S=None), prod_desc(n_out=64),
           prod_desc(ch=np.array([[3, 3, 40], [0, 1, 63]], dtype=np.int32)),
           prod_desc(ch=np.array([[3, 9, 64], [0, 1, 63]], dtype=np.int32)), prod_desc(split=-1)]
    for pd in bad:
        assert lib.kvc_store_bytes_prod(ctypes.byref(desc), ctypes.byref(pd), ctypes.byref(n)) == -1
    assert lib.kvc_store_bytes_prod(ctypes.byref(desc), None, ctypes.byref(n)) == -1
    udesc, ukeep = kvc._build_desc("uniform", B, H, D, None, R[:, :8], None, np.full(8, 2),
                                   np.zeros(8), np.ones(8), None, 1, 32, None, "f16", "f16", cap)
    pd = prod_desc()
    assert lib.kvc_store_bytes_prod(ctypes.byref(udesc), ctypes.byref(pd), ctypes.byref(n)) == -1
