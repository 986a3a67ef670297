"""GB300-native projected-and-quantized KV cache: Python binding of libkvc.

The binding only marshals arguments: every step of append and fetch runs in
the library's CUDA kernels.  PyTorch provides device memory and streams.
If libkvc.so is missing or cannot be loaded, every entry point raises; there
is no CPU fallback.

    layer = KVCacheLayer("uniform", B, H, D, V=V, mean=mean, bits=bits,
                         qmin=lo, qstep=step, in_dtype="bf16", capacity=S)
    layer.append(x)            # x: [B, H, T, D] on the layer's device
    k_hat = layer.fetch()      # [B, H, S, D] fp16
"""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import POINTER, byref, c_float, c_int32, c_int64, c_size_t, c_uint8, c_void_p

import numpy as np

__all__ = ["KVCacheLayer", "load_library", "library_path", "KvcError", "MODES", "DTYPES",
           "EXPORTED_SYMBOLS", "store_bytes", "attend", "attend_workspace_bytes", "fit_uniform",
           "fit_outliers"]

MODES = {"uniform": 0, "group": 1, "codebook": 2, "int8": 3}
DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
PATHS = {"auto": 0, "generic": 1}
STATUS = {0: "KVC_OK", -1: "KVC_EINVAL", -2: "KVC_ESTATE", -3: "KVC_ECAPACITY",
          -4: "KVC_ECUDA", -5: "KVC_ETIMEOUT", -6: "KVC_EDEVICE"}

# Every function include/kvc.h declares.
EXPORTED_SYMBOLS = (
    "kvc_abi_version", "kvc_last_error", "kvc_store_bytes", "kvc_init_layer", "kvc_append",
    "kvc_append_strided", "kvc_fetch", "kvc_trim", "kvc_length", "kvc_nbytes",
    "kvc_get_slot_layout", "kvc_set_path", "kvc_sync_status", "kvc_counters", "kvc_destroy",
    "kvc_append_noalloc", "kvc_set_wait_limit", "kvc_attend", "kvc_attend_workspace_bytes",
    "kvc_code_histogram_bytes", "kvc_code_histogram", "kvc_entropy_bytes",
    "kvc_fit_uniform_workspace_bytes", "kvc_fit_uniform", "kvc_store_bytes_prod",
    "kvc_init_layer_prod", "kvc_fit_outliers",
)

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.environ.get("KVC_LIBRARY", os.path.join(_HERE, "_lib", "libkvc.so"))


class KvcError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class _Entropy(ctypes.Structure):
    _fields_ = [("pre_entropy", c_int64), ("stored_payload", c_int64), ("params", c_int64),
                ("gain", ctypes.c_double)]


class _Desc(ctypes.Structure):
    _fields_ = [
        ("mode", c_int32), ("B", c_int32), ("H", c_int32), ("D", c_int32),
        ("heads_per_group", c_int32), ("r", c_int32), ("n_bases", c_int32),
        ("basis_of", POINTER(c_int32)), ("V", POINTER(c_float)), ("mean", POINTER(c_float)),
        ("bits", POINTER(c_uint8)), ("qmin", POINTER(c_float)), ("qstep", POINTER(c_float)),
        ("group_size", c_int32), ("codebook", POINTER(c_float)), ("cb_bits", c_int32),
        ("in_dtype", c_int32), ("out_dtype", c_int32), ("capacity", c_int64),
        ("store", c_void_p), ("store_bytes", c_size_t),
    ]


class _FitDesc(ctypes.Structure):
    _fields_ = [
        ("x", c_void_p), ("in_dtype", c_int32), ("B", c_int32), ("H", c_int32), ("D", c_int32),
        ("S_fit", c_int64), ("stride_b", c_int64), ("stride_h", c_int64), ("stride_t", c_int64),
        ("r", c_int32), ("bit_choices", POINTER(c_int32)), ("n_choices", c_int32),
        ("bit_budget", c_int32), ("V", c_void_p), ("mean", c_void_p), ("bits", c_void_p),
        ("qmin", c_void_p), ("qstep", c_void_p), ("lam", c_void_p),
    ]


class _ProdDesc(ctypes.Structure):
    _fields_ = [("m", c_int32), ("S", POINTER(c_float)), ("n_outliers", c_int32),
                ("channels", POINTER(c_int32)), ("split_from", c_int64)]


class _Bytes(ctypes.Structure):
    _fields_ = [("payload", c_int64), ("side", c_int64), ("fixed", c_int64),
                ("fp16_equiv", c_int64)]


class _SlotLayout(ctypes.Structure):
    _fields_ = [("payload_offset", c_int64), ("row_bytes", c_int64),
                ("side_offset", c_int64), ("side_bytes", c_int64)]


_lib = None
_lock = threading.Lock()


def load_library():
    """Load libkvc.so once; raises if it is missing (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"libkvc.so not found at {path}; build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        # Bind to the CUDA runtime torch already loaded (same libcudart.so.13),
        # so that torch's streams and allocations are this library's too.
        import torch  # noqa: F401

        lib = ctypes.CDLL(path)
        P = c_void_p
        sig = {
            "kvc_abi_version": (c_int32, []),
            "kvc_last_error": (ctypes.c_char_p, []),
            "kvc_store_bytes": (c_int32, [POINTER(_Desc), POINTER(c_size_t)]),
            "kvc_init_layer": (c_int32, [POINTER(_Desc), POINTER(c_void_p)]),
            "kvc_append": (c_int32, [P, P, c_int64, P]),
            "kvc_append_strided": (c_int32, [P, P, c_int64, c_int64, c_int64, c_int64, P]),
            "kvc_fetch": (c_int32, [P, P, c_int64, POINTER(c_int64), P]),
            "kvc_trim": (c_int32, [P, c_int64, POINTER(c_int64)]),
            "kvc_length": (c_int32, [P, POINTER(c_int64)]),
            "kvc_nbytes": (c_int32, [P, POINTER(_Bytes)]),
            "kvc_get_slot_layout": (c_int32, [P, c_int32, POINTER(_SlotLayout)]),
            "kvc_set_path": (c_int32, [P, c_int32]),
            "kvc_set_wait_limit": (c_int32, [P, c_int64]),
            "kvc_attend": (c_int32, [P, P, P, c_int32, ctypes.c_float, P, P, c_size_t, P]),
            "kvc_attend_workspace_bytes": (c_int32, [P, P, c_int32, POINTER(c_size_t)]),
            "kvc_code_histogram_bytes": (c_int32, [P, POINTER(c_size_t)]),
            "kvc_code_histogram": (c_int32, [P, P, c_size_t, P]),
            "kvc_entropy_bytes": (c_int32, [P, P, POINTER(_Entropy)]),
            "kvc_fit_uniform_workspace_bytes": (c_int32, [POINTER(_FitDesc), POINTER(c_size_t)]),
            "kvc_fit_uniform": (c_int32, [POINTER(_FitDesc), P, c_size_t, P]),
            "kvc_store_bytes_prod": (c_int32, [POINTER(_Desc), POINTER(_ProdDesc),
                                               POINTER(c_size_t)]),
            "kvc_init_layer_prod": (c_int32, [POINTER(_Desc), POINTER(_ProdDesc), POINTER(c_void_p)]),
            "kvc_fit_outliers": (c_int32, [P, c_int32, c_int32, c_int32, c_int32, c_int64, c_int64,
                                           c_int64, c_int64, c_int32, P, P]),
            "kvc_sync_status": (c_int32, [P, P]),
            "kvc_counters": (c_int32, [P, POINTER(c_int64), c_int32, P]),
            "kvc_destroy": (None, [P]),
            "kvc_append_noalloc": (c_int32, [POINTER(_Desc), c_int64, P, c_int64, c_int64,
                                             c_int64, c_int64, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if lib.kvc_abi_version() != 1:
            raise ImportError("libkvc ABI version mismatch")
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        raise KvcError(status, _lib.kvc_last_error().decode())


def _f32(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    if shape is not None:
        a = a.reshape(shape)
    return a


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(POINTER(ctype))


def _build_desc(mode, B, H, D, r, V, mean, bits, qmin, qstep, basis_of, heads_per_group,
                group_size, codebook, in_dtype, out_dtype, capacity):
    """Marshal arguments into a descriptor; returns (desc, keepalive arrays)."""
    if mode not in MODES:
        raise ValueError(f"mode must be one of {list(MODES)}")
    d_in = heads_per_group * D
    keep = {}
    desc = _Desc()
    desc.mode = MODES[mode]
    desc.B, desc.H, desc.D = B, H, D
    desc.heads_per_group = heads_per_group
    desc.in_dtype = DTYPES[in_dtype]
    desc.out_dtype = DTYPES[out_dtype]
    desc.capacity = int(capacity)
    desc.group_size = int(group_size)
    if mode != "int8":
        Vn = np.asarray(V, dtype=np.float32)
        if Vn.ndim == 2:
            Vn = Vn[None]
        nb, rows, rr = Vn.shape
        if r is not None and r != rr:
            raise ValueError("r disagrees with V")
        keep["V"] = np.ascontiguousarray(Vn)
        desc.r, desc.n_bases = rr, nb
        desc.V = _ptr(keep["V"], c_float)
        if mean is not None:
            keep["mean"] = _f32(mean, (nb, d_in))
            desc.mean = _ptr(keep["mean"], c_float)
        if bits is not None:
            keep["bits"] = np.ascontiguousarray(np.asarray(bits, dtype=np.uint8).reshape(nb, rr))
            desc.bits = _ptr(keep["bits"], c_uint8)
        if qmin is not None:
            keep["qmin"] = _f32(qmin, (nb, rr))
            keep["qstep"] = _f32(qstep, (nb, rr))
            desc.qmin = _ptr(keep["qmin"], c_float)
            desc.qstep = _ptr(keep["qstep"], c_float)
        if basis_of is not None:
            keep["basis_of"] = np.ascontiguousarray(np.asarray(basis_of, dtype=np.int32))
            desc.basis_of = _ptr(keep["basis_of"], c_int32)
        if codebook is not None:
            keep["codebook"] = _f32(codebook)
            desc.codebook = _ptr(keep["codebook"], c_float)
            desc.cb_bits = int(round(np.log2(keep["codebook"].shape[0])))
    return desc, keep


def store_bytes(mode, B, H, D, *, capacity, r=None, V=None, bits=None, qmin=None, qstep=None,
                basis_of=None, heads_per_group=1, group_size=32, codebook=None,
                in_dtype="bf16", out_dtype="f16", mean=None) -> int:
    """Bytes of device store a layer with these parameters needs."""
    lib = load_library()
    desc, keep = _build_desc(mode, B, H, D, r, V, mean, bits, qmin, qstep, basis_of,
                             heads_per_group, group_size, codebook, in_dtype, out_dtype, capacity)
    n = c_size_t()
    _check(lib.kvc_store_bytes(byref(desc), byref(n)))
    return int(n.value)


def _stream_ptr(stream, device):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return c_void_p(stream.cuda_stream)


_TORCH_DT = None


def _torch_dtypes():
    global _TORCH_DT
    if _TORCH_DT is None:
        import torch

        _TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
    return _TORCH_DT


class KVCacheLayer:
    """One K or V tensor of one attention layer, stored projected and quantised.

    mode: "uniform" (KVTC-style), "group" (PALU-style), "codebook"
    (TurboQuant-MSE-style) or "int8" (per-token int8 values).  Parameters are
    host arrays (numpy or CPU tensors) with the shapes of include/kvc.h; the
    store is a torch uint8 tensor on ``device`` owned by this object.
    """

    def __init__(self, mode, B, H, D, *, capacity, r=None, V=None, mean=None, bits=None,
                 qmin=None, qstep=None, basis_of=None, heads_per_group=1, group_size=32,
                 codebook=None, in_dtype="bf16", out_dtype="f16", device=None, path="auto",
                 sketch=None, outlier_channels=None, split_from=0):
        import torch

        lib = load_library()
        self.mode, self.B, self.H, self.D = mode, B, H, D
        self.hpg = heads_per_group
        self.Hg = H // heads_per_group
        self.n_slots = B * self.Hg
        self.in_dtype, self.out_dtype = in_dtype, out_dtype
        self.device = torch.device(device if device is not None else "cuda")
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.capacity = int(capacity)
        desc, keep = _build_desc(mode, B, H, D, r, V, mean, bits, qmin, qstep, basis_of,
                                 heads_per_group, group_size, codebook, in_dtype, out_dtype,
                                 capacity)
        # codebook keys with a residual sketch S [m, D] and/or outlier channels
        # [B*H, n_outliers] (kvc_init_layer_prod)
        self.prod = sketch is not None or outlier_channels is not None
        pd = None
        if self.prod:
            pd = _ProdDesc()
            if sketch is not None:
                keep["S"] = _f32(sketch)
                pd.m = keep["S"].shape[0]
                pd.S = _ptr(keep["S"], c_float)
            if outlier_channels is not None:
                keep["channels"] = np.ascontiguousarray(np.asarray(outlier_channels, dtype=np.int32))
                pd.n_outliers = keep["channels"].shape[-1]
                pd.channels = _ptr(keep["channels"], c_int32)
            pd.split_from = int(split_from)
        n = c_size_t()
        if pd is None:
            _check(lib.kvc_store_bytes(byref(desc), byref(n)))
        else:
            _check(lib.kvc_store_bytes_prod(byref(desc), byref(pd), byref(n)))
        self.store = torch.zeros(int(n.value), dtype=torch.uint8, device=self.device)
        desc.store = c_void_p(self.store.data_ptr())
        desc.store_bytes = n.value
        handle = c_void_p()
        with torch.cuda.device(self.device):
            if pd is None:
                _check(lib.kvc_init_layer(byref(desc), byref(handle)))
            else:
                _check(lib.kvc_init_layer_prod(byref(desc), byref(pd), byref(handle)))
        self._h = handle
        self._lib = lib
        self.set_path(path)

    # -- hot path ------------------------------------------------------------------------
    def append(self, x, stream=None):
        """Append x [B, H, T, D] (device tensor of in_dtype; last dim contiguous)."""
        if x.dim() != 4 or x.shape[0] != self.B or x.shape[1] != self.H or x.shape[3] != self.D:
            raise ValueError(f"x must be [{self.B}, {self.H}, T, {self.D}], got {tuple(x.shape)}")
        if x.dtype != _torch_dtypes()[self.in_dtype]:
            raise TypeError(f"x must be {self.in_dtype}")
        if x.shape[2] and x.stride(3) != 1:
            raise ValueError("the head dimension of x must be contiguous")
        sb, sh, st, _ = x.stride()
        _check(self._lib.kvc_append_strided(self._h, c_void_p(x.data_ptr()), x.shape[2], sb, sh,
                                            st, _stream_ptr(stream, self.device)))

    def fetch(self, out=None, stream=None):
        """Reconstruct everything stored into out [B, H, ld_s, D] (allocated if None)."""
        import torch

        S = len(self)
        if out is None:
            out = torch.empty(self.B, self.H, S, self.D, dtype=_torch_dtypes()[self.out_dtype],
                              device=self.device)
        if out.dtype != _torch_dtypes()[self.out_dtype] or not out.is_contiguous():
            raise ValueError("out must be a contiguous tensor of out_dtype")
        if out.shape[0] != self.B or out.shape[1] != self.H or out.shape[3] != self.D:
            raise ValueError("out must be [B, H, ld_s, D]")
        s_out = c_int64()
        _check(self._lib.kvc_fetch(self._h, c_void_p(out.data_ptr()), out.shape[2], byref(s_out),
                                   _stream_ptr(stream, self.device)))
        return out

    # -- state -----------------------------------------------------------------------------
    def trim(self, n: int) -> int:
        d = c_int64()
        _check(self._lib.kvc_trim(self._h, int(n), byref(d)))
        return int(d.value)

    def __len__(self) -> int:
        n = c_int64()
        _check(self._lib.kvc_length(self._h, byref(n)))
        return int(n.value)

    def nbytes(self) -> dict:
        b = _Bytes()
        _check(self._lib.kvc_nbytes(self._h, byref(b)))
        return {"payload": b.payload, "side": b.side, "fixed": b.fixed, "fp16_equiv": b.fp16_equiv}

    def slot_layout(self, slot: int) -> dict:
        s = _SlotLayout()
        _check(self._lib.kvc_get_slot_layout(self._h, int(slot), byref(s)))
        return {"payload_offset": s.payload_offset, "row_bytes": s.row_bytes,
                "side_offset": s.side_offset, "side_bytes": s.side_bytes}

    def slot_rows(self, slot: int):
        """Views into the store: (packed rows [len, P] uint8, side words [len, side_bytes] or None)."""
        lay = self.slot_layout(slot)
        n = len(self)
        P, o = lay["row_bytes"], lay["payload_offset"]
        rows = self.store[o:o + n * P].view(n, P)
        side = None
        if lay["side_bytes"]:
            so, sb = lay["side_offset"], lay["side_bytes"]
            side = self.store[so:so + n * sb].view(n, sb)
        return rows, side

    def set_path(self, path: str):
        _check(self._lib.kvc_set_path(self._h, PATHS[path]))

    def code_histogram(self, stream=None):
        """Per (slot, packed position, code value) counts of the stored codes,
        a device uint32 tensor [n_slots, NC, 256] (kvc_code_histogram)."""
        import torch

        n = c_size_t()
        _check(self._lib.kvc_code_histogram_bytes(self._h, byref(n)))
        counts = torch.empty(int(n.value) // 4, dtype=torch.int32, device=self.device)
        _check(self._lib.kvc_code_histogram(self._h, c_void_p(counts.data_ptr()), n.value,
                                            _stream_ptr(stream, self.device)))
        return counts.view(self.n_slots, -1, 256)

    def entropy_bytes(self, stream=None) -> dict:
        """Order-0 Huffman accounting of the stored codes (kvc_entropy_bytes)."""
        import torch

        counts = self.code_histogram(stream).cpu().contiguous()
        e = _Entropy()
        _check(self._lib.kvc_entropy_bytes(self._h, c_void_p(counts.data_ptr()), byref(e)))
        return {"pre_entropy": e.pre_entropy, "stored_payload": e.stored_payload,
                "params": e.params, "gain": e.gain}

    def set_wait_limit(self, ns: int):
        """Limit (ns) of the append kernel's waits; 0 restores the default (2 s)."""
        _check(self._lib.kvc_set_wait_limit(self._h, int(ns)))

    def sync_status(self, stream=None) -> int:
        """Synchronise and return the device status (0 = ok); clears it."""
        return int(self._lib.kvc_sync_status(self._h, _stream_ptr(stream, self.device)))

    def counters(self, reset=False, stream=None):
        out = (c_int64 * 6)()
        _check(self._lib.kvc_counters(self._h, out, int(bool(reset)),
                                      _stream_ptr(stream, self.device)))
        return {"refined_codes": out[0], "refined_side": out[1], "appended": out[2],
                "launches": out[3], "max_error_ratio": out[4] / 1e6}

    def close(self):
        if getattr(self, "_h", None):
            self._lib.kvc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def attend_workspace_bytes(keys: "KVCacheLayer", values: "KVCacheLayer", Hq: int) -> int:
    """Device workspace bytes kvc_attend needs at the layers' current length."""
    n = c_size_t()
    _check(load_library().kvc_attend_workspace_bytes(keys._h, values._h, int(Hq), byref(n)))
    return int(n.value)


def attend(keys: "KVCacheLayer", values: "KVCacheLayer", q, scale: float = 0.0, out=None,
           workspace=None, stream=None):
    """Decode attention on the stored codes: q [B, Hq, D] fp32 (device) over
    every stored token of ``keys`` and ``values`` (kvc_attend).  Returns out
    [B, Hq, D] in the value layer's out_dtype; the workspace (device bytes) is
    allocated when not given."""
    import torch

    lib = load_library()
    if q.dtype != torch.float32 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be a contiguous fp32 [B, Hq, D] tensor")
    Hq = q.shape[1]
    n = c_size_t()
    _check(lib.kvc_attend_workspace_bytes(keys._h, values._h, Hq, byref(n)))
    if workspace is None:
        workspace = torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=_torch_dtypes()[values.out_dtype], device=q.device)
    _check(lib.kvc_attend(keys._h, values._h, c_void_p(q.data_ptr()), Hq, float(scale),
                          c_void_p(out.data_ptr()), c_void_p(workspace.data_ptr()),
                          workspace.numel() * workspace.element_size(),
                          _stream_ptr(stream, q.device)))
    return out


def fit_uniform(x, S_fit: int, r: int, choices, budget: int, stream=None):
    """On-device prefill fit of the uniform mode (kvc_fit_uniform): per (b, h)
    of x [B, H, T, D] (device; fp32, fp16 or bf16; last dimension contiguous),
    over its first S_fit rows: the local PCA, the DP bit allocation and the
    frozen minimum and step.  Returns a dict of device tensors V [B*H, D, r]
    fp32, mean [B*H, D] fp32, bits [B*H, r] uint8, qmin and qstep [B*H, r]
    fp32 and lam [B*H, D] float64 (the sorted eigenvalues); V, mean, bits,
    qmin and qstep are the uniform layer's parameters with one basis per slot."""
    import torch

    lib = load_library()
    rev = {v: k for k, v in _torch_dtypes().items()}
    if x.dim() != 4 or x.dtype not in rev or x.stride(3) != 1:
        raise ValueError("x must be [B, H, T, D] fp32/fp16/bf16 with a contiguous last dimension")
    B, H, T, D = x.shape
    if S_fit > T:
        raise ValueError("S_fit exceeds the rows of x")
    # outputs on x's GPU; rows in host memory reach the library, which rejects them
    dev = x.device if x.is_cuda else torch.device("cuda", torch.cuda.current_device())
    ns = B * H
    out = dict(V=torch.empty(ns, D, r, dtype=torch.float32, device=dev),
               mean=torch.empty(ns, D, dtype=torch.float32, device=dev),
               bits=torch.empty(ns, r, dtype=torch.uint8, device=dev),
               qmin=torch.empty(ns, r, dtype=torch.float32, device=dev),
               qstep=torch.empty(ns, r, dtype=torch.float32, device=dev),
               lam=torch.empty(ns, D, dtype=torch.float64, device=dev))
    ch = (c_int32 * len(choices))(*[int(c) for c in choices])
    d = _FitDesc(x=x.data_ptr(), in_dtype=DTYPES[rev[x.dtype]], B=B, H=H, D=D, S_fit=int(S_fit),
                 stride_b=x.stride(0), stride_h=x.stride(1), stride_t=x.stride(2), r=int(r),
                 bit_choices=ch, n_choices=len(choices), bit_budget=int(budget),
                 V=out["V"].data_ptr(), mean=out["mean"].data_ptr(), bits=out["bits"].data_ptr(),
                 qmin=out["qmin"].data_ptr(), qstep=out["qstep"].data_ptr(),
                 lam=out["lam"].data_ptr())
    n = c_size_t()
    _check(lib.kvc_fit_uniform_workspace_bytes(byref(d), byref(n)))
    ws = torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib.kvc_fit_uniform(byref(d), c_void_p(ws.data_ptr()), int(n.value),
                                   _stream_ptr(stream, dev)))
    out["workspace"] = ws  # kept alive until the caller synchronises
    return out


def fit_outliers(x, n_calib: int, n_outliers: int, stream=None):
    """Outlier channels of every (b, h) from the first n_calib rows of x
    [B, H, T, D] (kvc_fit_outliers): device int32 [B*H, n_outliers], the
    channels of largest mean |x| in ascending order."""
    import torch

    lib = load_library()
    rev = {v: k for k, v in _torch_dtypes().items()}
    if x.dim() != 4 or x.dtype not in rev or (x.shape[2] and x.stride(3) != 1):
        raise ValueError("x must be [B, H, T, D] fp32/fp16/bf16 with a contiguous last dimension")
    B, H, T, D = x.shape
    dev = x.device if x.is_cuda else torch.device("cuda", torch.cuda.current_device())
    out = torch.empty(B * H, n_outliers, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.kvc_fit_outliers(c_void_p(x.data_ptr()), DTYPES[rev[x.dtype]], B, H, D,
                                    int(n_calib), x.stride(0), x.stride(1), x.stride(2),
                                    int(n_outliers), c_void_p(out.data_ptr()),
                                    _stream_ptr(stream, dev)))
    return out
