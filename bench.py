#!/usr/bin/env python3
"""Throughput of the projected-and-quantized KV cache hot path on GB300.

One step = for K and for V: empty the layer (kvc_trim), append the whole
context in one call (project + quantise + bit-pack), fetch it back
(unpack + dequantise + reconstruct to fp16 [B, H, S, D]).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload turboquant|llama3-8b|palu-group|kvtc-tiny|sweep]
                    [--path auto|generic] [--no-configs]
    python bench.py --sweep [--steps K]     # the Llama-3-70B-like grid, one line per point

Prints one JSON line (rank 0).  ``value`` is KV tokens per second over all
ranks, a KV token being one (batch, kv-head, position): its key row and its
value row are each appended and fetched once per step.  The default workload
is the largest single-GPU configuration, the TurboQuant-style one (B 16,
H_kv 8, S 16384: codebook keys, int8 values).  ``configs`` adds the other
configurations measured in the same run (the tiny KVTC-style case as
latencies, the Llama-3-8B-like and the PALU-style workloads, and the
one-token append).  Inputs are resident in HBM; L2 is flushed (a 256 MiB
write) between timed steps.  ``e2e`` times the same step through the public
API with the inputs copied from pinned host memory and the fetched rows
copied back, every step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV tokens/s for fetch (unpack+reconstruct) and append; % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}

WORKLOADS = {
    # TurboQuant-MSE-style: rotation + 3-bit codebook keys, int8 values
    "turboquant": dict(B=16, H=8, D=128, S=16384, mode="codebook", dtype="f16"),
    # Llama-3-8B-like decode layer: KVTC-style uniform mode, local PCA per (b, h)
    "llama3-8b": dict(B=8, H=8, D=128, S=4096, fit=512, r=32, choices=(0, 2, 4, 8),
                      budget=128, mode="uniform", dtype="bf16", alpha=1.0, seed=2000,
                      outliers=3),
    # PALU-style group-head mode: 4 groups of 8 heads (D_in = 1024 -> r = 256)
    "palu-group": dict(B=4, H=32, D=128, S=8192, hpg=8, r=256, mode="group", dtype="bf16"),
    # tiny KVTC-style correctness case: fp32, prefill 64 then 16 single-token appends
    "kvtc-tiny": dict(B=1, H=2, D=64, S=80, fit=64, r=16, choices=(0, 1, 2, 4, 8), budget=48,
                      mode="uniform", dtype="f32", alpha=0.8, seed=1000, outliers=0),
    # the TurboQuant workload with the prod quantiser's keys: b = 3 bits split as
    # 2-bit codebook indices plus a 128-row residual sketch, and 8 outlier
    # channels per (b, h) calibrated on the first 128 keys
    "turboquant-prod": dict(B=16, H=8, D=128, S=16384, mode="codebook", dtype="f16",
                            prod=dict(b_mse=2, m=128, n_out=8, n_calib=128)),
    # Llama-3-70B-like KV shape, uniform all-b allocation (one sweep point)
    "sweep": dict(B=8, H=8, D=128, S=8192, r=32, bits=4, mode="uniform", dtype="bf16"),
}
DEFAULT_WORKLOAD = "turboquant"


# Llama-3-70B-like KV throughput grid (H_kv = 8, D = 128): per rank r and
# uniform width, per batch and context, the fetch of the whole context and the
# append of one token; batch x context bounded by the fp16 output's bytes.
SWEEP = dict(H=8, D=128, B=(1, 8, 32, 64), S=(1024, 8192, 32768, 131072), r=(32, 64),
             bits=(2, 4), max_out_bytes=180e9, chunk=8192)


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.idx = gpu_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.p = None
        return self

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(", ") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# DRAM traffic (ncu dram__bytes_read.sum + dram__bytes_write.sum) per
# token-head of a kernel, from one capture of the kernel as it stands (the
# capture and its command are recorded with the ncu summaries); an entry is
# removed whenever its kernel changes.  The roofline's "traffic" scales it to
# the launch.
TRAFFIC_PER_UNIT = {
    # codebook append: 268.83 MB read + 39.68 MB written for 16 x 8 x 8192 token-heads
    ("append", "codebook"): (268.83e6 + 39.68e6) / (16 * 8 * 8192),
}


# ----------------------------------------------------------------------------- multi-rank

def max_over_ranks(values, dist=None, device="cpu"):
    """Each value's maximum over the ranks (a job takes as long as its slowest
    rank); the values unchanged on one rank."""
    if dist is None:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world, units_per_rank, ms):
    """Whole-job units per second: every rank processes units_per_rank (weak
    scaling replicas) in ms milliseconds."""
    return world * units_per_rank / (ms / 1e3)


# ----------------------------------------------------------------------------- GPU arm

def build_layers(wl, dev):
    """Synthetic inputs (seeded, generated on the GPU) and fitted layers for K and V."""
    import torch

    import rank_quantized_kv_gb300 as kvc
    import synth
    from rank_quantized_kv_gb300 import calib

    B, H, D, S = wl["B"], wl["H"], wl["D"], wl["S"]
    layers, inputs = [], []
    f32 = torch.float32
    for tensor in (0, 1):
        if wl["mode"] == "group":
            x = synth.group_spectral(B, H, S, D, wl["hpg"], alpha=1.0, seed=3000, tensor=tensor,
                                     n_outliers=20, dtype="bf16", device=dev, work_dtype=f32)
            params = calib.fit_group(x, wl["hpg"], wl["r"])
            L = kvc.KVCacheLayer("group", B, H, D, in_dtype="bf16", capacity=S, device=dev,
                                 **params)
        elif wl["mode"] == "codebook":
            pr = wl.get("prod")
            if tensor == 0 and pr:
                x = synth.heavy_tailed_keys(B, H, S, D, seed=4000, dtype="f16", device=dev)
                ch = kvc.fit_outliers(x, pr["n_calib"], pr["n_out"]).cpu().numpy()
                sketch = np.random.default_rng(1235).standard_normal((pr["m"], D)).astype(
                    np.float32)
                L = kvc.KVCacheLayer(
                    "codebook", B, H, D, in_dtype="f16", capacity=S, device=dev,
                    V=calib.rotation(D, 1234),
                    codebook=calib.gaussian_codebook(pr["b_mse"], 1 / math.sqrt(D)),
                    sketch=sketch, outlier_channels=ch, split_from=pr["n_calib"] - 1)
            elif tensor == 0:
                x = synth.heavy_tailed_keys(B, H, S, D, seed=4000, dtype="f16", device=dev)
                L = kvc.KVCacheLayer("codebook", B, H, D, in_dtype="f16", capacity=S, device=dev,
                                     V=calib.rotation(D, 1234),
                                     codebook=calib.gaussian_codebook(3, 1 / math.sqrt(D)))
            else:
                x = synth.kv_spectral(B, H, S, D, alpha=1.0, seed=4100, tensor=1, dtype="f16",
                                      device=dev, work_dtype=f32)
                L = kvc.KVCacheLayer("int8", B, H, D, in_dtype="f16", capacity=S, device=dev)
        else:
            fitted = "fit" in wl
            x = synth.kv_spectral(B, H, S, D, alpha=wl.get("alpha", 1.0),
                                  seed=wl.get("seed", 5000), tensor=tensor,
                                  n_outliers=wl.get("outliers", 0), dtype=wl["dtype"], device=dev,
                                  work_dtype=f32)
            if fitted:
                params = calib.fit_uniform(x[:, :, :wl["fit"]], wl["r"], wl["choices"],
                                           wl["budget"])
            else:
                params = calib.fit_uniform_shared(x[:, :, :min(S, 4096)], wl["r"], wl["bits"])
            L = kvc.KVCacheLayer("uniform", B, H, D, in_dtype=wl["dtype"], capacity=S,
                                 device=dev, **params)
        layers.append(L)
        inputs.append(x.contiguous())
    return layers, inputs


def algorithmic(wl, layers):
    """Per tensor: (fetch bytes, append bytes, flops) per full-context launch."""
    out = []
    B, H, D, S = wl["B"], wl["H"], wl["D"], wl["S"]
    for L in layers:
        n_slots = L.n_slots
        P = np.mean([L.slot_layout(s)["row_bytes"] for s in range(n_slots)])
        side = L.slot_layout(0)["side_bytes"]
        in_b = {"bf16": 2, "f16": 2, "f32": 4}[L.in_dtype]
        rows = n_slots * S
        d_in = L.hpg * D
        coded = rows * (P + side)
        fetch_b = coded + B * H * S * D * 2
        append_b = B * H * S * D * in_b + coded
        r = 0 if L.mode == "int8" else (D if L.mode == "codebook" else wl["r"])
        flops = 2.0 * rows * d_in * r
        out.append((fetch_b, append_b, flops))
    return out


def _event_ms(fn, reps, flush):
    """Mean CUDA-event time (ms) of fn() on the current stream, L2 flushed before each."""
    import torch

    total = 0.0
    for _ in range(reps):
        flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        total += e0.elapsed_time(e1)
    return total / reps


def launch_floor_us(flush, reps=50):
    """Event-timed launch of a trivial kernel: the floor under any one-launch latency."""
    tiny = flush[:16]
    tiny.zero_()
    return _event_ms(lambda: tiny.zero_(), reps, flush) * 1e3


def tensor_name(i, L):
    return ("keys" if i == 0 else "values") + f"/{L.mode}"


def time_steps(layers, inputs, outs, steps, flush):
    """K timed steps (trim, append S, fetch S per tensor): per-step ms and
    per-tensor summed append / fetch ms, all from CUDA events."""
    import torch

    nten = len(layers)
    step_ms, app_ms, fet_ms = [], np.zeros(nten), np.zeros(nten)
    for _ in range(steps):
        flush.fill_(1)                       # L2 flush, outside the timed events
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nten)]
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        for i, (L, x, o) in enumerate(zip(layers, inputs, outs)):
            L.trim(len(L))
            ev[i][0].record()
            L.append(x)
            ev[i][1].record()
            L.fetch(out=o)
            ev[i][2].record()
        s1.record()
        s1.synchronize()
        step_ms.append(s0.elapsed_time(s1))
        for i in range(nten):
            app_ms[i] += ev[i][0].elapsed_time(ev[i][1])
            fet_ms[i] += ev[i][1].elapsed_time(ev[i][2])
    return step_ms, app_ms, fet_ms


def op_table(wl, layers, app_ms, fet_ms, steps, peaks):
    """Per tensor: append / fetch time, tokens/s and roofline fraction."""
    B, H, S = wl["B"], wl["H"], wl["S"]
    hbm = peaks["hbm_gbs"] * 1e9
    tflops = peaks["bf16_tflops"] * 1e12
    alg = algorithmic(wl, layers)
    ops = {}
    for i, L in enumerate(layers):
        fb, ab, fl = alg[i]
        ta, tf = app_ms[i] / steps / 1e3, fet_ms[i] / steps / 1e3
        ops[tensor_name(i, L)] = {
            "append_us": ta * 1e6, "fetch_us": tf * 1e6,
            "append_tokens_per_s": B * H * S / ta, "fetch_tokens_per_s": B * H * S / tf,
            "append_roofline_frac": max(ab / hbm, fl / tflops) / ta,
            "fetch_roofline_frac": max(fb / hbm, fl / tflops) / tf,
            "append_bytes": ab, "fetch_bytes": fb, "flops": fl,
        }
    return ops


def attend_op(layers, flush, peaks, reps, rep=4):
    """Decode attention on the stored codes (kvc_attend): one query per
    (batch, query head), rep query heads per key/value head, over every
    stored token.  Bytes: the key and value rows and side words, read once."""
    import torch

    import rank_quantized_kv_gb300 as kvc

    K, V = layers
    dev = K.device
    q = torch.randn(K.B, K.H * rep, K.D, device=dev,
                    generator=torch.Generator(device=dev).manual_seed(11))
    out = torch.empty(K.B, K.H * rep, K.D, dtype=torch.float16, device=dev)
    ws = torch.empty(kvc.attend_workspace_bytes(K, V, K.H * rep), dtype=torch.uint8, device=dev)
    for _ in range(3):
        kvc.attend(K, V, q, out=out, workspace=ws)
    ms = _event_ms(lambda: kvc.attend(K, V, q, out=out, workspace=ws), reps, flush)
    S = len(K)
    nbytes = 0
    for L in layers:
        lay = L.slot_layout(0)
        nbytes += L.n_slots * S * (lay["row_bytes"] + lay["side_bytes"])
    t = ms / 1e3
    return {"us": ms * 1e3, "query_heads_per_kv_head": rep, "tokens": S,
            "kv_tokens_per_s": K.B * K.H * S / t, "bytes": nbytes,
            "roofline_frac": nbytes / (peaks["hbm_gbs"] * 1e9) / t,
            "what": "softmax(scale q . k_hat) v_hat from the codes, keys and values never "
                    "reconstructed"}


def extra_configs(dev, flush, peaks, steps):
    """The configurations beside the headline, measured in the same run: the
    tiny KVTC-style case (latencies: a 64-token prefill append, single-token
    appends, the fetch of all 80 tokens), the Llama-3-8B-like layer (bulk
    append and fetch, and the one-token decode append at S = 4096) and the
    PALU-style group workload (bulk append and fetch)."""
    import torch

    res = {"launch_floor_us": launch_floor_us(flush)}
    # tiny KVTC-style case, as latencies
    wl = WORKLOADS["kvtc-tiny"]
    layers, inputs = build_layers(wl, dev)
    tiny = {}
    for i, (L, x) in enumerate(zip(layers, inputs)):
        pre = x[:, :, :wl["fit"]].contiguous()
        one = [x[:, :, t:t + 1].contiguous() for t in range(wl["fit"], wl["S"])]
        out = torch.empty(wl["B"], wl["H"], wl["S"], wl["D"], dtype=torch.float16, device=dev)

        def prefill():
            L.trim(len(L))
            L.append(pre)

        def decode_all():
            L.trim(len(L) - wl["fit"])
            for xt in one:
                L.append(xt)

        for _ in range(3):
            prefill()
            decode_all()
            L.fetch(out=out)
        reps = max(5, min(steps, 50))
        t_pre = _event_ms(prefill, reps, flush)
        decode_all()
        t_dec = _event_ms(decode_all, reps, flush) / len(one)
        t_fet = _event_ms(lambda: L.fetch(out=out), reps, flush)
        if L.sync_status() != 0:
            raise RuntimeError("device error in the tiny case")
        tiny[tensor_name(i, L)] = {"prefill_append_64_us": t_pre * 1e3,
                                   "single_token_append_us": t_dec * 1e3,
                                   "fetch_80_us": t_fet * 1e3}
    res["kvtc-tiny"] = {"shape": "B 1, H 2, D 64, fp32, r 16, {0,1,2,4,8}, 48 bits",
                        "latency": tiny,
                        "note": "160 token-heads: launch-latency bound; compare with "
                                "launch_floor_us, not with a roofline"}
    del layers, inputs
    # Llama-3-8B-like layer and the PALU-style group workload, bulk
    for name in ("llama3-8b", "palu-group"):
        wl = WORKLOADS[name]
        layers, inputs = build_layers(wl, dev)
        outs = [torch.empty(wl["B"], wl["H"], wl["S"], wl["D"], dtype=torch.float16, device=dev)
                for _ in layers]
        time_steps(layers, inputs, outs, 3, flush)
        n = max(3, min(steps, 20))
        _, app_ms, fet_ms = time_steps(layers, inputs, outs, n, flush)
        entry = {"ops": op_table(wl, layers, app_ms, fet_ms, n, peaks), "steps": n}
        if name == "llama3-8b":
            one = []
            for L, x in zip(layers, inputs):
                x1 = x[:, :, :1]

                def append_one():
                    L.trim(1)
                    L.append(x1)

                one.append(_event_ms(append_one, n, flush) * 1e3)
            entry["one_token_append_us"] = {tensor_name(i, L): one[i]
                                            for i, L in enumerate(layers)}
            entry["one_token_note"] = ("one token appended to each of the 64 (b, h) at S = 4096: "
                                       "launch-latency bound, compare with launch_floor_us")
            import rank_quantized_kv_gb300 as kvc

            xf = inputs[0][:, :, :wl["fit"]]
            kvc.fit_uniform(xf, wl["fit"], wl["r"], wl["choices"], wl["budget"])
            fit_ms = _event_ms(lambda: kvc.fit_uniform(xf, wl["fit"], wl["r"], wl["choices"],
                                                       wl["budget"]), 3, flush)
            entry["prefill_fit_us"] = fit_ms * 1e3
            entry["prefill_fit_note"] = (
                "kvc_fit_uniform over the 64 (b, h) slots' first 512 key rows: covariance, "
                "Jacobi eigendecomposition, DP allocation and min/step in float64, four "
                "launches; once per layer before the hot path")
        for L in layers:
            if L.sync_status() != 0:
                raise RuntimeError(f"device error in {name}")
        res[name] = entry
        del layers, inputs, outs
        torch.cuda.empty_cache()
    res["turboquant-prod"] = prod_config(dev, flush, peaks, steps)
    return res


def prod_config(dev, flush, peaks, steps):
    """The TurboQuant workload with residual-sketch / outlier-stream keys: bulk
    append and fetch of both tensors, and decode attention on the codes.  The
    key kernels run on the CUDA cores: their roofline is the fp32 FMA rate
    (152 SMs x 128 lanes x 2 flops x the SM clock)."""
    import torch

    wl = WORKLOADS["turboquant-prod"]
    pr = wl["prod"]
    B, H, D, S = wl["B"], wl["H"], wl["D"], wl["S"]
    layers, inputs = build_layers(wl, dev)
    outs = [torch.empty(B, H, S, D, dtype=torch.float16, device=dev) for _ in layers]
    time_steps(layers, inputs, outs, 3, flush)
    n = max(3, min(steps, 20))
    _, app_ms, fet_ms = time_steps(layers, inputs, outs, n, flush)
    entry = {"ops": op_table(wl, layers, app_ms, fet_ms, n, peaks), "steps": n}
    sm_mhz = max((c for c in [peaks.get("sm_mhz")] if c), default=2070.0)
    alu = 152 * 128 * 2 * sm_mhz * 1e6
    tokens = B * H * S
    m = pr["m"]
    fl_app = 2.0 * tokens * (D * (128 + 128) + D * 128)   # x W1 (padded), c (S R)^T
    fl_fet = 2.0 * tokens * (D + m) * D                   # A [R^T ; S]
    ta, tf = app_ms[0] / n / 1e3, fet_ms[0] / n / 1e3
    entry["keys_alu"] = {
        "bound": "alu", "peak_tflops": alu / 1e12, "peak_source": "152 SMs x 128 fp32 lanes x 2 "
        "flops x SM clock", "append_flops": fl_app, "fetch_flops": fl_fet,
        "append_frac": fl_app / ta / alu, "fetch_frac": fl_fet / tf / alu}
    entry["attend"] = attend_op(layers, flush, peaks, reps=max(5, min(steps, 20)))
    for L in layers:
        if L.sync_status() != 0:
            raise RuntimeError("device error in turboquant-prod")
    entry["shape"] = (f"B {B}, H {H}, D {D}, S {S}; keys: 2-bit indices, {m}-row sketch, "
                      f"{pr['n_out']} outlier channels after {pr['n_calib']} keys; values int8")
    del layers, inputs, outs
    torch.cuda.empty_cache()
    return entry


def gpu_arm(args, rank, world):
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = dict(WORKLOADS[args.workload])
    if args.seq:
        wl["S"] = args.seq
    B, H, D, S = wl["B"], wl["H"], wl["D"], wl["S"]
    layers, inputs = build_layers(wl, dev)
    for L in layers:
        L.set_path(args.path)
    outs = [torch.empty(B, H, S, D, dtype=torch.float16, device=dev) for _ in layers]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    alg = algorithmic(wl, layers)

    time_steps(layers, inputs, outs, args.warmup, flush)
    torch.cuda.synchronize()
    for L in layers:
        if L.sync_status() != 0:
            raise RuntimeError("device error during warm-up")
        L.counters(reset=True)

    dist = None
    if world > 1:
        import torch.distributed as dist
    sampler = ClockSampler(dev.index).start() if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    step_ms, app_ms, fet_ms = time_steps(layers, inputs, outs, args.steps, flush)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    total_ms = float(np.sum(step_ms))
    counters = [L.counters() for L in layers]
    for L in layers:
        if L.sync_status() != 0:
            raise RuntimeError("device error in the timed region")
    total_ms, = max_over_ranks([total_ms], dist, dev)
    ms_per_step = total_ms / args.steps
    units = B * H * S                                   # KV tokens per step per rank
    value = job_throughput(world, units, ms_per_step)

    # e2e: pinned host inputs in, fetched rows out, every step
    hosts_in = [x.cpu().pin_memory() for x in inputs]
    hosts_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    h2d = sum(h.numel() * h.element_size() for h in hosts_in)
    d2h = sum(h.numel() * h.element_size() for h in hosts_out)
    e2e_steps = max(3, min(args.steps, 20))
    # Three streams: host->device copies, the library's calls, device->host
    # copies.  A tensor's upload waits for its previous use of the input buffer
    # to finish, its calls for its upload and for the previous download of its
    # output buffer, its download for its calls: uploads, compute and downloads
    # of different tensors (and steps) overlap on the full-duplex host link.
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nt = len(layers)
    up = [torch.cuda.Event() for _ in range(nt)]
    ran = [torch.cuda.Event() for _ in range(nt)]
    down = [torch.cuda.Event() for _ in range(nt)]

    def e2e_step():
        for i in range(nt):
            s_in.wait_event(ran[i])
            with torch.cuda.stream(s_in):
                inputs[i].copy_(hosts_in[i], non_blocking=True)
            up[i].record(s_in)
        for i, L in enumerate(layers):
            s_run.wait_event(up[i])
            s_run.wait_event(down[i])
            L.trim(len(L))
            L.append(inputs[i], stream=s_run)
            L.fetch(out=outs[i], stream=s_run)
            ran[i].record(s_run)
            s_out.wait_event(ran[i])
            with torch.cuda.stream(s_out):
                hosts_out[i].copy_(outs[i], non_blocking=True)
            down[i].record(s_out)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(dev)
    e0.record(cur)
    for sd in (s_in, s_run, s_out):
        sd.wait_event(e0)
    for _ in range(e2e_steps):
        e2e_step()
    for sd in (s_in, s_run, s_out):
        cur.wait_stream(sd)
    e1.record(cur)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms /= e2e_steps
    e2e_ms, = max_over_ranks([e2e_ms], dist, dev)
    del hosts_in, hosts_out
    if rank != 0:
        return None

    peaks = load_peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    tflops = peaks["bf16_tflops"] * 1e12
    ops = op_table(wl, layers, app_ms, fet_ms, args.steps, peaks)
    # dominant kernel: the op with the largest time per launch
    cand = []
    for i, L in enumerate(layers):
        fb, ab, fl = alg[i]
        cand.append((fet_ms[i], "fetch", i, fb, fl))
        cand.append((app_ms[i], "append", i, ab, fl))
    t_ms, kind, i, nbytes, fl = max(cand)
    t = t_ms / args.steps / 1e3
    tensor_bound = fl / tflops > nbytes / hbm
    roof = {
        "kernel": f"{kind} ({'keys' if i == 0 else 'values'}, {layers[i].mode})",
        "bound": "tensor" if tensor_bound else "hbm",
        "achieved": (fl / t / 1e12) if tensor_bound else (nbytes / t / 1e9),
        "peak": peaks["bf16_tflops"] if tensor_bound else peaks["hbm_gbs"],
        "unit": "TFLOP/s" if tensor_bound else "GB/s",
        "peak_source": peaks["source"],
        "traffic": None,
        "algorithmic_bytes_per_launch": nbytes,
        "launch_us": t * 1e6,
    }
    tr = TRAFFIC_PER_UNIT.get((kind, layers[i].mode))
    if tr is not None and not args.seq:
        roof["traffic"] = tr * layers[i].n_slots * S
    roof["frac"] = roof["achieved"] / roof["peak"]
    launches = sum(c["launches"] for c in counters)
    line = {
        "metric": METRIC, "value": value, "unit": "KV tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, **{k: v for k, v in wl.items() if k != "choices"},
                   "choices": list(wl.get("choices", [])), "path": args.path,
                   "parallelism": f"replicas{world}", "l2": "flushed between timed steps",
                   "step": "per tensor (K, V): trim all, append S tokens, fetch S tokens"},
        "e2e": {"value": job_throughput(world, units, e2e_ms), "unit": "KV tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": ("public API calls on one stream; the step's inputs uploaded from pinned "
                        "host memory and its fetched rows downloaded by torch copies on two "
                        "side streams, ordered by events and pipelined across steps")},
        "gpu_launches": launches,
        "roofline": roof,
        "ops": ops,
        "refined": {f"{'keys' if i == 0 else 'values'}": c for i, c in enumerate(counters)},
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    if len(layers) == 2 and layers[0].mode in ("uniform", "codebook") and \
            layers[1].mode in ("int8", "uniform"):
        line["attend"] = attend_op(layers, flush, peaks, max(3, min(args.steps, 50)))
    if not args.no_configs and world == 1 and not args.seq:
        line["configs"] = extra_configs(dev, flush, peaks, args.steps)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds,
                                            workload=None if args.seq else args.workload)
    return line


# ----------------------------------------------------------------------------- oracle legs

def _oracle_sample(wl, n_slots_sample):
    """Fitted oracle layers for K and V on a few slots of the workload (CPU, float64)."""
    import torch

    import synth
    from oracle import codec, fit
    from oracle.layer import OracleLayer

    D, S = wl["D"], wl["S"]
    jobs = []
    for tensor in (0, 1):
        if wl["mode"] == "group":
            hpg = wl["hpg"]
            x = synth.group_spectral(1, hpg, S, D, hpg, alpha=1.0, seed=3000, tensor=tensor,
                                     n_outliers=20, dtype="bf16")
            x64 = x.double().numpy()
            rows = np.concatenate(list(x64[0]), axis=1)
            mean, lam, U = fit.pca_fit(rows)
            bits = fit.palu_bits(wl["r"], 4, 2, 0.25)
            L = OracleLayer("group", 1, hpg, D, heads_per_group=hpg, V=U[:, :wl["r"]].astype(
                np.float32).astype(np.float64), mean=mean.astype(np.float32).astype(np.float64),
                bits=bits, group_size=32)
        elif wl["mode"] == "codebook":
            pr = wl.get("prod")
            if tensor == 0 and pr:
                from oracle import prod

                x = synth.heavy_tailed_keys(1, n_slots_sample, S, D, seed=4000, dtype="f16")
                x64 = x.double().numpy()
                ch = np.stack([prod.outlier_channels(x64[0, h, :pr["n_calib"]], pr["n_out"])
                               for h in range(n_slots_sample)])
                L = prod.ProdKeyLayer(
                    1, n_slots_sample, D, R=fit.seeded_rotation(D, 1234).astype(np.float32),
                    centroids=fit.lloyd_max_gaussian(1 << pr["b_mse"], 1 / math.sqrt(D)).astype(
                        np.float32),
                    S=np.random.default_rng(1235).standard_normal((pr["m"], D)).astype(np.float32),
                    channels=ch, split_from=pr["n_calib"] - 1)
            elif tensor == 0:
                x = synth.heavy_tailed_keys(1, n_slots_sample, S, D, seed=4000, dtype="f16")
                L = OracleLayer("codebook", 1, n_slots_sample, D,
                                V=fit.seeded_rotation(D, 1234).astype(np.float32),
                                codebook=fit.lloyd_max_gaussian(8, 1 / math.sqrt(D)).astype(
                                    np.float32))
            else:
                x = synth.kv_spectral(1, n_slots_sample, S, D, alpha=1.0, seed=4100, tensor=1,
                                      dtype="f16")
                L = OracleLayer("int8", 1, n_slots_sample, D)
            x64 = x.double().numpy()
        else:
            fit_len = wl.get("fit", min(S, 4096))
            x = synth.kv_spectral(1, n_slots_sample, S, D, alpha=wl.get("alpha", 1.0),
                                  seed=wl.get("seed", 5000), tensor=tensor,
                                  n_outliers=wl.get("outliers", 0), dtype=wl["dtype"])
            x64 = x.double().numpy()
            Vs, ms, bs, los, sts = [], [], [], [], []
            for h in range(n_slots_sample):
                mean, lam, U = fit.pca_fit(x64[0, h, :fit_len])
                V32 = U[:, :wl["r"]].astype(np.float32)
                m32 = mean.astype(np.float32)
                bits = (fit.dp_allocate(lam[:wl["r"]], wl["choices"], wl["budget"])
                        if "fit" in wl else np.full(wl["r"], wl["bits"]))
                lo, st = fit.uniform_params(codec.project(x64[0, h, :fit_len], m32, V32), bits)
                Vs.append(V32), ms.append(m32), bs.append(bits)
                los.append(lo.astype(np.float32)), sts.append(st.astype(np.float32))
            L = OracleLayer("uniform", 1, n_slots_sample, D, V=np.stack(Vs), mean=np.stack(ms),
                            bits=np.stack(bs), qmin=np.stack(los), qstep=np.stack(sts),
                            basis_of=np.arange(n_slots_sample))
        jobs.append((L, x64))
    return jobs


def _cores_used():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def _oracle_once(jobs):
    """Append then fetch every job's tokens; returns the KV tokens processed."""
    for L, x64 in jobs:
        L.trim(L.len)
        L.append(x64)
        L.fetch()
    x0 = jobs[0][1]
    return x0.shape[0] * x0.shape[1] * x0.shape[2]


def _oracle_rate(wl, budget_s):
    """KV tokens/s of the oracle, as it stands, on a bounded sample of the
    workload: (rate, seconds, KV heads sampled)."""
    n_sample = 2 if wl["mode"] != "group" else wl["hpg"]
    jobs = _oracle_sample(wl, n_sample)
    t0 = time.perf_counter()
    done = 0
    while True:
        done += _oracle_once(jobs)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, dt, n_sample


_ONE_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                   "VECLIB_MAXIMUM_THREADS": "1", "NUMEXPR_NUM_THREADS": "1",
                   "CUDA_VISIBLE_DEVICES": ""}


def _oracle_single_thread(workload, budget_s):
    """The same oracle timing in a child process whose BLAS and torch use one thread."""
    env = dict(os.environ, **_ONE_THREAD_ENV)
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-single-thread",
                          workload, "--cpu-seconds", str(budget_s)], env=env, capture_output=True,
                         text=True, timeout=600)
    if res.returncode:
        return {"error": res.stderr.strip().splitlines()[-1:] or ["failed"]}
    return json.loads(res.stdout.strip().splitlines()[-1])


def cpu_baseline(wl, budget_s=12.0, workload=None):
    """The float64 oracle, as it stands, on a bounded sample of the workload:
    on all host cores (BLAS threads) and on one thread."""
    rate, dt, n_sample = _oracle_rate(wl, budget_s / 2)
    sample = (f"{n_sample} of the workload's KV heads x {wl['S']} tokens (K and V), "
              f"appended and fetched repeatedly for {dt:.1f} s")
    out = {"value": rate, "unit": "KV tokens/s", "cores": _cores_used(), "kind": "oracle",
           "sample": sample, "host_cpus": os.cpu_count()}
    if workload is not None:
        out["single_thread"] = _oracle_single_thread(workload, budget_s / 2)
    return out


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    wl = WORKLOADS[args.workload]
    n_sample = 2 if wl["mode"] != "group" else wl["hpg"]
    jobs = _oracle_sample(wl, n_sample)
    for _ in range(args.warmup):
        _oracle_once(jobs)
    t0 = time.perf_counter()
    done = 0
    for _ in range(args.steps):
        done += _oracle_once(jobs)
    dt = time.perf_counter() - t0
    value = done / dt
    sample = f"{n_sample} KV heads x {wl['S']} tokens (K and V) per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "KV tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, **{k: v for k, v in wl.items() if k != "choices"},
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": "KV tokens/s", "cores": _cores_used(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "KV tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def _timed_ms(fn, reps, flush):
    """Mean CUDA-event time of fn() after two untimed calls, L2 flushed before each."""
    import torch

    fn()
    fn()
    total = 0.0
    for _ in range(reps):
        flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        total += e0.elapsed_time(e1)
    return total / reps


def sweep_arm(args):
    """The throughput grid: one JSON line per (r, bits, B, S), then a summary line.

    The cache of each point is filled with S tokens (appended in chunks of the
    same seeded rows); then the fetch of all S tokens and the append of one
    more token (after dropping the last, so the length stays S) are timed.
    """
    import torch

    import rank_quantized_kv_gb300 as kvc
    import synth
    from rank_quantized_kv_gb300 import calib

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    H, D, chunk = SWEEP["H"], SWEEP["D"], SWEEP["chunk"]
    reps = max(3, min(args.steps, 20))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    f32 = torch.float32
    x_fit = synth.kv_spectral(1, H, 4096, D, alpha=1.0, seed=5000, tensor=0, dtype="bf16",
                              device=dev, work_dtype=f32)
    src = synth.kv_spectral(1, H, chunk, D, alpha=1.0, seed=5001, tensor=0, dtype="bf16",
                            device=dev, work_dtype=f32)
    sampler = ClockSampler(dev.index).start()
    points = []
    for r in SWEEP["r"]:
        for bits in SWEEP["bits"]:
            params = calib.fit_uniform_shared(x_fit, r, bits)
            for B in SWEEP["B"]:
                xin = src.repeat(B, 1, 1, 1)
                params["basis_of"] = np.array([h for _ in range(B) for h in range(H)],
                                              dtype=np.int32)
                for S in SWEEP["S"]:
                    out_bytes = B * H * S * D * 2
                    if out_bytes > SWEEP["max_out_bytes"]:
                        continue
                    L = kvc.KVCacheLayer("uniform", B, H, D, in_dtype="bf16", capacity=S,
                                         device=dev, **params)
                    for c0 in range(0, S, chunk):
                        L.append(xin[:, :, :min(chunk, S - c0)])
                    out = torch.empty(B, H, S, D, dtype=torch.float16, device=dev)
                    fetch_ms = _timed_ms(lambda: L.fetch(out=out), reps, flush)
                    x1 = xin[:, :, :1]

                    def append_one():
                        L.trim(1)
                        L.append(x1)

                    app_ms = _timed_ms(append_one, reps, flush)
                    if L.sync_status() != 0:
                        raise RuntimeError(f"device error at r={r} bits={bits} B={B} S={S}")
                    P = L.slot_layout(0)["row_bytes"]
                    fetch_bytes = B * H * S * (P + D * 2)
                    fetch_flops = 2.0 * B * H * S * D * r
                    t_roof = max(fetch_bytes / (peaks["hbm_gbs"] * 1e9),
                                 fetch_flops / (peaks["bf16_tflops"] * 1e12))
                    line = {"r": r, "bits": bits, "B": B, "S": S, "row_bytes": P,
                            "fetch_us": fetch_ms * 1e3,
                            "fetch_tokens_per_s": B * H * S / (fetch_ms * 1e-3),
                            "fetch_gbs": fetch_bytes / (fetch_ms * 1e-3) / 1e9,
                            "fetch_roofline_frac": t_roof / (fetch_ms * 1e-3),
                            "append_one_us": app_ms * 1e3,
                            "append_one_bytes": B * H * (D * 2 + P)}
                    print(json.dumps(line), flush=True)
                    points.append(line)
                    del out
                    L.close()
                del xin
    clocks = sampler.stop()
    best = max(points, key=lambda q: q["fetch_roofline_frac"])
    big = [q for q in points if q["B"] * q["S"] >= 8 * 131072]
    print(json.dumps({
        "sweep": "llama3-70b-like kv grid", "points": len(points), "unit": "KV tokens/s",
        "peak_hbm_gbs": peaks["hbm_gbs"], "peak_source": peaks["source"],
        "fetch_roofline_frac_best": best["fetch_roofline_frac"],
        "best_point": {k: best[k] for k in ("r", "bits", "B", "S")},
        "fetch_roofline_frac_min_at_B_S_ge_1M": min((q["fetch_roofline_frac"] for q in big),
                                                     default=None),
        "append_one_us_range": [min(q["append_one_us"] for q in points),
                                max(q["append_one_us"] for q in points)],
        "l2": "flushed before every timed call", "clocks": clocks}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--path", choices=["auto", "generic"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--seq", type=int, default=0,
                    help="tokens per (b, h) instead of the workload's S (profiling captures)")
    ap.add_argument("--sweep", action="store_true",
                    help="the Llama-3-70B-like throughput grid (one GPU), one line per point")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations measured beside the headline")
    ap.add_argument("--oracle-single-thread", metavar="WORKLOAD", default=None,
                    help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_single_thread:
        # child of cpu_baseline: the oracle with one BLAS / torch thread, no GPU
        import torch

        torch.set_num_threads(1)
        rate, dt, n = _oracle_rate(WORKLOADS[args.oracle_single_thread], args.cpu_seconds)
        print(json.dumps({"value": rate, "unit": "KV tokens/s", "cores": 1,
                          "blas_threads_reported": _cores_used(), "seconds": dt,
                          "sample": f"{n} KV heads x {WORKLOADS[args.oracle_single_thread]['S']} "
                                    f"tokens (K and V), repeatedly for {dt:.1f} s"}))
        return
    if args.sweep:
        sweep_arm(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", args.gpus))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    line = reference_arm(args, rank, world) if args.impl == "reference" else gpu_arm(args, rank,
                                                                                     world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
