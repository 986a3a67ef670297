"""CPU checks of the bench's roofline arithmetic and of its clock record.

The algorithmic bytes per token-head (packed row + side words + the 16-bit
row the append reads or the fetch writes), the per-op fractions and the
traffic constant, with stand-in layers that report the TurboQuant-style slot
layouts: 3-bit codebook keys (48 B of codes and a 2 B fp16 norm per token-head)
and int8 values (128 B of codes and a 2 B fp16 scale).  The clock sampler's
parser is fed canned nvidia-smi rows.
"""
import pytest

import bench

WL = dict(B=16, H=8, D=128, S=16384, r=128)


class _Layer:
    def __init__(self, mode, row_bytes, side_bytes, in_dtype="f16"):
        self.mode, self.in_dtype, self.hpg = mode, in_dtype, 1
        self.n_slots = WL["B"] * WL["H"]
        self._lay = {"row_bytes": row_bytes, "side_bytes": side_bytes}

    def slot_layout(self, slot):
        return dict(self._lay)


def _layers():
    return [_Layer("codebook", 48, 2), _Layer("int8", 128, 2)]


def test_algorithmic_bytes_per_token_head():
    units = WL["B"] * WL["H"] * WL["S"]
    (kf, ka, kfl), (vf, va, vfl) = bench.algorithmic(WL, _layers())
    assert kf / units == 48 + 2 + 256 and ka / units == 256 + 48 + 2
    assert vf / units == 128 + 2 + 256 and va / units == 256 + 128 + 2
    assert kfl == 2.0 * units * 128 * 128        # the rotation, D x D per token-head
    assert vfl == 0.0


def test_op_fractions_are_bytes_over_time_over_peak():
    peaks = {"hbm_gbs": 6794.8, "bf16_tflops": 1899.0}
    steps = 20
    app_ms = [20 * 0.63226, 20 * 0.190]
    fet_ms = [20 * 0.14947, 20 * 0.11673]
    ops = bench.op_table(WL, _layers(), app_ms, fet_ms, steps, peaks)
    k, v = ops["keys/codebook"], ops["values/int8"]
    assert k["append_us"] == pytest.approx(632.26)
    # 641.7 MB in 632.26 us against the 6794.8 GB/s copy
    assert k["append_roofline_frac"] == pytest.approx(641728512 / 632.26e-6 / 6794.8e9)
    assert k["append_roofline_frac"] == pytest.approx(0.1494, abs=1e-4)
    assert v["fetch_roofline_frac"] == pytest.approx(809500672 / 116.73e-6 / 6794.8e9)
    assert k["append_tokens_per_s"] == pytest.approx(WL["B"] * WL["H"] * WL["S"] / 632.26e-6)
    # the rotation's flops stay far below the ridge: the bytes set the bound
    assert k["flops"] / (peaks["bf16_tflops"] * 1e12) < k["append_bytes"] / (peaks["hbm_gbs"] * 1e9)


def test_traffic_constant_is_near_the_algorithmic_bytes():
    # the capture's DRAM bytes per token-head against the 306 B the append
    # must move: below it only by the write-back still in L2 at capture end
    tr = bench.TRAFFIC_PER_UNIT[("append", "codebook")]
    assert 0.9 * 306 < tr < 1.02 * 306


def test_clock_sampler_reads_median_max_and_reasons():
    s = bench.ClockSampler(0)
    s.f.write("0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
              "0, 1980, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active\n"
              "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
              "garbage line\n")
    c = s.stop()                     # no sampler process was started: parse only
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_sampler_flags_thermal_slowdown():
    s = bench.ClockSampler(0)
    s.f.write("0, 1500, 2070, 1000.0, 0x40, Not Active, Active, Not Active, Not Active\n")
    c = s.stop()
    assert c["reasons"] == ["hw_thermal_slowdown"] and c["sm_mhz"] == 1500.0
