"""The benchmark's host-side bookkeeping on CPU: the clock record binned against
the timed region, exponentials per second, the e4m3 peak and input helpers."""
import math

import bench
from tiled_attention_fwd_gb300.inputs import WORKLOADS


def _row(sm, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if n in reasons else "Not Active" for n in names]
    return f"0, {sm}, 2070, 900.0, 0x0, " + ", ".join(flags) + "\n"


def test_clock_summary_bins_samples_against_the_windows():
    c = bench.ClockSampler(0)
    c.proc = object()  # pretend nvidia-smi ran; summary() only reads the stamped samples
    c.samples = [(0.5, _row(1500)),                        # before the load window: ignored
                 (1.1, _row(2070)), (1.2, _row(2055, ["sw_power_cap"])),
                 (1.305, _row(2040)),                      # inside the timed region
                 (1.4, _row(2070)),
                 (2.5, _row(900, ["hw_slowdown"]))]        # after the load window: ignored
    c.marks = {"load_start": 1.0, "timed_start": 1.30, "timed_end": 1.31, "load_end": 1.5}
    s = c.summary()
    assert s["samples"] == 4 and s["samples_in_timed_region"] == 1
    assert s["sm_mhz"] == (2055 + 2070) / 2 and s["sm_mhz_timed_region"] == 2040
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070
    assert abs(s["timed_region_s"] - 0.01) < 1e-12 and abs(s["load_window_s"] - 0.5) < 1e-12


def test_clock_summary_without_nvidia_smi():
    s = bench.ClockSampler(0).summary()
    assert s["sm_mhz"] is None and s["reasons"] == ["nvidia-smi unavailable"]


def test_exponentials_per_second():
    w = WORKLOADS["bf16_b4h16n4096d128_causal"]
    e = bench.exp_rate(w, 0.2, 152, 2070.0)
    assert e["per_launch"] == 4 * 16 * 4096 * 4096 / 2
    assert math.isclose(e["per_s"], e["per_launch"] / 2e-4)
    assert math.isclose(e["peak_per_s"], 32 * 152 * 2070e6)
    assert math.isclose(e["frac"], e["per_s"] / e["peak_per_s"])
    w = WORKLOADS["bf16_b2h16n8192d32_qk3"]  # no mask: every score
    assert bench.exp_rate(w, 1.0, 152, None)["per_launch"] == 2 * 16 * 8192 * 8192


def test_e4m3_inputs_and_bytes():
    w = WORKLOADS["fp8_b4h16n4096d128_causal"]
    n = 4 * 16 * 4096 * 128
    assert w.elem_bytes == 1 and w.io_bytes == 3 * n + 2 * n + 4 * 16 * 4096 * 4
    assert w.flops == WORKLOADS["bf16_b4h16n4096d128_causal"].flops
    assert bench.FP8_OVER_BF16 == 2.0
    small = w.with_(name="fp8_small", B=1, H=2, N=64)
    (q8, k8, v8), f = bench.workload_inputs(small)
    real = bench.oracle_inputs(small, (q8, k8, v8), f)
    for x8, fx, r in zip((q8, k8, v8), f, real):
        assert (x8.float() * fx == r).all()
    qkv, none = bench.workload_inputs(WORKLOADS["f32_b1h1n128d16"])
    assert none is None and bench.oracle_inputs(WORKLOADS["f32_b1h1n128d16"], qkv, None) is qkv
