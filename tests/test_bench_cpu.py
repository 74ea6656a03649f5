"""bench.py's host logic on the CPU: workload selection, block options, roofline bytes."""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from transformer_mlp_gemms_gb300 import workloads as wl  # noqa: E402


def _args(**kw):
    a = types.SimpleNamespace(workload="siglip", block="", weights="in_out", h_path="memory", shape=None)
    a.__dict__.update(kw)
    return a


def test_kernel_bytes_count_each_operand_once():
    w = wl.WORKLOADS["siglip"]  # X 729x1152, W_up 1152x4304, W_down 4304x1152, f16, no bias
    x, h = 729 * 1152 * 2, 729 * 4304 * 2
    wu = wd = 1152 * 4304 * 2
    assert bench.kernel_bytes(w, "up", False) == x + wu + h
    assert bench.kernel_bytes(w, "down", False) == h + wd + x
    assert bench.kernel_bytes(w, "down", True) == h + wd + 2 * x           # the residual is read once
    assert bench.kernel_bytes(w, "fused", False) == x + wu + wd + x          # H never leaves the chip
    g = wl.WORKLOADS["sdxl_l2"]  # GEGLU: W_up is D x 2F, biases
    assert bench.kernel_bytes(g, "up", False) == (2048 * 1280 + 1280 * 10240 + 10240 + 2048 * 5120) * 2


def test_block_options_and_traffic_keys():
    assert bench.block_options(_args()) == (False, False, False)
    assert bench.block_options(_args(block="ln,res", weights="out_in")) == (True, True, True)
    with pytest.raises(SystemExit):
        bench.block_options(_args(block="ln,bogus"))
    w = wl.WORKLOADS["siglip"]
    assert bench.traffic_key(w, _args()) == "siglip"
    assert bench.traffic_key(w, _args(block="res", weights="out_in")) == "siglip[res,out_in]"
    assert bench.traffic_key(w, _args(h_path="on_chip")) == "siglip[h_on_chip]"


def test_custom_shape_workload():
    w = bench.pick_workload(_args(shape="40000,64,256,gelu_tanh,f16,0"))
    assert (w.M, w.D, w.F, w.act, w.dtype, w.bias) == (40000, 64, 256, wl.ACT_GELU_TANH, wl.DT_F16, False)
    assert bench.pick_workload(_args(workload="sdxl_l1")) is wl.WORKLOADS["sdxl_l1"]


def test_step_stats_and_clock_helpers():
    st = bench.step_stats([0.010, 0.020, 0.030, 0.040, 0.100])
    assert st["mean"] == pytest.approx(40.0) and st["median"] == pytest.approx(30.0)
    assert st["p90"] == pytest.approx(100.0) and st["min"] == pytest.approx(10.0) and st["steps"] == 5
    row = bench.parse_clock_line("0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active\n")
    assert row["sm"] == 2070.0 and row["power"] == 900.5 and row["sw_power_cap"] == "Active"
    assert bench.parse_clock_line("garbage") is None
    rows = [dict(row, t=1.0), dict(row, t=2.0, sm=1800.0), dict(row, t=3.0, sm=1810.0)]
    inside = bench.summarize_clocks(rows, window=(1.5, 3.5))
    assert inside["samples"] == 2 and inside["sm_mhz"] == pytest.approx(1805.0)
    assert inside["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks(rows, window=(5, 6))["samples"] == 0
    bins = bench.bin_by_clock([(0.5, 1.5, [0.02, 0.03]), (1.9, 2.1, [0.05]), (4, 5, [0.9])], rows)
    assert [(b["sm_mhz"], b["steps"]) for b in bins] == [(1800.0, 1), (2070.0, 2)]


def test_reference_arm_config_equals_the_gpu_arm_config():
    a = _args(launches="auto")
    w = wl.WORKLOADS["siglip"]
    assert bench.workload_config(w, bench.L2_LABEL, args=a) == bench.workload_config(w, bench.L2_LABEL, args=a)
    src = open(os.path.join(ROOT, "bench.py")).read()
    # both arms build their config with the same call
    assert src.count("workload_config(w, l2=L2_LABEL, args=args)") == 2
    assert set(bench.CONFIG_SUITE) <= set(wl.WORKLOADS)
