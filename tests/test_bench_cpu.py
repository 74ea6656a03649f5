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
