"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Every comparison is element by element (Y and the rounded H), at small shapes and at
the full workload sizes in the launch configuration the bench times: the oracle
computes every row (a few seconds per workload on the host cores), so every row
block of the one-launch work queue, of its readiness counters and of every split-K
reduction is checked.  Y and H buffers are poisoned with NaN before each run so that
an unwritten tile cannot pass.
"""
import re

import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_mlp_gemms_gb300 import kt_mlp
from transformer_mlp_gemms_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TDT = wl.TORCH_DTYPES


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_mlp_gemms_gb300 import build
    build.build()
    kt_mlp.load()


def _to_dev(t):
    return {k: v.cuda() for k, v in t.items()}


def _run(w, d, with_h=True, plan=None):
    own = plan is None
    if own:
        plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    Y = torch.full((w.M, w.D), float("nan"), dtype=TDT[w.dtype], device="cuda")
    H = torch.full((w.M, w.F), float("nan"), dtype=TDT[w.dtype], device="cuda") if with_h else None
    if with_h:
        plan.run_with_h(d["X"], d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Y, H)
    else:
        plan.run(d["X"], d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Y)
    torch.cuda.synchronize()
    assert plan.status() == kt_mlp.KT_OK, kt_mlp.kt_last_error()
    if own:
        plan.close()
    return Y.cpu(), (H.cpu() if with_h else None)


def _compare(w, t, Y, H, rows=None, what=""):
    b = {k: wl.bits(v) for k, v in t.items()}
    Ho, Yx, _ = oracle.mlp(b["X"], b["W_up"], b["W_down"], b.get("b_up"), b.get("b_down"),
                           act=w.act, dtype=w.dtype, rows=rows)
    yb = wl.bits(Y)
    if rows is not None:
        yb = yb[rows]
    parity.check_y(yb, Yx, w.dtype, what=f"Y {what}")
    if H is not None:
        hb = wl.bits(H)
        if rows is not None:
            hb = hb[rows]
        return parity.check_h(hb, Ho, parity.h_bound(w, b, rows), w.dtype, what=f"H {what}")


# --------------------------------------------------------------------------
# element by element on small shapes
# --------------------------------------------------------------------------

def test_tiny_workload():
    w = wl.WORKLOADS["tiny"]
    t = wl.generate(w)
    Y, H = _run(w, _to_dev(t))
    _compare(w, t, Y, H)


GRID = [
    # (M, D, F, act, dtype, bias)
    (1, 64, 64, wl.ACT_NONE, wl.DT_F16, False),
    (33, 64, 176, wl.ACT_NONE, wl.DT_F16, False),
    (128, 128, 256, wl.ACT_NONE, wl.DT_BF16, True),
    (129, 192, 320, wl.ACT_GELU_ERF, wl.DT_F16, True),
    (127, 64, 176, wl.ACT_GELU_TANH, wl.DT_F16, False),
    (300, 256, 1000, wl.ACT_GELU_TANH, wl.DT_BF16, False),
    (257, 1152, 4304, wl.ACT_GELU_TANH, wl.DT_F16, False),
    (64, 320, 640, wl.ACT_GEGLU, wl.DT_BF16, True),
    (200, 640, 2560, wl.ACT_GEGLU, wl.DT_BF16, True),
    (77, 128, 136, wl.ACT_GEGLU, wl.DT_F16, False),
    (5, 8, 8, wl.ACT_GELU_ERF, wl.DT_F16, True),
    (40, 24, 40, wl.ACT_GEGLU, wl.DT_BF16, True),
    (130, 72, 4104, wl.ACT_NONE, wl.DT_F16, True),
    (384, 1280, 512, wl.ACT_GELU_ERF, wl.DT_BF16, False),
]


@pytest.mark.parametrize("M,D,F,act,dt,bias", GRID)
def test_shape_grid(M, D, F, act, dt, bias):
    w = wl.custom(M, D, F, act, dt, bias, seed=1000 + M + D + F + act)
    t = wl.generate(w)
    Y, H = _run(w, _to_dev(t))
    _compare(w, t, Y, H)


# --------------------------------------------------------------------------
# full workload sizes, every element
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["siglip", "sdxl_l2", "sdxl_l1", "sweep_M256", "sweep_M1000", "sweep_M4096",
                                  "sweep_M16384"])
def test_full_size_workload_every_element(name):
    w = wl.WORKLOADS[name]
    t = wl.generate(w)
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    desc = plan.describe()
    Y, H = _run(w, _to_dev(t), plan=plan)
    plan.close()
    assert torch.isfinite(Y.float()).all(), "unwritten or non-finite Y"
    stats = _compare(w, t, Y, H, what=name)
    assert stats["elements"] == w.M * w.F, desc


@pytest.mark.parametrize("name", ["siglip", "sweep_M256", "sweep_M1000"])
@pytest.mark.parametrize("launches", [kt_mlp.KT_LAUNCH_ONE, kt_mlp.KT_LAUNCH_TWO])
def test_full_size_both_launch_modes_every_element(name, launches):
    # the small-M shapes in the launch mode the planner did not pick as well
    w = wl.WORKLOADS[name]
    t = wl.generate(w)
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias, launches=launches)
    assert plan.info()["one_launch"] == (launches == kt_mlp.KT_LAUNCH_ONE)
    Y, H = _run(w, _to_dev(t), plan=plan)
    plan.close()
    _compare(w, t, Y, H, what=f"{name} launches={launches}")


# --------------------------------------------------------------------------
# properties
# --------------------------------------------------------------------------

def test_runs_are_bitwise_deterministic_and_h_is_not_needed():
    w = wl.WORKLOADS["siglip"]
    t = wl.generate(w)
    d = _to_dev(t)
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    Y1, H1 = _run(w, d, with_h=True, plan=plan)
    Y2, _ = _run(w, d, with_h=False, plan=plan)
    Y3, _ = _run(w, d, with_h=False, plan=plan)
    plan.close()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    assert torch.equal(Y2.view(torch.int16), Y3.view(torch.int16))


@pytest.mark.parametrize("name", ["sdxl_l2", "siglip", "tiny"])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned_copy_kernels", "pageable_memcpy"])
def test_host_buffer_entry_point_matches_device_path(name, pinned):
    # pinned host buffers move through the copy kernels, pageable ones through
    # cudaMemcpyAsync; both calls twice in a row, bit-identical to the device path
    w = wl.WORKLOADS[name]
    t = wl.generate(w)
    d = _to_dev(t)
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    Yd, _ = _run(w, d, with_h=False, plan=plan)
    Xh = t["X"].pin_memory() if pinned else t["X"].clone()
    for _ in range(2):
        Yh = torch.full((w.M, w.D), float("nan"), dtype=TDT[w.dtype])
        if pinned:
            Yh = Yh.pin_memory()
        plan.run_host(Xh, d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Yh)
        assert plan.status() == kt_mlp.KT_OK
        assert torch.equal(Yd.view(torch.int16), Yh.view(torch.int16))
    plan.close()


def test_overflow_rounds_to_infinity_like_the_oracle():
    # fp16 H past 65504 must become +-inf (IEEE round to nearest), not saturate
    w = wl.custom(16, 64, 64, wl.ACT_NONE, wl.DT_F16, False, seed=7)
    t = wl.generate(w)
    t["W_up"] = (t["W_up"].float() * 40000.0).half()
    b = {k: wl.bits(v) for k, v in t.items()}
    Ho, _, _ = oracle.mlp(b["X"], b["W_up"], b["W_down"], act=w.act, dtype=w.dtype)
    assert np.isinf(oracle.decode(Ho, w.dtype)).any()
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    d = _to_dev(t)
    Y = torch.empty((w.M, w.D), dtype=torch.float16, device="cuda")
    H = torch.empty((w.M, w.F), dtype=torch.float16, device="cuda")
    plan.run_with_h(d["X"], d["W_up"], d["W_down"], None, None, Y, H)
    torch.cuda.synchronize()
    plan.close()
    hg = oracle.decode(wl.bits(H.cpu()), w.dtype)
    ho = oracle.decode(Ho, w.dtype)
    assert np.array_equal(np.isinf(hg), np.isinf(ho))
    assert np.array_equal(np.sign(hg[np.isinf(ho)]), np.sign(ho[np.isinf(ho)]))


def test_injected_stall_times_out_and_the_plan_recovers():
    w = wl.custom(256, 256, 512, wl.ACT_GELU_ERF, wl.DT_F16, False, seed=9)
    t = wl.generate(w)
    d = _to_dev(t)
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    kt_mlp.kt_mlp_debug_stall(plan.handle, True, 20000)  # 20 ms
    Y = torch.empty((w.M, w.D), dtype=torch.float16, device="cuda")
    plan.run(d["X"], d["W_up"], d["W_down"], None, None, Y)
    assert plan.status() == kt_mlp.KT_ERR_TIMEOUT
    assert "injected" in kt_mlp.kt_last_error()
    kt_mlp.kt_mlp_debug_stall(plan.handle, False, 0)
    Y2, H2 = _run(w, d, plan=plan)
    plan.close()
    _compare(w, t, Y2, H2)


def test_bad_pointers_are_rejected_before_launch():
    w = wl.custom(16, 64, 64, wl.ACT_GELU_ERF, wl.DT_F16, True, seed=3)
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    t = _to_dev(wl.generate(w))
    Y = torch.empty((w.M, w.D), dtype=torch.float16, device="cuda")
    with pytest.raises(kt_mlp.KtError) as e:
        plan.run(t["X"], t["W_up"], t["W_down"], None, None, Y)  # bias plan without biases
    assert e.value.status == kt_mlp.KT_ERR_INVALID
    with pytest.raises(kt_mlp.KtError) as e:
        plan.run(t["X"].data_ptr() + 2, t["W_up"], t["W_down"], t["b_up"], t["b_down"], Y)  # misaligned
    assert e.value.status == kt_mlp.KT_ERR_INVALID
    plan.close()


def test_plan_reports_its_choice():
    w = wl.WORKLOADS["siglip"]
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    info = plan.info()
    desc = plan.describe()
    plan.close()
    assert info["num_sms"] >= 148
    assert info["up"]["N"] == w.F and info["down"]["N"] == w.D
    assert re.search(r"up: (128|256)x\d+", desc) and re.search(r"down: (128|256)x\d+", desc)


ACTS = [wl.ACT_GELU_ERF, wl.ACT_GELU_TANH, wl.ACT_GEGLU, wl.ACT_GELU_SIGMOID, wl.ACT_SILU]


@pytest.mark.parametrize("form", [0, kt_mlp.KT_ACTIVATION_SCALAR_FORM], ids=["paired", "scalar"])
@pytest.mark.parametrize("act", ACTS)
def test_device_activation_accuracy(act, form):
    # the epilogue's fp32 activations against the float64 oracle on a dense grid:
    # relative error <= 2e-5, over 10x below half an fp16 ulp (2.4e-4)
    z = torch.linspace(-9.0, 9.0, 400001, dtype=torch.float32)
    g = torch.flip(z, [0]).contiguous()
    zd, gd = z.cuda(), g.cuda()
    out = torch.empty_like(zd)
    kt_mlp.kt_debug_activation(act | form, zd, gd, out, z.numel())
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    zz = z.double().numpy()
    if act == wl.ACT_GEGLU:
        ref = zz * oracle.gelu(g.double().numpy(), oracle.GELU_ERF)
    elif act in (wl.ACT_GELU_SIGMOID, wl.ACT_SILU):
        ref = oracle.gelu(zz, act)
    else:
        ref = oracle.gelu(zz, oracle.GELU_TANH if act == wl.ACT_GELU_TANH else oracle.GELU_ERF)
    big = np.abs(ref) > 1e-30
    rel = np.abs(got[big] - ref[big]) / np.abs(ref[big])
    assert rel.max() <= 2e-5, (float(rel.max()), float(zz[big][np.argmax(rel)]))
    assert np.all(np.abs(got[~big]) <= 1e-29)


@pytest.mark.parametrize("act", ACTS)
def test_paired_and_scalar_forms_agree_bit_for_bit(act):
    # the epilogues' paired fp32 instructions against the same steps as scalar
    # instructions, each rounded once either way: the bits must agree everywhere,
    # signed zeros, tiny, huge and odd-length tails included (an odd count leaves the
    # last element paired with itself)
    z = torch.cat([torch.linspace(-40.0, 40.0, 1000001, dtype=torch.float32),
                   torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e-40, -1e-40, 88.0, -88.0, 1e30, -1e30],
                                dtype=torch.float32)])
    g = torch.flip(z, [0]).contiguous()
    zd, gd = z.cuda(), g.cuda()
    outs = []
    for form in (0, kt_mlp.KT_ACTIVATION_SCALAR_FORM):
        out = torch.empty_like(zd)
        kt_mlp.kt_debug_activation(act | form, zd, gd, out, z.numel())
        outs.append(out.cpu().view(torch.int32))
    torch.cuda.synchronize()
    differ = (outs[0] != outs[1]).nonzero().flatten()
    assert differ.numel() == 0, (differ[:5].tolist(), z[differ[:5]].tolist())


def test_activation_rejects_unknown_form():
    z = torch.zeros(4, device="cuda")
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.kt_debug_activation(wl.ACT_GELU_TANH | 0x200, z, z, z, 4)
    assert e.value.status == kt_mlp.KT_ERR_INVALID
