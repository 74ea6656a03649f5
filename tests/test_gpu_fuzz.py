"""Seeded random problems through every option of the C ABI, against the oracle.

Each case draws a shape (M up to 4096, D and F multiples of 8 up to 1280 / 3000), an
activation, a dtype, biases, the block options (LayerNorm, residual), the weight order
and the H path (the planner's choice or H through memory), runs kt_mlp_plan_ex /
kt_mlp_run_ex, and compares every element of Y, and of the rounded H where the plan
writes H (H through memory), with the float64 oracle.  The planner picks its own tiles for each shape, so the cases reach tile
modes (CTA pairs, BK, split-K kinds, the fused kernel) that no hand-written case pins.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_mlp_gemms_gb300 import kt_mlp
from transformer_mlp_gemms_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

EPS = 1e-5
N_CASES = 48


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_mlp_gemms_gb300 import build
    build.build()
    kt_mlp.load()


def _case(i):
    rng = np.random.default_rng(9000 + i)
    M = int(rng.choice([1, 7, 33, 128, 129, 255, 300, 511, 700, 1024, 2100, 4096]))
    D = int(8 * rng.integers(1, 161))
    F = int(8 * rng.integers(1, 376))
    act = int(rng.integers(0, 6))
    dt = int(rng.integers(0, 2))
    bias = bool(rng.integers(0, 2))
    res = bool(rng.integers(0, 2))
    ln = bool(rng.integers(0, 2))
    layout = int(rng.integers(0, 2))
    h_path = kt_mlp.KT_H_AUTO if rng.integers(0, 2) else kt_mlp.KT_H_MEMORY
    return M, D, F, act, dt, bias, res, ln, layout, h_path


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_problem(i):
    _run_case(i, None)


# more seeds, H through memory, each problem in both launch modes (one persistent kernel
# for both projections, and two kernels): the work queue, the item ring, the early first
# copies and the split-K exchanges of both schedules on shapes no hand-written case has
N_CASES_BOTH = 64


@pytest.mark.parametrize("launches", [kt_mlp.KT_LAUNCH_ONE, kt_mlp.KT_LAUNCH_TWO], ids=["one", "two"])
@pytest.mark.parametrize("i", range(N_CASES, N_CASES + N_CASES_BOTH))
def test_random_problem_both_launch_modes(i, launches):
    _run_case(i, launches)


def _run_case(i, launches):
    M, D, F, act, dt, bias, res, ln, layout, h_path = _case(i)
    if launches is not None:
        h_path = kt_mlp.KT_H_MEMORY
    w = wl.custom(M, D, F, act, dt, bias, seed=9000 + i)
    t = wl.generate(w, residual=res, layernorm=ln)
    dev = wl.torch_order(t) if layout else t
    d = {k: v.cuda() for k, v in dev.items()}
    opts = {} if launches is None else {"launches": launches}
    plan = kt_mlp.Plan(M, D, F, act, dt, bias, residual=res, layernorm=ln, weight_layout=layout, ln_eps=EPS,
                       h_path=h_path, **opts)
    if launches is not None:
        assert plan.info()["one_launch"] == (launches == kt_mlp.KT_LAUNCH_ONE)
    Y = torch.full((M, D), float("nan"), dtype=wl.TORCH_DTYPES[dt], device="cuda")
    h_mem = not plan.info()["h_on_chip"]
    H = torch.full((M, F), float("nan"), dtype=wl.TORCH_DTYPES[dt], device="cuda") if h_mem else None
    plan.run_ex(d["X"], d["W_up"], d["W_down"], Y, d.get("b_up"), d.get("b_down"), d.get("R"),
                d.get("ln_gamma"), d.get("ln_beta"), H_out=H)
    torch.cuda.synchronize()
    assert plan.status() == kt_mlp.KT_OK, kt_mlp.kt_last_error()
    desc = plan.describe()
    plan.close()
    b = {k: wl.bits(v) for k, v in t.items()}
    lnarg = (b["ln_gamma"], b["ln_beta"], EPS) if ln else None
    Ho, Yx, _ = oracle.mlp(b["X"], b["W_up"], b["W_down"], b.get("b_up"), b.get("b_down"), act=act, dtype=dt,
                           R=b.get("R"), ln=lnarg)
    parity.check_y(wl.bits(Y.cpu()), Yx, dt, what=f"Y ({desc})")
    if h_mem:
        bb = dict(b)
        extra = None
        if ln:  # the up projection reads the normalised X (elements near a rounding boundary may differ)
            bb["X"], extra, _ = parity.ln_input_bound(b["X"], b["ln_gamma"], b["ln_beta"], EPS, dt)
        parity.check_h(wl.bits(H.cpu()), Ho, parity.h_bound(w, bb, x_extra=extra), dt, what=f"H ({desc})",
                       min_within_1ulp=parity.MIN_WITHIN_1ULP_LN if ln else parity.MIN_WITHIN_1ULP)
