"""GPU parity of the H-on-chip kernel (one kernel, H kept in shared memory slice by slice).

The variant applies where Y[128 x D] fits tensor memory beside two 64-column slice
accumulators (D <= 256; D <= 192 for GEGLU) and to [in][out] weights.  Y is compared
with the float64 oracle element by element on small shapes and on sampled rows of a
many-wave shape; H is not written by this path, so only Y is checked.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_mlp_gemms_gb300 import build
    build.build()
    kt_mlp.load()


def _run(w, residual=False, layernorm=False, rows=None):
    t = wl.generate(w, residual=residual, layernorm=layernorm)
    d = {k: v.cuda() for k, v in t.items()}
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias, residual=residual, layernorm=layernorm,
                       ln_eps=EPS, h_path=kt_mlp.KT_H_ON_CHIP)
    assert plan.info()["h_on_chip"] == 1
    Y = torch.full((w.M, w.D), float("nan"), dtype=wl.TORCH_DTYPES[w.dtype], device="cuda")
    plan.run_ex(d["X"], d["W_up"], d["W_down"], Y, d.get("b_up"), d.get("b_down"), d.get("R"),
                d.get("ln_gamma"), d.get("ln_beta"))
    torch.cuda.synchronize()
    assert plan.status() == kt_mlp.KT_OK, kt_mlp.kt_last_error()
    plan.close()
    b = {k: wl.bits(v) for k, v in t.items()}
    ln = (b["ln_gamma"], b["ln_beta"], EPS) if layernorm else None
    _, Yx, _ = oracle.mlp(b["X"], b["W_up"], b["W_down"], b.get("b_up"), b.get("b_down"), act=w.act,
                          dtype=w.dtype, rows=rows, R=b.get("R"), ln=ln)
    yb = wl.bits(Y.cpu())
    if rows is not None:
        yb = yb[rows]
    parity.check_y(yb, Yx, w.dtype)


CASES = [
    # M, D, F, act, dtype, bias, residual, layernorm
    (33, 64, 176, wl.ACT_GELU_ERF, wl.DT_F16, False, False, False),       # the tiny workload's shape
    (1, 64, 64, wl.ACT_NONE, wl.DT_F16, True, False, False),              # one row, one slice
    (300, 128, 200, wl.ACT_GEGLU, wl.DT_BF16, True, False, False),        # ragged M and F, GEGLU
    (257, 256, 512, wl.ACT_SILU, wl.DT_F16, True, True, True),            # widest D, block options
    (64, 192, 128, wl.ACT_GEGLU, wl.DT_F16, False, True, False),          # widest GEGLU D
    (129, 72, 136, wl.ACT_GELU_TANH, wl.DT_BF16, False, False, False),    # D not a multiple of 64
    (200, 64, 1000, wl.ACT_GELU_SIGMOID, wl.DT_F16, True, False, False),  # many slices
]


@pytest.mark.parametrize("M,D,F,act,dt,bias,res,ln", CASES)
def test_h_on_chip_matches_the_oracle(M, D, F, act, dt, bias, res, ln):
    _run(wl.custom(M, D, F, act, dt, bias, seed=5000 + M + D + F + act), res, ln)


def test_h_on_chip_many_waves_every_element():
    # 313 row blocks over 152 SMs: every CTA runs several row blocks
    w = wl.custom(40000, 64, 256, wl.ACT_GELU_TANH, wl.DT_F16, False, seed=77)
    _run(w)


def test_h_on_chip_matches_the_two_kernel_path_closely():
    w = wl.WORKLOADS["tiny"]
    d = {k: v.cuda() for k, v in wl.generate(w).items()}
    out = []
    for hp in (kt_mlp.KT_H_MEMORY, kt_mlp.KT_H_ON_CHIP):
        plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias, h_path=hp)
        Y = torch.empty((w.M, w.D), dtype=torch.float16, device="cuda")
        plan.run_ex(d["X"], d["W_up"], d["W_down"], Y)
        torch.cuda.synchronize()
        assert plan.status() == kt_mlp.KT_OK
        plan.close()
        out.append(Y.float().cpu())
    # the same H (one rounding of the same fp32 values) and the same fp32 sums up to order
    assert torch.allclose(out[0], out[1], rtol=2e-3, atol=2e-3)


def test_h_on_chip_plan_errors():
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.Plan(64, 320, 128, wl.ACT_GELU_ERF, wl.DT_F16, False, h_path=kt_mlp.KT_H_ON_CHIP)
    assert e.value.status == kt_mlp.KT_ERR_UNSUPPORTED
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.Plan(64, 64, 128, wl.ACT_GELU_ERF, wl.DT_F16, False, weight_layout=kt_mlp.KT_W_OUT_IN,
                    h_path=kt_mlp.KT_H_ON_CHIP)
    assert e.value.status == kt_mlp.KT_ERR_UNSUPPORTED
    w = wl.custom(64, 64, 128, wl.ACT_GELU_ERF, wl.DT_F16, False, seed=1)
    d = {k: v.cuda() for k, v in wl.generate(w).items()}
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias, h_path=kt_mlp.KT_H_ON_CHIP)
    Y = torch.empty((w.M, w.D), dtype=torch.float16, device="cuda")
    H = torch.empty((w.M, w.F), dtype=torch.float16, device="cuda")
    with pytest.raises(kt_mlp.KtError) as e:
        plan.run_ex(d["X"], d["W_up"], d["W_down"], Y, H_out=H)
    assert e.value.status == kt_mlp.KT_ERR_INVALID
    with pytest.raises(kt_mlp.KtError) as e:
        plan.run_with_h(d["X"], d["W_up"], d["W_down"], None, None, Y, H)
    assert e.value.status == kt_mlp.KT_ERR_INVALID
    # the host-buffer entry point runs the fused kernel like any other plan
    Xh = d["X"].cpu().pin_memory()
    Yh = torch.empty((w.M, w.D), dtype=torch.float16).pin_memory()
    plan.run_host(Xh, d["W_up"], d["W_down"], None, None, Yh)
    Yd = torch.empty_like(Y)
    plan.run_ex(d["X"], d["W_up"], d["W_down"], Yd)
    torch.cuda.synchronize()
    assert torch.equal(Yh.view(torch.int16), Yd.cpu().view(torch.int16))
    plan.close()
