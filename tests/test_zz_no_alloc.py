"""The allocation-free down projection, kt_down_proj_noalloc, against the oracle.

Some callers of this library cannot allocate device memory where they call it: a
host framework's plugin hook that is handed only input / output pointers and a
stream, or a latency-critical serving loop that must never call cudaMalloc /
cudaFree (cudaFree synchronises the whole device).  For them the library offers the
down projection with its split-K scratch in a static device array instead of a
plan's workspace.  These tests call it through the C ABI on the H that the regular
entry point (kt_mlp_run_with_h) writes, and compare its Y with the float64 oracle's
down projection of that same H, on two calls in a row, within the Y tolerance of the
parity tests; and with the regular entry point's Y, which runs the same kernel.

This file is named so that pytest collects it last.
"""
import pytest
import torch

import oracle
import parity
from transformer_mlp_gemms_gb300 import kt_mlp
from transformer_mlp_gemms_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_mlp_gemms_gb300 import build
    build.build()
    kt_mlp.load()


CASES = [
    # (workload, KT_FORCE_DOWN for both the regular plan and the entry point's own plan)
    (wl.WORKLOADS["siglip"], None),                          # the planner's choice (no cluster split-K)
    (wl.WORKLOADS["siglip"], "96,2,1,128,0"),                # split-K: partials in the static scratch
    (wl.WORKLOADS["sdxl_l2"], None),                         # bf16 with b_down, the planner's choice
    (wl.custom(300, 1280, 5120, wl.ACT_GEGLU, wl.DT_BF16, True, seed=32), "128,3,1,128,0"),  # bf16, three splits
    (wl.custom(33, 64, 176, wl.ACT_GELU_ERF, wl.DT_F16, True, seed=31), None),  # ragged, tiny
]


@pytest.mark.parametrize("w,force", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_noalloc_down_projection_matches_the_oracle(monkeypatch, w, force):
    # the regular path as two launches, whose down projection runs the same kernel as the
    # allocation-free entry point; KT_FORCE_DOWN (read by the planner on both paths) pins
    # a split-K plan whose partials go through global memory, that is, through the static
    # scratch of the entry point
    monkeypatch.setenv("KT_FORCE_LAUNCHES", "2")
    if force:
        monkeypatch.setenv("KT_FORCE_DOWN", force)
    t = wl.generate(w)
    d = {k: v.cuda() for k, v in t.items()}
    tdt = wl.TORCH_DTYPES[w.dtype]
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    dn = plan.info()["down"]
    if force:
        assert dn["split_k"] == int(force.split(",")[1]) > 1 and dn["cluster_sk"] == 0
    Y_ref = torch.empty((w.M, w.D), dtype=tdt, device="cuda")
    H = torch.empty((w.M, w.F), dtype=tdt, device="cuda")
    plan.run_with_h(d["X"], d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Y_ref, H)
    torch.cuda.synchronize()
    assert plan.status() == kt_mlp.KT_OK
    plan.close()
    # the oracle's down projection of the H the GPU wrote (float64, natural order)
    b = {k: wl.bits(v) for k, v in t.items()}
    Yx = oracle.linear(oracle.decode(wl.bits(H.cpu()), w.dtype), oracle.decode(b["W_down"], w.dtype),
                       oracle.decode(b["b_down"], w.dtype) if w.bias else None)
    ref_bits = wl.bits(Y_ref.cpu())
    for call in range(2):
        Y = torch.full((w.M, w.D), float("nan"), dtype=tdt, device="cuda")
        kt_mlp.kt_down_proj_noalloc(w.M, w.F, w.D, w.dtype, H, d["W_down"], d.get("b_down"), Y)
        torch.cuda.synchronize()
        got = wl.bits(Y.cpu())
        parity.check_y(got, Yx, w.dtype, what=f"Y of call {call + 1}")
        if force:  # the same kernel and plan as the regular down projection: the same bits
            assert (got == ref_bits).all(), f"call {call + 1} differs from the regular entry point"


def test_noalloc_rejects_a_problem_beyond_its_scratch(monkeypatch):
    # a split-K plan whose fp32 partials (4 x 4096 x 1152 x 4 bytes = 75.5 MB) exceed the
    # 16 MiB static scratch; the size check comes before any launch, so small stand-in
    # buffers are enough here
    monkeypatch.setenv("KT_FORCE_DOWN", "128,4,1,128,0")
    w = wl.WORKLOADS["sweep_M4096"]
    buf = torch.empty(1024, dtype=torch.float16, device="cuda")
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.kt_down_proj_noalloc(w.M, w.F, w.D, w.dtype, buf, buf, None, buf)
    assert e.value.status == kt_mlp.KT_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()


def test_noalloc_rejects_bad_arguments():
    buf = torch.empty(1024, dtype=torch.float16, device="cuda")
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.kt_down_proj_noalloc(16, 64, 64, wl.DT_F16, None, buf, None, buf)
    assert e.value.status == kt_mlp.KT_ERR_INVALID
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.kt_down_proj_noalloc(16, 64, 64, wl.DT_F16, buf.data_ptr() + 2, buf, None, buf)
    assert e.value.status == kt_mlp.KT_ERR_INVALID
