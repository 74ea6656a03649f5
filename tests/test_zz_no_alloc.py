"""The allocation-free down projection, kt_down_proj_noalloc, against the regular path.

Some callers of this library cannot allocate device memory where they call it: a
host framework's plugin hook that is handed only input / output pointers and a
stream, or a latency-critical serving loop that must never call cudaMalloc /
cudaFree (cudaFree synchronises the whole device).  For them the library offers the
down projection with its split-K scratch in a static device array instead of a
plan's workspace.  These tests call it through the C ABI and compare its Y with the Y
of the regular entry point (kt_mlp_run_with_h, which also returns the H the down
projection reads), on two calls in a row, within the Y tolerance of the parity tests.

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
    wl.WORKLOADS["siglip"],                                        # split-K: partials in the static scratch
    wl.WORKLOADS["sdxl_l2"],                                       # bf16 with b_down
    wl.custom(33, 64, 176, wl.ACT_GELU_ERF, wl.DT_F16, True, seed=31),  # ragged, tiny
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_down_projection_matches_the_regular_entry_point(monkeypatch, w):
    # the regular path as two launches, whose down projection the allocation-free entry
    # point runs (with the split-K reduction through global memory)
    monkeypatch.setenv("KT_FORCE_LAUNCHES", "2")
    t = wl.generate(w)
    d = {k: v.cuda() for k, v in t.items()}
    tdt = wl.TORCH_DTYPES[w.dtype]
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    if w.name == "siglip":
        assert plan.info()["down"]["split_k"] > 1  # the case exercises the static split-K scratch
    Y_ref = torch.empty((w.M, w.D), dtype=tdt, device="cuda")
    H = torch.empty((w.M, w.F), dtype=tdt, device="cuda")
    plan.run_with_h(d["X"], d["W_up"], d["W_down"], d.get("b_up"), d.get("b_down"), Y_ref, H)
    torch.cuda.synchronize()
    assert plan.status() == kt_mlp.KT_OK
    plan.close()
    ref = oracle.decode(wl.bits(Y_ref.cpu()), w.dtype)
    for call in range(2):
        Y = torch.full((w.M, w.D), float("nan"), dtype=tdt, device="cuda")
        kt_mlp.kt_down_proj_noalloc(w.M, w.F, w.D, w.dtype, H, d["W_down"], d.get("b_down"), Y)
        torch.cuda.synchronize()
        parity.check_y(wl.bits(Y.cpu()), ref, w.dtype, what=f"Y of call {call + 1}")


def test_noalloc_rejects_a_problem_beyond_its_scratch():
    w = wl.WORKLOADS["sweep_M16384"]
    info = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias,
                                   torch.cuda.get_device_properties(0).multi_processor_count)
    dn = info["down"]
    need = dn["split_k"] * dn["tiles_m"] * 128 * dn["tiles_n"] * dn["BN"] * 4 if dn["split_k"] > 1 else 0
    if need <= 16 << 20:
        pytest.skip("the planner needs no large scratch for this shape")
    # the size check comes before any launch, so small stand-in buffers are enough here
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
