"""kt_mlp_run / kt_mlp_run_ex captured into a CUDA graph and replayed.

Every launch parameter of a run stays the same from call to call (the down
projection's per-row-block readiness counters are reset by their last reader), so a
captured graph replays the kernels correctly.  Each replay gets new inputs copied into
the captured buffers and must give bit for bit the Y of an eager call on them.
"""
import pytest
import torch

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


SIGLIP = (729, 1152, 4304, wl.ACT_GELU_TANH, wl.DT_F16, False)
CASES = [
    # (M, D, F, act, dtype, bias), block options, h_path, launches
    (SIGLIP, {}, kt_mlp.KT_H_MEMORY, kt_mlp.KT_LAUNCH_ONE),   # one launch, down tiles split along K
    (SIGLIP, {}, kt_mlp.KT_H_MEMORY, kt_mlp.KT_LAUNCH_TWO),   # two launches, cluster split-K
    ((2048, 1280, 5120, wl.ACT_GEGLU, wl.DT_BF16, True), {}, kt_mlp.KT_H_MEMORY, kt_mlp.KT_LAUNCH_AUTO),  # pairs
    # SDXL level 1: one launch of CTA pairs over many waves (the work counter reset by the last unit)
    ((8192, 640, 2560, wl.ACT_GEGLU, wl.DT_BF16, True), {}, kt_mlp.KT_H_MEMORY, kt_mlp.KT_LAUNCH_ONE),
    ((300, 256, 1000, wl.ACT_SILU, wl.DT_F16, True), {"residual": True, "layernorm": True}, kt_mlp.KT_H_MEMORY,
     kt_mlp.KT_LAUNCH_AUTO),
    ((33, 64, 176, wl.ACT_GELU_ERF, wl.DT_F16, False), {}, kt_mlp.KT_H_ON_CHIP, kt_mlp.KT_LAUNCH_AUTO),  # fused
]


@pytest.mark.parametrize("shape,opts,h_path,launches", CASES,
                         ids=["siglip_one", "siglip_two", "sdxl_l2", "sdxl_l1_one", "block", "h_on_chip"])
def test_graph_replay_matches_eager_runs(shape, opts, h_path, launches):
    M, D, F, act, dt, bias = shape
    res, ln = opts.get("residual", False), opts.get("layernorm", False)
    w = wl.custom(M, D, F, act, dt, bias, seed=123)
    t = wl.generate(w, residual=res, layernorm=ln)
    d = {k: v.cuda() for k, v in t.items()}
    plan = kt_mlp.Plan(M, D, F, act, dt, bias, residual=res, layernorm=ln, h_path=h_path, launches=launches)
    tdt = wl.TORCH_DTYPES[dt]
    X = torch.empty_like(d["X"])
    Y = torch.empty((M, D), dtype=tdt, device="cuda")
    kw = dict(b_up=d.get("b_up"), b_down=d.get("b_down"), R=d.get("R"), ln_gamma=d.get("ln_gamma"),
              ln_beta=d.get("ln_beta"))
    inputs = [(torch.randn(M, D, generator=torch.Generator("cpu").manual_seed(s)) * (1 + s)).to(tdt).cuda()
              for s in range(4)]
    # eager results, one per input
    ref = []
    for x in inputs:
        X.copy_(x)
        plan.run_ex(X, d["W_up"], d["W_down"], Y, **kw)
        torch.cuda.synchronize()
        ref.append(Y.clone())
    assert plan.status() == kt_mlp.KT_OK
    # capture one call on the static buffers, replay it on each input (twice over)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan.run_ex(X, d["W_up"], d["W_down"], Y, **kw)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        plan.run_ex(X, d["W_up"], d["W_down"], Y, **kw)
    for _ in range(2):
        for x, r in zip(inputs, ref):
            X.copy_(x)
            Y.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(Y.view(torch.int16), r.view(torch.int16))
    assert plan.status() == kt_mlp.KT_OK, kt_mlp.kt_last_error()
    del g
    plan.close()
