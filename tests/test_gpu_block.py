"""GPU parity of the transformer-block options against the float64 oracle.

The feed-forward as a transformer block applies it ("SDXL as a requirements
inventory", section 1.3, BasicTransformerBlock: x = ff(LayerNorm(x)) + x): a
LayerNorm prologue, the residual add fused into the down projection's epilogue,
the sigmoid GELU and SiLU activations (sections 9.3 and 1.3) and weights in
PyTorch's nn.Linear order [out][in] (section 1.4), each through kt_mlp_plan_ex /
kt_mlp_run_ex.  Every comparison is element by element, the full SDXL and SigLIP
sizes included.  Forced tile plans put the [out][in] weights through
every kernel mode: one CTA per tile, CTA pairs, 128-deep k-blocks, split-K through
global memory and through a cluster's shared memory.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_mlp_gemms_gb300 import kt_mlp
from transformer_mlp_gemms_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TDT = wl.TORCH_DTYPES
EPS = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_mlp_gemms_gb300 import build
    build.build()
    kt_mlp.load()


def _run_block(w, d, residual, layernorm, layout, plan=None, Y=None, launches=kt_mlp.KT_LAUNCH_AUTO):
    own = plan is None
    if own:
        plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias, residual=residual, layernorm=layernorm,
                           weight_layout=layout, ln_eps=EPS, launches=launches)
    if Y is None:
        Y = torch.full((w.M, w.D), float("nan"), dtype=TDT[w.dtype], device="cuda")
    H = torch.full((w.M, w.F), float("nan"), dtype=TDT[w.dtype], device="cuda")
    plan.run_ex(d["X"], d["W_up"], d["W_down"], Y, d.get("b_up"), d.get("b_down"), d.get("R"),
                d.get("ln_gamma"), d.get("ln_beta"), H_out=H)
    torch.cuda.synchronize()
    assert plan.status() == kt_mlp.KT_OK, kt_mlp.kt_last_error()
    if own:
        plan.close()
    return Y.cpu(), H.cpu()


def _oracle(w, t, layout, rows=None):
    """The oracle's (H bits, Yx) for the block, and the H accumulation bound."""
    b = {k: wl.bits(v) for k, v in t.items()}
    ln = (b["ln_gamma"], b["ln_beta"], EPS) if "ln_gamma" in b else None
    Wu, Wd = b["W_up"], b["W_down"]
    if layout == kt_mlp.KT_W_OUT_IN:
        Wu, Wd = np.ascontiguousarray(Wu.T), np.ascontiguousarray(Wd.T)
    Ho, Yx, _ = oracle.mlp(b["X"], Wu, Wd, b.get("b_up"), b.get("b_down"), act=w.act, dtype=w.dtype, rows=rows,
                           R=b.get("R"), ln=ln, w_layout=layout)
    # the accumulation bound of H is that of the up projection of the (normalised) X, plus,
    # with LayerNorm, the effect of the normalised elements the GPU may round the other way
    bb = dict(b)
    extra = None
    if ln is not None:
        bb["X"], extra, _ = parity.ln_input_bound(b["X"], ln[0], ln[1], EPS, w.dtype)
        if rows is not None:
            extra = extra[rows]
    return Ho, Yx, parity.h_bound(w, bb, rows, x_extra=extra)


def _floor(t):
    """The within-one-step floor of H: lower with the LayerNorm prologue."""
    return parity.MIN_WITHIN_1ULP_LN if "ln_gamma" in t else parity.MIN_WITHIN_1ULP


def _inputs(w, residual, layernorm, layout):
    t = wl.generate(w, residual=residual, layernorm=layernorm)
    dev = wl.torch_order(t) if layout == kt_mlp.KT_W_OUT_IN else t
    return t, {k: v.cuda() for k, v in dev.items()}


CASES = [
    # id, (M, D, F, act, dtype, bias), residual, layernorm, layout, KT_FORCE_UP, KT_FORCE_DOWN
    ("silu_outin_ragged", (33, 64, 176, wl.ACT_SILU, wl.DT_F16, True), 1, 0, 1, None, None),
    ("sigmoid_gelu_ln", (129, 192, 320, wl.ACT_GELU_SIGMOID, wl.DT_BF16, False), 0, 1, 0, None, None),
    ("geglu_outin_ln_res", (200, 640, 2560, wl.ACT_GEGLU, wl.DT_BF16, True), 1, 1, 1, None, None),
    ("tanh_outin_pair", (300, 256, 1000, wl.ACT_GELU_TANH, wl.DT_F16, False), 1, 0, 1, "128,2,64", "64,1,2,64"),
    ("erf_outin_bk128_splitk", (257, 1152, 4304, wl.ACT_GELU_ERF, wl.DT_F16, False), 1, 1, 1, "192,1,128",
     "96,4,1,128,0"),
    ("none_outin_cluster_sk", (130, 72, 4104, wl.ACT_NONE, wl.DT_F16, True), 1, 0, 1, None, "96,4,1,64,1"),
    ("geglu_outin_pair_bn128", (64, 320, 640, wl.ACT_GEGLU, wl.DT_BF16, True), 0, 0, 1, "128,2,64", None),
    ("geglu_outin_pair_share32", (300, 136, 200, wl.ACT_GEGLU, wl.DT_F16, True), 1, 0, 1, "64,2,128", None),
    ("geglu_inout_pair_bk128", (520, 264, 648, wl.ACT_GEGLU, wl.DT_BF16, True), 0, 1, 0, "128,2,128", None),
    ("geglu_inout_bn64", (129, 200, 136, wl.ACT_GEGLU, wl.DT_F16, False), 1, 0, 0, "64,1,64", None),
    ("geglu_outin_bn96_bk128", (77, 128, 136, wl.ACT_GEGLU, wl.DT_F16, False), 1, 0, 1, "96,1,128", "32,2,1,128,0"),
    ("silu_pair_splitk_res", (384, 1280, 512, wl.ACT_SILU, wl.DT_BF16, True), 1, 1, 0, "128,2,128",
     "128,2,2,64,0"),
    ("tiny_everything", (5, 8, 8, wl.ACT_GELU_SIGMOID, wl.DT_F16, True), 1, 1, 1, None, None),
    ("geglu_pair_ln_bk128", (520, 264, 648, wl.ACT_GEGLU, wl.DT_BF16, True), 0, 1, 0, "128,2,128", None),
    ("wide_ln_reread", (40, 4096, 64, wl.ACT_GELU_ERF, wl.DT_BF16, False), 1, 1, 1, None, None),
    # [in][out] weights whose CTA column share is an odd multiple of 32: 32-column weight
    # boxes with 64-byte swizzle (single CTAs of 160 and 96 columns, a pair of 96 + 96)
    ("tanh_inout_box32", (300, 352, 1000, wl.ACT_GELU_TANH, wl.DT_F16, True), 1, 0, 0, "160,1,64", "96,1,1,128"),
    ("erf_inout_pair_box32", (520, 400, 776, wl.ACT_GELU_ERF, wl.DT_BF16, True), 0, 1, 0, "192,2,128",
     "192,1,2,64"),
]


@pytest.mark.parametrize("cid,shape,residual,layernorm,layout,fu,fd", CASES, ids=[c[0] for c in CASES])
def test_block_options_element_by_element(monkeypatch, cid, shape, residual, layernorm, layout, fu, fd):
    if fu:
        monkeypatch.setenv("KT_FORCE_UP", fu)
    if fd:
        monkeypatch.setenv("KT_FORCE_DOWN", fd)
    M, D, F, act, dt, bias = shape
    w = wl.custom(M, D, F, act, dt, bias, seed=3000 + M + D + F + act)
    t, d = _inputs(w, residual, layernorm, layout)
    Y, H = _run_block(w, d, residual, layernorm, layout)
    Ho, Yx, bound = _oracle(w, t, layout)
    parity.check_y(wl.bits(Y), Yx, w.dtype)
    parity.check_h(wl.bits(H), Ho, bound, w.dtype, min_within_1ulp=_floor(t))


@pytest.mark.parametrize("name,act", [("sdxl_l2", None), ("sdxl_l1", None), ("siglip", None),
                                      ("siglip", wl.ACT_GELU_SIGMOID)])
def test_full_size_block_every_element(name, act):
    base = wl.WORKLOADS[name]
    w = wl.custom(base.M, base.D, base.F, base.act if act is None else act, base.dtype, base.bias, seed=base.seed)
    t, d = _inputs(w, True, True, kt_mlp.KT_W_OUT_IN)
    Y, H = _run_block(w, d, True, True, kt_mlp.KT_W_OUT_IN)
    assert torch.isfinite(Y.float()).all(), "unwritten or non-finite Y"
    Ho, Yx, bound = _oracle(w, t, kt_mlp.KT_W_OUT_IN)
    parity.check_y(wl.bits(Y), Yx, w.dtype, what=f"Y {name} block")
    parity.check_h(wl.bits(H), Ho, bound, w.dtype, what=f"H {name} block", min_within_1ulp=_floor(t))


def test_layernorm_output_through_identity_weights():
    # with W_up = W_down = I and no activation, H = round(Xn) and Y = H exactly, so the
    # kernel's normalised X is visible.  It computes in fp32, the oracle in float64: an
    # element must round to within 1 ulp of the oracle's, or, where gamma * n and beta
    # cancel to a value near zero, lie within 1 ulp plus the fp32 error of the affine
    # step's operands, 2^-20 * (|gamma| (|n| + 1) + |beta|)  (n the normalised value).
    M, D = 300, 640
    for dt in (wl.DT_F16, wl.DT_BF16):
        w = wl.custom(M, D, D, wl.ACT_NONE, dt, False, seed=41)
        t = wl.generate(w, layernorm=True)
        # a residual stream with a per-row offset and scale, as LayerNorm sees in a network
        g = torch.Generator("cpu").manual_seed(42)
        scale = torch.rand(M, 1, generator=g) * 4 + 0.25
        shift = torch.randn(M, 1, generator=g) * 3
        t["X"] = (t["X"].float() * scale + shift).to(TDT[dt])
        eye = torch.eye(D, dtype=TDT[dt])
        t["W_up"], t["W_down"] = eye, eye
        d = {k: v.cuda() for k, v in t.items()}
        Y, H = _run_block(w, d, False, True, kt_mlp.KT_W_IN_OUT)
        assert torch.equal(Y.view(torch.int16), H.view(torch.int16))
        b = {k: wl.bits(v) for k, v in t.items()}
        gam, bet = oracle.decode(b["ln_gamma"], dt), oracle.decode(b["ln_beta"], dt)
        exact = oracle.layernorm(oracle.decode(b["X"], dt), gam, bet, EPS)
        n = oracle.layernorm(oracle.decode(b["X"], dt), np.ones(D), np.zeros(D), EPS)
        ref = oracle.encode(exact, dt)
        got = wl.bits(Y)
        dist = np.abs(parity.ordered(got) - parity.ordered(ref))
        err = np.abs(oracle.decode(got, dt) - exact)
        budget = parity.ulp(exact, dt) + 2.0 ** -20 * (np.abs(gam) * (np.abs(n) + 1) + np.abs(bet))
        ok = (dist <= 1) | (err <= budget)
        assert ok.all(), (int(dist.max()), np.argwhere(~ok)[:5])
        assert (dist == 0).mean() >= 0.99
        # an element rounds the other way only where its exact value lies within the GPU's
        # fp32 error of a rounding boundary: the premise of the H bound of the block tests
        _, _, ambiguous = parity.ln_input_bound(b["X"], b["ln_gamma"], b["ln_beta"], EPS, dt)
        assert not np.any((dist > 0) & ~ambiguous), np.argwhere((dist > 0) & ~ambiguous)[:5]


def test_in_place_residual_stream_update():
    # x = ff(LayerNorm(x)) + x with Y, R and X the same buffer
    w = wl.WORKLOADS["sdxl_l2"]
    t = wl.generate(w, layernorm=True)
    t["R"] = t["X"]
    d = {k: v.cuda() for k, v in wl.torch_order(t).items()}
    x = d["X"].clone()
    d["X"] = x
    d["R"] = x
    Y, H = _run_block(w, d, True, True, kt_mlp.KT_W_OUT_IN, Y=x)
    Ho, Yx, bound = _oracle(w, t, kt_mlp.KT_W_OUT_IN)
    parity.check_y(wl.bits(Y), Yx, w.dtype, what="Y in place")
    parity.check_h(wl.bits(H), Ho, bound, w.dtype, what="H in place", min_within_1ulp=_floor(t))


def test_run_ex_on_a_plain_plan_matches_kt_mlp_run_bitwise():
    w = wl.WORKLOADS["sdxl_l2"]
    d = {k: v.cuda() for k, v in wl.generate(w).items()}
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias)
    Y1 = torch.empty((w.M, w.D), dtype=TDT[w.dtype], device="cuda")
    Y2 = torch.empty_like(Y1)
    plan.run(d["X"], d["W_up"], d["W_down"], d["b_up"], d["b_down"], Y1)
    plan.run_ex(d["X"], d["W_up"], d["W_down"], Y2, d["b_up"], d["b_down"])
    torch.cuda.synchronize()
    assert plan.status() == kt_mlp.KT_OK
    plan.close()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))


def test_run_ex_rejects_tensors_that_do_not_match_the_plan():
    w = wl.custom(64, 64, 128, wl.ACT_SILU, wl.DT_F16, False, seed=5)
    d = {k: v.cuda() for k, v in wl.generate(w, residual=True, layernorm=True).items()}
    Y = torch.empty((w.M, w.D), dtype=torch.float16, device="cuda")
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias, residual=True, layernorm=True)
    for kw in (dict(R=None, ln_gamma=d["ln_gamma"], ln_beta=d["ln_beta"]),   # residual plan without R
               dict(R=d["R"], ln_gamma=None, ln_beta=d["ln_beta"]),          # LayerNorm plan without gamma
               dict(R=d["R"], ln_gamma=d["ln_gamma"], ln_beta=d["ln_beta"], b_up=d["X"])):  # stray bias
        with pytest.raises(kt_mlp.KtError) as e:
            plan.run_ex(d["X"], d["W_up"], d["W_down"], Y, **kw)
        assert e.value.status == kt_mlp.KT_ERR_INVALID
    with pytest.raises(kt_mlp.KtError) as e:
        plan.run(d["X"], d["W_up"], d["W_down"], None, None, Y)  # the plain call has no R
    assert e.value.status == kt_mlp.KT_ERR_INVALID
    plan.close()


def test_timed_block_reports_three_kernels():
    w = wl.WORKLOADS["sdxl_l2"]
    t, d = _inputs(w, True, True, kt_mlp.KT_W_OUT_IN)
    plan = kt_mlp.Plan(w.M, w.D, w.F, w.act, w.dtype, w.bias, residual=True, layernorm=True,
                       weight_layout=kt_mlp.KT_W_OUT_IN, ln_eps=EPS)
    Y = torch.empty((w.M, w.D), dtype=TDT[w.dtype], device="cuda")
    for _ in range(3):
        ms = plan.run_ex_timed(d["X"], d["W_up"], d["W_down"], Y, d["b_up"], d["b_down"], d["R"],
                               d["ln_gamma"], d["ln_beta"])
    assert plan.status() == kt_mlp.KT_OK
    plan.close()
    assert all(0 < m < 5.0 for m in ms), ms


# Both projections in one persistent launch (tiles from one work queue) against two launches,
# each element by element against the oracle: CTA pairs and single CTAs, GEGLU and elementwise
# activations, both weight orders, LayerNorm and residual, whole down tiles and down tiles
# split along K (the last CTA to finish a tile sums the partials; ragged tiles and splits).
ONE_LAUNCH_CASES = [
    # id, (M, D, F, act, dtype, bias), residual, layernorm, layout, KT_FORCE_UP, KT_FORCE_DOWN
    ("geglu_pair_whole", (520, 264, 648, wl.ACT_GEGLU, wl.DT_BF16, True), 0, 1, 0, "128,2,128", "64,1,2,128"),
    ("geglu_pair_split3", (520, 264, 648, wl.ACT_GEGLU, wl.DT_BF16, True), 1, 0, 0, "128,2,128", "128,3,2,128"),
    ("erf_outin_ln_res", (700, 320, 1000, wl.ACT_GELU_ERF, wl.DT_F16, False), 1, 1, 1, None, None),
    ("erf_outin_split2", (700, 320, 1000, wl.ACT_GELU_ERF, wl.DT_F16, True), 1, 0, 1, "128,1,64", "64,2,1,64"),
    ("tanh_single_cta", (300, 256, 1000, wl.ACT_GELU_TANH, wl.DT_F16, True), 1, 0, 0, "128,1,64", None),
    ("tanh_split4_ragged", (729, 192, 1000, wl.ACT_GELU_TANH, wl.DT_F16, False), 0, 0, 0, "192,1,64",
     "192,4,1,64"),
    ("silu_many_tiles", (1500, 136, 776, wl.ACT_SILU, wl.DT_BF16, True), 0, 0, 0, None, None),
    ("tiny", (33, 64, 176, wl.ACT_GELU_ERF, wl.DT_F16, False), 0, 0, 0, None, None),
]


@pytest.mark.parametrize("cid,shape,residual,layernorm,layout,fu,fd", ONE_LAUNCH_CASES,
                         ids=[c[0] for c in ONE_LAUNCH_CASES])
@pytest.mark.parametrize("launches", [kt_mlp.KT_LAUNCH_ONE, kt_mlp.KT_LAUNCH_TWO])
def test_one_launch_and_two_launches_match_the_oracle(monkeypatch, cid, shape, residual, layernorm, layout, fu, fd,
                                                      launches):
    if fu:
        monkeypatch.setenv("KT_FORCE_UP", fu)
    if fd:
        monkeypatch.setenv("KT_FORCE_DOWN", fd)
    M, D, F, act, dt, bias = shape
    w = wl.custom(M, D, F, act, dt, bias, seed=5000 + M + D + F + act)
    info = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(M, D, F, act, dt, bias, residual, layernorm, layout,
                                                     launches=launches), 152)
    assert info["one_launch"] == (launches == kt_mlp.KT_LAUNCH_ONE)
    if fd:
        assert info["down"]["split_k"] == int(fd.split(",")[1]) and info["down"]["cluster_sk"] == 0
    t, d = _inputs(w, residual, layernorm, layout)
    Y, H = _run_block(w, d, residual, layernorm, layout, launches=launches)
    Ho, Yx, bound = _oracle(w, t, layout)
    parity.check_y(wl.bits(Y), Yx, w.dtype)
    parity.check_h(wl.bits(H), Ho, bound, w.dtype, min_within_1ulp=_floor(t))
