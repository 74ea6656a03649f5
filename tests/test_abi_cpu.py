"""The C-ABI library on the CPU: it loads, exports every declared symbol, and its
host-only planner keeps the grid invariants ("The software stack", sections 2.1
and 2.2: padding-discounted tile choice; every output element produced exactly
once; SK > 1 only with a reduction).  No compute call is made here."""
import os
import re

import pytest

from transformer_mlp_gemms_gb300 import build as kbuild
from transformer_mlp_gemms_gb300 import kt_mlp
from transformer_mlp_gemms_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kt_mlp.h")
SMS = 152  # GB300


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kt_mlp.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kt_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("kt_mlp_plan", "kt_mlp_run", "kt_mlp_destroy", "kt_mlp_status", "kt_last_error",
                     "kt_mlp_describe", "kt_mlp_run_with_h"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_symbols()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding wraps each of them under the same name
    assert set(names) <= set(kt_mlp.SIGNATURES)
    assert lib.kt_mlp_abi_version() == 3


def test_plan_without_a_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.kt_mlp_plan(33, 64, 176, 0, 0, False)
    assert e.value.status in (kt_mlp.KT_ERR_CUDA, kt_mlp.KT_ERR_UNSUPPORTED)


@pytest.mark.parametrize("args,status", [
    ((0, 64, 64, 0, 0, 0), kt_mlp.KT_ERR_INVALID),
    ((8, -8, 64, 0, 0, 0), kt_mlp.KT_ERR_INVALID),
    ((8, 64, 64, 7, 0, 0), kt_mlp.KT_ERR_INVALID),
    ((8, 64, 64, 0, 2, 0), kt_mlp.KT_ERR_INVALID),
    ((8, 64, 64, 0, 0, 2), kt_mlp.KT_ERR_INVALID),
    ((8, 60, 64, 0, 0, 0), kt_mlp.KT_ERR_UNSUPPORTED),
    ((8, 64, 20, 0, 0, 0), kt_mlp.KT_ERR_UNSUPPORTED),
])
def test_argument_errors(lib, args, status):
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.kt_mlp_plan_info(*args, SMS)
    assert e.value.status == status
    assert kt_mlp.kt_last_error()


def test_null_handles_are_rejected(lib):
    assert lib.kt_mlp_destroy(None) == kt_mlp.KT_ERR_INVALID
    assert lib.kt_mlp_status(None) == kt_mlp.KT_ERR_INVALID
    assert lib.kt_mlp_run(None, None, None, None, None, None, None, None) == kt_mlp.KT_ERR_INVALID
    assert lib.kt_mlp_debug_stall(None, 1, 10) == kt_mlp.KT_ERR_INVALID
    t = kt_mlp.tensors(None, None, None, None)
    assert lib.kt_mlp_run_ex(None, t, None) == kt_mlp.KT_ERR_INVALID
    assert lib.kt_mlp_run_ex_timed(None, t, None, None) == kt_mlp.KT_ERR_INVALID
    assert lib.kt_mlp_plan_ex(None, None) == kt_mlp.KT_ERR_INVALID


@pytest.mark.parametrize("kw,status", [
    (dict(residual=2), kt_mlp.KT_ERR_INVALID),
    (dict(layernorm=2), kt_mlp.KT_ERR_INVALID),
    (dict(layernorm=1, ln_eps=0.0), kt_mlp.KT_ERR_INVALID),
    (dict(layernorm=1, ln_eps=-1e-5), kt_mlp.KT_ERR_INVALID),
    (dict(layernorm=1, ln_eps=float("inf")), kt_mlp.KT_ERR_INVALID),
    (dict(weight_layout=2), kt_mlp.KT_ERR_INVALID),
    (dict(act=6), kt_mlp.KT_ERR_INVALID),
    (dict(D=60), kt_mlp.KT_ERR_UNSUPPORTED),
])
def test_option_errors(lib, kw, status):
    base = dict(M=8, D=64, F=64, act=0, dtype=0, bias=0, residual=0, layernorm=0, weight_layout=0, ln_eps=1e-5)
    base.update(kw)
    o = kt_mlp.kt_mlp_options(**base)
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.kt_mlp_plan_info_ex(o, SMS)
    assert e.value.status == status
    assert kt_mlp.kt_last_error()


def test_options_are_reported_and_default_to_the_plain_plan(lib):
    w = wl.WORKLOADS["sdxl_l2"]
    plain = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, SMS)
    same = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(w.M, w.D, w.F, w.act, w.dtype, w.bias), SMS)
    assert same == plain
    assert (plain["residual"], plain["layernorm"], plain["weight_layout"]) == (0, 0, 0)
    ex = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(w.M, w.D, w.F, w.act, w.dtype, w.bias, residual=True,
                                                   layernorm=True, ln_eps=1e-6), SMS)
    assert (ex["residual"], ex["layernorm"]) == (1, 1)
    assert ex["ln_eps"] == pytest.approx(1e-6)
    assert ex["workspace_bytes"] == plain["workspace_bytes"] + 2 * w.M * w.D  # the normalised X


def _check_gemm(g, M, N, K):
    assert (g["M"], g["N"], g["K"]) == (M, N, K)
    BM, BN, BK, SK = g["BM"], g["BN"], g["BK"], g["split_k"]
    assert BM in (128, 256) and BK in (64, 128)  # 256: a CTA pair (cta_group::2) per tile
    pair = BM // 128
    assert BN % 32 == 0 and 32 <= BN <= 256
    assert (BN // pair) % 16 == 0  # a pair's column share: whole 16-column weight boxes
    # the grid covers every output element exactly once: tiles_m * BM >= M > (tiles_m - 1) * BM
    assert (g["tiles_m"] - 1) * BM < M <= g["tiles_m"] * BM
    assert (g["tiles_n"] - 1) * BN < N <= g["tiles_n"] * BN
    assert g["kblocks"] == -(-K // BK)
    kps = -(-g["kblocks"] // SK)
    assert (SK - 1) * kps < g["kblocks"]  # no empty split: every partial is real
    ctas = g["tiles_m"] * g["tiles_n"] * SK * pair
    slots = (SMS // pair) * pair
    assert g["grid"] == min(ctas, slots) and g["grid"] % pair == 0
    assert g["waves"] == -(-ctas // slots)
    assert 0 < g["useful_over_padded"] <= 1.0
    assert g["useful_over_padded"] == pytest.approx(
        M * N * K / ((g["tiles_m"] * BM) * (g["tiles_n"] * BN) * (g["kblocks"] * BK)))
    assert 2 <= g["stages"] <= 8
    assert g["smem_bytes"] <= 227 * 1024
    assert g["smem_bytes"] > 227 * 1024 // 2  # one CTA per SM: the 512-column TMEM allocation never contends
    assert g["est_us"] > 0


def test_launch_policy_on_the_benchmark_shapes(lib):
    # the planner's own choice between one and two launches, as measured on GB300: one
    # launch wherever a one-launch plan exists (every benchmark shape)
    expect = {"siglip": 1, "sweep_M729": 1, "tiny": 1, "sweep_M256": 1, "sweep_M1000": 1, "sweep_M4096": 1,
              "sweep_M16384": 1, "sdxl_l2": 1, "sdxl_l1": 1}
    for name, one in expect.items():
        w = wl.WORKLOADS[name]
        assert kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, SMS)["one_launch"] == one, name


def _check_one_launch(info):
    # both projections in one persistent launch: down tiles whole or split along K (never
    # through a cluster: the last CTA of a tile sums its partials), one CTA pairing, one
    # shared-memory ring, at most one unit per resident CTA (pair), never more units than items
    if not info["one_launch"]:
        return
    up, dn = info["up"], info["down"]
    pair = up["BM"] // 128
    assert dn["BM"] == up["BM"] and dn["cluster_sk"] == 0 and info["h_on_chip"] == 0
    assert 1 <= dn["split_k"] <= 4
    assert up["stages"] == dn["stages"] == info["one_launch_stages"] >= 2
    assert up["smem_bytes"] == dn["smem_bytes"] == info["one_launch_smem_bytes"] <= 227 * 1024
    g = info["one_launch_grid"]
    assert g % pair == 0 and g <= (SMS // pair) * pair
    assert g // pair <= up["tiles_m"] * up["tiles_n"] + dn["tiles_m"] * dn["tiles_n"] * dn["split_k"]
    assert info["one_launch_est_us"] > 0


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_planner_invariants_on_every_workload(lib, name):
    w = wl.WORKLOADS[name]
    info = kt_mlp.kt_mlp_plan_info(w.M, w.D, w.F, w.act, w.dtype, w.bias, SMS)
    _check_gemm(info["up"], w.M, w.F, w.D)
    _check_gemm(info["down"], w.M, w.D, w.F)
    _check_one_launch(info)
    assert info["up"]["split_k"] == 1  # the activation is not linear: no split of the up projection
    if w.act == wl.ACT_GEGLU:
        assert info["up"]["BN"] <= 128  # value and gate columns: one MMA of N = 2 BN <= 256


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
@pytest.mark.parametrize("act", [wl.ACT_GELU_SIGMOID, wl.ACT_SILU, None])
def test_planner_invariants_with_pytorch_order_weights(lib, name, act):
    w = wl.WORKLOADS[name]
    a = w.act if act is None else act
    o = kt_mlp.options(w.M, w.D, w.F, a, w.dtype, w.bias, weight_layout=kt_mlp.KT_W_OUT_IN)
    info = kt_mlp.kt_mlp_plan_info_ex(o, SMS)
    _check_gemm(info["up"], w.M, w.F, w.D)
    _check_gemm(info["down"], w.M, w.D, w.F)
    assert info["weight_layout"] == kt_mlp.KT_W_OUT_IN


def _stage_check(g, n_b):
    # one stage holds the CTA's 128 x BK A tile and n_b B tiles of exactly its column share
    # (K-major: BN / pair rows; N-major: 64- or 32-column boxes, no column padded)
    pair = g["BM"] // 128
    share = g["BN"] // pair
    stage = 128 * g["BK"] * 2 + n_b * share * g["BK"] * 2
    reserve = 8 * 2048 + 512 + 2048 + 1024  # staging, barriers, bias, alignment
    # (a second set of output staging buffers where it costs no stage)
    assert g["smem_bytes"] - g["stages"] * stage in (reserve, reserve + 8 * 2048)


def test_weight_tiles_need_no_column_padding_in_shared_memory(lib, monkeypatch):
    # the planner's own choices in both weight orders (the up projection's own ring: two launches)
    monkeypatch.setenv("KT_FORCE_LAUNCHES", "2")
    for M, D, F, act in [(729, 1152, 4304, 1), (2048, 1280, 5120, 2), (8192, 640, 2560, 2)]:
        for layout in (0, 1):
            g = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(M, D, F, act, 0, False, weight_layout=layout), SMS)["up"]
            _stage_check(g, 2 if act == 2 else 1)


@pytest.mark.parametrize("force", ["96,1,64", "160,1,128", "192,2,128", "64,2,64", "32,1,64", "96,2,128",
                                   "32,2,64", "160,2,64"])
def test_n_major_shares_of_odd_multiples_of_32_are_not_padded(lib, monkeypatch, force):
    # column shares of 96, 160, 96, 32 and 32 (32-column boxes instead of padding to 64), and
    # of 48, 16 and 80 (16-column boxes instead of padding to 32)
    monkeypatch.setenv("KT_FORCE_LAUNCHES", "2")
    monkeypatch.setenv("KT_FORCE_UP", force)
    g = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(1000, 1152, 4304, 1, 0, False), SMS)["up"]
    assert (g["BN"], g["BM"] // 128, g["BK"]) == tuple(int(x) for x in force.split(","))
    _stage_check(g, 1)


@pytest.mark.parametrize("act,dtype,bias", [(1, 0, False), (0, 0, True), (2, 1, True)])
@pytest.mark.parametrize("M", [1, 77, 256, 729, 1024, 4096])
def test_auto_launches_once_wherever_one_launch_applies(lib, M, act, dtype, bias):
    # the planner's own choice is one launch exactly when the one-launch planner has a plan
    # (H through memory), and then the same plan as KT_LAUNCH_ONE
    D, F = (1280, 5120) if act == 2 else (1152, 4304)
    auto = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(M, D, F, act, dtype, bias, h_path=kt_mlp.KT_H_MEMORY), SMS)
    try:
        one = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(M, D, F, act, dtype, bias, h_path=kt_mlp.KT_H_MEMORY,
                                                        launches=kt_mlp.KT_LAUNCH_ONE), SMS)
    except kt_mlp.KtError:
        one = None
    assert auto["one_launch"] == (1 if one is not None and one["one_launch"] else 0)
    if auto["one_launch"]:
        for k in ("up", "down"):
            assert auto[k] == one[k]
        assert auto["one_launch_grid"] == one["one_launch_grid"]


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_one_launch_split_items_fit_one_round(lib, name):
    # in one launch, a down projection split along K runs all its items in one round
    w = wl.WORKLOADS[name]
    info = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(w.M, w.D, w.F, w.act, w.dtype, w.bias,
                                                     launches=kt_mlp.KT_LAUNCH_ONE), SMS)
    assert info["one_launch"] == 1
    d = info["down"]
    if d["split_k"] > 1:
        assert d["tiles_m"] * d["tiles_n"] * d["split_k"] <= SMS // (d["BM"] // 128)


@pytest.mark.parametrize("M", [1, 33, 127, 128, 129, 729, 1000, 4097])
@pytest.mark.parametrize("F", [8, 176, 4304])
def test_planner_invariants_on_a_shape_grid(lib, M, F):
    for act in (0, 1, 2, 3):
        info = kt_mlp.kt_mlp_plan_info(M, 1152, F, act, 0, act == 2, SMS)
        _check_gemm(info["up"], M, F, 1152)
        _check_gemm(info["down"], M, 1152, F)


def test_planner_avoids_a_second_wave_on_siglip(lib):
    # M = 729 leaves 6 row tiles; BN = 176 gives 25 column tiles = 150 CTAs <= 152 SMs,
    # where BN = 160 would need 162 (two waves) and BN = 256 wastes a third of the machine
    info = kt_mlp.kt_mlp_plan_info(729, 1152, 4304, 1, 0, False, SMS)
    assert info["up"]["waves"] == 1
    assert info["up"]["grid"] >= 138
    assert info["down"]["waves"] == 1


def test_planner_padding_discount_prefers_less_padding(lib):
    # a problem that fits a 128-wide tile exactly must not be planned on a tile that pads it
    info = kt_mlp.kt_mlp_plan_info(128, 64, 128, 3, 0, False, 1)
    assert info["up"]["useful_over_padded"] == pytest.approx(1.0)


def test_planner_uses_split_k_for_a_deep_narrow_down_projection(lib):
    # D = 128 output columns, F = 16384-deep reduction, M = 128: one output tile,
    # so only split-K can occupy more than one SM
    info = kt_mlp.kt_mlp_plan_info(128, 128, 16384, 3, 0, False, SMS)
    assert info["down"]["split_k"] > 1


def test_h_path_planning(lib):
    on = kt_mlp.KT_H_ON_CHIP
    # the tiny workload's shape fits the fused kernel and the model prefers it
    i = kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(33, 64, 176, 0, 0, False, h_path=kt_mlp.KT_H_AUTO), SMS)
    assert i["h_on_chip"] == 1 and i["fused_grid"] == 1 and 2 <= i["fused_stages"] <= 8
    assert i["fused_smem_bytes"] <= 227 * 1024
    # the default path and kt_mlp_plan write H
    assert kt_mlp.kt_mlp_plan_info(33, 64, 176, 0, 0, False, SMS)["h_on_chip"] == 0
    assert kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(33, 64, 176, 0, 0, False), SMS)["h_on_chip"] == 0
    # where it does not fit: SigLIP's D, GEGLU beyond D = 192, [out][in] weights
    for args, kw in [((729, 1152, 4304, 1, 0, False), {}), ((64, 256, 128, 2, 1, True), {}),
                     ((64, 64, 128, 0, 0, False), {"weight_layout": kt_mlp.KT_W_OUT_IN})]:
        assert kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(*args, h_path=kt_mlp.KT_H_AUTO, **kw), SMS)["h_on_chip"] == 0
        with pytest.raises(kt_mlp.KtError) as e:
            kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(*args, h_path=on, **kw), SMS)
        assert e.value.status == kt_mlp.KT_ERR_UNSUPPORTED
    with pytest.raises(kt_mlp.KtError) as e:
        kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(33, 64, 176, 0, 0, False, h_path=3), SMS)
    assert e.value.status == kt_mlp.KT_ERR_INVALID
    # a wide-D shape with few row blocks stays on the two-kernel path
    assert kt_mlp.kt_mlp_plan_info_ex(kt_mlp.options(8192, 256, 1024, 1, 0, False, h_path=kt_mlp.KT_H_AUTO),
                                      SMS)["h_on_chip"] == 0
