"""Pins of the float64 oracle against things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle -- a dropped term, a
wrong sign or index, a transposed operand, the wrong GELU form, the wrong GEGLU
half, a double rounding -- fails at least one test here:

* codecs: every fp16 / bf16 bit pattern, numpy's float16 conversion, a
  brute-force nearest-value search for bf16, hand-picked ties and overflow;
* GELU: the literal erf and tanh definitions evaluated by mpmath at 120 digits,
  gelu(0) = 0 and the odd-part identity gelu(z) - gelu(-z) = z;
* linear: brute-force scalar loops, the identity matrix, zero padding;
* GEGLU: the explicit split into two GELU-free projections, a zero gate, a
  constant gate, and a swapped-halves check ("SDXL as a requirements
  inventory", sections 1.3 and 9.3);
* the whole MLP: a pure-Python brute force with mpmath activations and
  library / brute-force rounding on tiny shapes, W_down = I, one-hot W_up and
  row subsets;
* the options of a transformer block's feed-forward ("SDXL as a requirements
  inventory", sections 1.3, 1.4, 3 and 9.3): the sigmoid GELU x*sigmoid(1.702 x)
  and SiLU against mpmath, torch's float64 silu and their odd-part identity;
  LayerNorm against a hand-worked row and torch's float64 layer_norm; the residual
  and the [out][in] weight order against the brute force fed [in][out] copies.
"""
import math
import struct

import numpy as np
import pytest

import oracle
from transformer_mlp_gemms_gb300 import workloads as wl

mpmath = pytest.importorskip("mpmath")
mpmath.mp.dps = 120  # the literal forms cancel ~60 digits at z = -12

ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


# --------------------------------------------------------------------------
# codecs
# --------------------------------------------------------------------------

def _bf16_values_by_bits(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_f16_decode_every_pattern_matches_numpy():
    got = oracle.decode(ALL, oracle.F16)
    ref = ALL.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, got[0x8000]) == -1.0


def test_bf16_decode_every_pattern_matches_bit_shift():
    got = oracle.decode(ALL, oracle.BF16)
    ref = _bf16_values_by_bits(ALL)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("dt", [oracle.F16, oracle.BF16])
def test_encode_decode_roundtrip_every_pattern(dt):
    vals = oracle.decode(ALL, dt)
    back = oracle.encode(vals, dt)
    nan = np.isnan(vals)
    assert np.array_equal(back[~nan], ALL[~nan])
    assert np.all(np.isnan(oracle.decode(back[nan], dt)))


def _random_doubles(rng, n, lo_exp, hi_exp):
    mant = rng.uniform(1.0, 2.0, n)
    ex = rng.integers(lo_exp, hi_exp, n)
    sign = rng.choice([-1.0, 1.0], n)
    return sign * np.ldexp(mant, ex)


def test_f16_encode_matches_numpy_direct_rounding():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        _random_doubles(rng, 200000, -30, 17),          # subnormal .. overflow
        rng.standard_normal(100000),
        # exact midpoints between neighbouring fp16 values, both signs
        (lambda v: (v[:-1] + v[1:]) / 2)(np.sort(ALL[:0x7C00].view(np.float16).astype(np.float64))),
    ])
    got = oracle.encode(x, oracle.F16)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encode_matches_bruteforce_nearest_even():
    finite_pos = np.arange(0x0000, 0x7F80, dtype=np.uint32).astype(np.uint16)
    vals = _bf16_values_by_bits(finite_pos)  # strictly increasing
    maxf = vals[-1]
    rng = np.random.default_rng(1)
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([
        np.abs(_random_doubles(rng, 100000, -140, 128)),
        np.abs(rng.standard_normal(50000)),
        mids[rng.choice(mids.size, 20000, replace=False)],
        [maxf, maxf * (1 + 2.0 ** -9), maxf * (1 + 2.0 ** -8.5)],
    ])
    got = oracle.encode(x, oracle.BF16)
    # brute force: nearest representable value, ties to the even pattern,
    # anything at or past the midpoint between maxf and 2^128 becomes +inf
    overflow_mid = (maxf + 2.0 ** 128) / 2
    idx = np.searchsorted(vals, x)
    idx = np.clip(idx, 1, vals.size - 1)
    lo, hi = vals[idx - 1], vals[idx]
    dlo, dhi = x - lo, hi - x
    pick = np.where(dlo < dhi, idx - 1, idx)
    tie = dlo == dhi
    even_lo = (finite_pos[idx - 1] & 1) == 0
    pick = np.where(tie, np.where(even_lo, idx - 1, idx), pick)
    ref = finite_pos[pick].copy()
    ref[x >= overflow_mid] = 0x7F80
    ref[x > maxf] = np.where(x[x > maxf] >= overflow_mid, 0x7F80, 0x7F7F)
    assert np.array_equal(got, ref)
    # negative values are the mirror image
    assert np.array_equal(oracle.encode(-x, oracle.BF16), ref | 0x8000)


def test_hand_picked_ties_overflow_and_subnormals():
    f16 = lambda v: int(oracle.encode(np.array([v]), oracle.F16)[0])
    bf = lambda v: int(oracle.encode(np.array([v]), oracle.BF16)[0])
    assert f16(1.0 + 2.0 ** -11) == 0x3C00           # tie -> even (down)
    assert f16(1.0 + 3 * 2.0 ** -11) == 0x3C02       # tie -> even (up)
    assert f16(65504.0) == 0x7BFF
    assert f16(65519.99) == 0x7BFF
    assert f16(65520.0) == 0x7C00                    # tie at the top rounds to inf
    assert f16(-1e6) == 0xFC00
    assert f16(2.0 ** -24) == 0x0001                 # smallest subnormal
    assert f16(2.0 ** -25) == 0x0000                 # tie with zero -> even (zero)
    assert f16(3 * 2.0 ** -26) == 0x0001
    assert f16(-1.4333e-6) == 0x8018                 # gelu_erf(-5) lands on a subnormal
    assert bf(1.0 + 2.0 ** -8) == 0x3F80
    assert bf(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert bf(2.0 ** -133) == 0x0001
    assert bf(float("inf")) == 0x7F80
    assert np.isnan(oracle.decode(np.array([bf(float("nan"))], dtype=np.uint16), oracle.BF16)[0])


# --------------------------------------------------------------------------
# GELU
# --------------------------------------------------------------------------

def _gelu_erf_mp(z):
    z = mpmath.mpf(z)
    return 0.5 * z * (1 + mpmath.erf(z / mpmath.sqrt(2)))


def _gelu_tanh_mp(z):
    z = mpmath.mpf(z)
    u = mpmath.sqrt(2 / mpmath.pi) * (z + mpmath.mpf("0.044715") * z ** 3)
    return 0.5 * z * (1 + mpmath.tanh(u))


POINTS = [-12.0, -10.0, -7.0, -5.0, -4.0, -3.0, -2.7, -1.0, -0.5, -1e-3, -1e-30,
          0.0, 1e-30, 1e-3, 0.5, 1.0, 1.5, 2.0, 3.0, 5.0, 10.0, 100.0]


@pytest.mark.parametrize("form,ref", [(oracle.GELU_ERF, _gelu_erf_mp), (oracle.GELU_TANH, _gelu_tanh_mp)])
def test_gelu_matches_literal_definition_at_high_precision(form, ref):
    got = oracle.gelu(np.array(POINTS), form)
    for z, g in zip(POINTS, got):
        r = float(ref(z))
        if r == 0.0:
            assert g == 0.0
        else:
            assert abs(g - r) <= 1e-13 * abs(r) + 1e-300, (z, g, r)


def test_gelu_known_values():
    # closed-form values quoted to 15 digits
    e = oracle.gelu(np.array([1.0, -1.0, 0.5, 3.0]), oracle.GELU_ERF)
    assert np.allclose(e, [0.841344746068543, -0.158655253931457, 0.345731230637007,
                           2.995950305905110], rtol=0, atol=5e-15)
    t = oracle.gelu(np.array([1.0, -1.0, 3.0]), oracle.GELU_TANH)
    assert np.allclose(t, [0.841191990608277, -0.158808009391723, 2.996362607918227],
                       rtol=0, atol=5e-15)


@pytest.mark.parametrize("form", [oracle.GELU_ERF, oracle.GELU_TANH])
def test_gelu_odd_part_identity(form):
    z = np.linspace(-8, 8, 4001)
    d = oracle.gelu(z, form) - oracle.gelu(-z, form)
    assert np.max(np.abs(d - z)) < 1e-14 * 8
    assert oracle.gelu(np.array([0.0]), form)[0] == 0.0


def _gelu_sigmoid_mp(z):
    z = mpmath.mpf(z)
    return z / (1 + mpmath.exp(-mpmath.mpf("1.702") * z))


def _silu_mp(z):
    z = mpmath.mpf(z)
    return z / (1 + mpmath.exp(-z))


@pytest.mark.parametrize("form,ref", [(oracle.GELU_SIGMOID, _gelu_sigmoid_mp), (oracle.SILU, _silu_mp)])
def test_sigmoid_forms_match_definition_at_high_precision(form, ref):
    got = oracle.gelu(np.array(POINTS), form)
    for z, g in zip(POINTS, got):
        r = float(ref(z))
        if r == 0.0:
            assert g == 0.0
        else:
            assert abs(g - r) <= 1e-13 * abs(r) + 1e-300, (z, g, r)


def test_silu_matches_torch_float64():
    torch = pytest.importorskip("torch")
    z = np.linspace(-30, 30, 6001)
    ref = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    assert np.allclose(oracle.gelu(z, oracle.SILU), ref, rtol=1e-14, atol=1e-300)


@pytest.mark.parametrize("form", [oracle.GELU_SIGMOID, oracle.SILU])
def test_sigmoid_forms_odd_part_identity(form):
    z = np.linspace(-8, 8, 4001)
    d = oracle.gelu(z, form) - oracle.gelu(-z, form)
    assert np.max(np.abs(d - z)) < 1e-14 * 8
    assert oracle.gelu(np.array([0.0]), form)[0] == 0.0


def test_sigmoid_gelu_is_scaled_silu_and_near_the_erf_form():
    z = np.linspace(-6, 6, 12001)
    sg = oracle.gelu(z, oracle.GELU_SIGMOID)
    assert np.allclose(sg, oracle.gelu(1.702 * z, oracle.SILU) / 1.702, rtol=1e-14, atol=1e-15)
    # the approximation is good to about 2e-2 and no better: it is a different function
    d = np.max(np.abs(sg - oracle.gelu(z, oracle.GELU_ERF)))
    assert 1.5e-2 < d < 2.5e-2


def test_gelu_forms_are_distinguishable():
    z = np.linspace(-6, 6, 120001)
    d = oracle.gelu(z, oracle.GELU_ERF) - oracle.gelu(z, oracle.GELU_TANH)
    i = int(np.argmax(np.abs(d)))
    # the two forms differ by ~4.7e-4 at z ~ -2.7: far above fp32 evaluation noise
    assert 4.5e-4 < abs(d[i]) < 5.0e-4
    assert -2.9 < z[i] < -2.5


# --------------------------------------------------------------------------
# linear
# --------------------------------------------------------------------------

def _brute_linear(A, B, bias):
    M, K = A.shape
    N = B.shape[1]
    C = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s = s + float(A[m, k]) * float(B[k, n])
            if bias is not None:
                s = s + float(bias[n])
            C[m, n] = s
    return C


@pytest.mark.parametrize("M,K,N,with_bias", [(1, 1, 1, False), (3, 5, 4, True), (5, 8, 6, False), (4, 7, 9, True)])
def test_linear_matches_bruteforce_exactly(M, K, N, with_bias):
    rng = np.random.default_rng(M * 100 + K * 10 + N)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N))
    b = rng.standard_normal(N) if with_bias else None
    assert np.array_equal(oracle.linear(A, B, b), _brute_linear(A, B, b))


def test_linear_identity_and_orientation():
    rng = np.random.default_rng(7)
    A = rng.standard_normal((6, 5))
    assert np.array_equal(oracle.linear(A, np.eye(5)), A)
    # a non-square B distinguishes A @ B from A @ B.T and B @ A
    B = np.arange(15, dtype=np.float64).reshape(5, 3)
    C = oracle.linear(np.eye(5)[:2], B)
    assert np.array_equal(C, B[:2])


def test_linear_zero_padding_is_invisible():
    rng = np.random.default_rng(8)
    A = rng.standard_normal((4, 6))
    B = rng.standard_normal((6, 5))
    Ap = np.concatenate([A, np.zeros((4, 3))], axis=1)
    Bp = np.concatenate([B, np.zeros((3, 5))], axis=0)
    assert np.array_equal(oracle.linear(Ap, Bp), oracle.linear(A, B))


# --------------------------------------------------------------------------
# activation step (GELU and GEGLU)
# --------------------------------------------------------------------------

def test_geglu_equals_explicit_split():
    rng = np.random.default_rng(9)
    M, D, F = 5, 7, 6
    X = rng.standard_normal((M, D))
    Wv, Wg = rng.standard_normal((D, F)), rng.standard_normal((D, F))
    bv, bg = rng.standard_normal(F), rng.standard_normal(F)
    P = oracle.linear(X, np.concatenate([Wv, Wg], axis=1), np.concatenate([bv, bg]))
    got = oracle.activation(P, F, oracle.GEGLU)
    value = oracle.linear(X, Wv, bv)
    gate = oracle.linear(X, Wg, bg)
    ref = value * np.array([[float(_gelu_erf_mp(g)) for g in row] for row in gate])
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-300)


def test_geglu_gate_special_cases_and_swapped_halves():
    rng = np.random.default_rng(10)
    M, F = 4, 8
    value = rng.standard_normal((M, F))
    assert np.array_equal(oracle.activation(np.concatenate([value, np.zeros((M, F))], 1), F, oracle.GEGLU),
                          np.zeros((M, F)))
    c = 0.75
    got = oracle.activation(np.concatenate([value, np.full((M, F), c)], 1), F, oracle.GEGLU)
    assert np.allclose(got, value * float(_gelu_erf_mp(c)), rtol=1e-15, atol=0)
    gate = rng.standard_normal((M, F))
    right = oracle.activation(np.concatenate([value, gate], 1), F, oracle.GEGLU)
    wrong = oracle.activation(np.concatenate([gate, value], 1), F, oracle.GEGLU)
    rel = np.abs(right - wrong) / np.max(np.abs(right))
    assert np.median(rel) > 0.05  # gating on the wrong half is grossly wrong


def test_gelu_activation_step_is_elementwise():
    z = np.linspace(-5, 5, 24).reshape(3, 8)
    for form in (oracle.GELU_ERF, oracle.GELU_TANH):
        assert np.array_equal(oracle.activation(z, 8, form), oracle.gelu(z, form))


# --------------------------------------------------------------------------
# the whole MLP
# --------------------------------------------------------------------------

def _round_bits(x, dt):
    """Library / brute-force rounding, independent of the oracle's encoder."""
    if dt == oracle.F16:
        return np.float64(x).astype(np.float16).view(np.uint16)
    finite_pos = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)
    vals = _bf16_values_by_bits(finite_pos)
    a = abs(float(x))
    i = int(np.clip(np.searchsorted(vals, a), 1, vals.size - 1))
    lo, hi = vals[i - 1], vals[i]
    j = i - 1 if (a - lo < hi - a or (a - lo == hi - a and finite_pos[i - 1] % 2 == 0)) else i
    b = int(finite_pos[j])
    return np.uint16(b | (0x8000 if math.copysign(1.0, x) < 0 else 0))


def _dec(b, dt):
    b = np.asarray(b, dtype=np.uint16)
    if dt == oracle.F16:
        return b.view(np.float16).astype(np.float64)
    return _bf16_values_by_bits(b)


def _brute_layernorm_row(row, g, b, eps):
    D = len(row)
    mean = 0.0
    for v in row:
        mean = mean + v
    mean = mean / D
    var = 0.0
    for v in row:
        var = var + (v - mean) * (v - mean)
    var = var / D
    inv = 1.0 / math.sqrt(var + eps)
    return [(row[k] - mean) * inv * g[k] + b[k] for k in range(D)]


def _brute_mlp(X, Wu, Wd, bu, bd, act, dt, R=None, ln=None):
    """Pure-Python MLP: scalar loops, mpmath activations, independent rounding."""
    x, wu, wd = _dec(X, dt), _dec(Wu, dt), _dec(Wd, dt)
    if ln is not None:
        g, b = _dec(ln[0], dt), _dec(ln[1], dt)
        x = np.array([[float(_dec(_round_bits(v, dt), dt)) for v in _brute_layernorm_row(list(r), g, b, ln[2])]
                      for r in x])
    M, D = x.shape
    F = wd.shape[0]
    Fup = wu.shape[1]
    bu_ = _dec(bu, dt) if bu is not None else None
    bd_ = _dec(bd, dt) if bd is not None else None
    H = np.zeros((M, F), dtype=np.uint16)
    Yx = np.zeros((M, D))
    for m in range(M):
        p = []
        for j in range(Fup):
            s = 0.0
            for k in range(D):
                s = s + x[m, k] * wu[k, j]
            if bu_ is not None:
                s = s + bu_[j]
            p.append(s)
        h = []
        for j in range(F):
            if act == oracle.GEGLU:
                v = float(mpmath.mpf(p[j]) * _gelu_erf_mp(p[F + j]))
            elif act == oracle.GELU_TANH:
                v = float(_gelu_tanh_mp(p[j]))
            elif act == oracle.NONE:
                v = p[j]
            elif act == oracle.GELU_SIGMOID:
                v = float(_gelu_sigmoid_mp(p[j]))
            elif act == oracle.SILU:
                v = float(_silu_mp(p[j]))
            else:
                v = float(_gelu_erf_mp(p[j]))
            H[m, j] = _round_bits(v, dt)
            h.append(float(_dec(H[m, j], dt)))
        for n in range(D):
            s = 0.0
            for j in range(F):
                s = s + h[j] * wd[j, n]
            if bd_ is not None:
                s = s + bd_[n]
            if R is not None:
                s = s + float(_dec(R[m, n], dt))
            Yx[m, n] = s
    return H, Yx


CASES = [
    (3, 8, 6, wl.ACT_GELU_ERF, wl.DT_F16, False),
    (4, 8, 8, wl.ACT_GELU_TANH, wl.DT_F16, True),
    (2, 16, 8, wl.ACT_GEGLU, wl.DT_BF16, True),
    (5, 8, 4, wl.ACT_GEGLU, wl.DT_F16, False),
    (3, 8, 16, wl.ACT_GELU_TANH, wl.DT_BF16, False),
    (2, 24, 8, wl.ACT_GELU_ERF, wl.DT_BF16, True),
    (3, 8, 8, wl.ACT_NONE, wl.DT_F16, True),
    (2, 16, 8, wl.ACT_NONE, wl.DT_BF16, False),
]


@pytest.mark.parametrize("M,D,F,act,dt,bias", CASES)
def test_mlp_matches_pure_python_bruteforce(M, D, F, act, dt, bias):
    w = wl.custom(M, D, F, act, dt, bias, seed=100 + M + D + F)
    t = wl.generate(w)
    b = {k: wl.bits(v) for k, v in t.items()}
    H, Yx, Y = oracle.mlp(b["X"], b["W_up"], b["W_down"], b.get("b_up"), b.get("b_down"), act=act, dtype=dt)
    Hb, Yxb = _brute_mlp(b["X"], b["W_up"], b["W_down"], b.get("b_up"), b.get("b_down"), act, dt)
    assert np.array_equal(H, Hb)
    assert np.allclose(Yx, Yxb, rtol=1e-13, atol=1e-15)
    assert np.array_equal(Y, oracle.encode(Yx, dt))


@pytest.mark.parametrize("act", [wl.ACT_GELU_ERF, wl.ACT_GELU_TANH])
def test_mlp_identity_down_projection_returns_h(act):
    M, D = 6, 16
    w = wl.custom(M, D, D, act, wl.DT_F16, False, seed=5)
    t = wl.generate(w)
    X, Wu = wl.bits(t["X"]), wl.bits(t["W_up"])
    I = np.eye(D).astype(np.float16).view(np.uint16)
    H, Yx, Y = oracle.mlp(X, Wu, I, act=act, dtype=wl.DT_F16)
    assert np.array_equal(Y, H)
    assert np.array_equal(Yx, oracle.decode(H, wl.DT_F16))


@pytest.mark.parametrize("act,dt", [(wl.ACT_GELU_ERF, wl.DT_F16), (wl.ACT_GELU_TANH, wl.DT_F16),
                                    (wl.ACT_GELU_ERF, wl.DT_BF16)])
def test_mlp_one_hot_up_projection_is_elementwise_gelu(act, dt):
    # W_up = I makes P = X, so H must be round(gelu(x)) element by element
    M, D = 8, 16
    rng = np.random.default_rng(11)
    xs = np.concatenate([rng.standard_normal(M * D - 6) * 2, [-5.0, -3.0, 0.0, 1.0, 3.0, -7.5]])
    X = oracle.encode(xs.reshape(M, D), dt)
    I = oracle.encode(np.eye(D), dt)
    H, _, _ = oracle.mlp(X, I, I, act=act, dtype=dt)
    ref_fn = _gelu_tanh_mp if act == wl.ACT_GELU_TANH else _gelu_erf_mp
    xd = _dec(X, dt)
    for (m, j), v in np.ndenumerate(xd):
        assert H[m, j] == _round_bits(float(ref_fn(v)), dt), (v,)


def test_mlp_gate_is_second_half():
    # GEGLU with the gate projection forced to a constant c and the value
    # projection = identity: H = round(x * gelu_erf(c)).  Swapping halves
    # (gating on the first) would give round(c * gelu_erf(x)) instead.
    M, D = 4, 8
    rng = np.random.default_rng(12)
    dt = wl.DT_F16
    X = oracle.encode(rng.standard_normal((M, D)), dt)
    Wu = oracle.encode(np.concatenate([np.eye(D), np.zeros((D, D))], 1), dt)
    bu = oracle.encode(np.concatenate([np.zeros(D), np.full(D, 0.75)]), dt)
    bd = oracle.encode(np.zeros(D), dt)
    Wd = oracle.encode(np.eye(D), dt)
    H, _, _ = oracle.mlp(X, Wu, Wd, bu, bd, act=wl.ACT_GEGLU, dtype=dt)
    g = float(_gelu_erf_mp(float(_dec(bu[D], dt))))
    ref = np.array([[_round_bits(float(v) * g, dt) for v in row] for row in _dec(X, dt)])
    assert np.array_equal(H, ref)


def test_mlp_row_subset_equals_full():
    w = wl.custom(37, 32, 48, wl.ACT_GEGLU, wl.DT_BF16, True, seed=13)
    t = wl.generate(w)
    b = {k: wl.bits(v) for k, v in t.items()}
    H, Yx, Y = oracle.mlp(b["X"], b["W_up"], b["W_down"], b["b_up"], b["b_down"], act=w.act, dtype=w.dtype)
    rows = np.array([36, 0, 17, 5])
    Hs, Yxs, Ys = oracle.mlp(b["X"], b["W_up"], b["W_down"], b["b_up"], b["b_down"], act=w.act,
                             dtype=w.dtype, rows=rows)
    assert np.array_equal(Hs, H[rows]) and np.array_equal(Yxs, Yx[rows]) and np.array_equal(Ys, Y[rows])


# --------------------------------------------------------------------------
# LayerNorm, residual and [out][in] weights
# --------------------------------------------------------------------------

def test_layernorm_hand_worked_row():
    # x = 1..4: mean 2.5, biased variance 1.25, so (x - 2.5) / sqrt(1.25) = +-3/sqrt(5), +-1/sqrt(5).
    # An unbiased (D - 1) divisor would give variance 5/3 and fail this.
    out = oracle.layernorm(np.array([[1.0, 2.0, 3.0, 4.0]]), np.ones(4), np.zeros(4), 0.0)[0]
    s = math.sqrt(5.0)
    assert np.allclose(out, [-3 / s, -1 / s, 1 / s, 3 / s], rtol=0, atol=1e-15)
    # gamma scales and beta shifts after the normalisation
    g = np.array([2.0, -1.0, 0.5, 3.0])
    b = np.array([0.25, 0.0, -1.0, 7.0])
    out2 = oracle.layernorm(np.array([[1.0, 2.0, 3.0, 4.0]]), g, b, 0.0)[0]
    assert np.allclose(out2, out * g + b, rtol=0, atol=1e-14)
    # eps enters under the square root: a constant row normalises to beta
    out3 = oracle.layernorm(np.array([[5.0, 5.0, 5.0, 5.0]]), g, b, 1e-5)[0]
    assert np.array_equal(out3, b)


def test_layernorm_matches_torch_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    x = rng.standard_normal((7, 640)) * 3 + 1.5
    g = rng.standard_normal(640)
    b = rng.standard_normal(640)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (640,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    assert np.allclose(oracle.layernorm(x, g, b, 1e-5), ref, rtol=1e-12, atol=1e-12)


OPT_CASES = [
    # M, D, F, act, dt, bias, residual, layernorm, w_layout
    (4, 16, 8, wl.ACT_GELU_SIGMOID, wl.DT_F16, True, True, True, 1),
    (3, 8, 8, wl.ACT_SILU, wl.DT_BF16, False, True, False, 0),
    (2, 16, 8, wl.ACT_GEGLU, wl.DT_BF16, True, True, True, 1),
    (3, 24, 8, wl.ACT_GELU_ERF, wl.DT_F16, False, False, True, 0),
    (2, 8, 16, wl.ACT_GELU_TANH, wl.DT_F16, True, False, False, 1),
]


@pytest.mark.parametrize("M,D,F,act,dt,bias,res,ln,layout", OPT_CASES)
def test_mlp_options_match_pure_python_bruteforce(M, D, F, act, dt, bias, res, ln, layout):
    w = wl.custom(M, D, F, act, dt, bias, seed=200 + M + D + F)
    t = wl.generate(w, residual=res, layernorm=ln)
    b = {k: wl.bits(v) for k, v in t.items()}
    lnarg = (b["ln_gamma"], b["ln_beta"], 1e-5) if ln else None
    Wu, Wd = b["W_up"], b["W_down"]
    if layout == 1:
        Wu_o, Wd_o = np.ascontiguousarray(Wu.T), np.ascontiguousarray(Wd.T)
    else:
        Wu_o, Wd_o = Wu, Wd
    H, Yx, Y = oracle.mlp(b["X"], Wu_o, Wd_o, b.get("b_up"), b.get("b_down"), act=act, dtype=dt,
                          R=b.get("R"), ln=lnarg, w_layout=layout)
    Hb, Yxb = _brute_mlp(b["X"], Wu, Wd, b.get("b_up"), b.get("b_down"), act, dt, R=b.get("R"), ln=lnarg)
    assert np.array_equal(H, Hb)
    assert np.allclose(Yx, Yxb, rtol=1e-13, atol=1e-15)
    assert np.array_equal(Y, oracle.encode(Yx, dt))


def test_weight_order_is_a_pure_transpose():
    w = wl.custom(9, 32, 48, wl.ACT_GEGLU, wl.DT_BF16, True, seed=22)
    t = wl.generate(w)
    b = {k: wl.bits(v) for k, v in t.items()}
    args = (b.get("b_up"), b.get("b_down"))
    ref = oracle.mlp(b["X"], b["W_up"], b["W_down"], *args, act=w.act, dtype=w.dtype)
    got = oracle.mlp(b["X"], np.ascontiguousarray(b["W_up"].T), np.ascontiguousarray(b["W_down"].T), *args,
                     act=w.act, dtype=w.dtype, w_layout=1)
    for r, g in zip(ref, got):
        assert np.array_equal(r, g)
    # the same arrays read in the other order are a different (wrong) problem
    sq = wl.custom(9, 32, 32, wl.ACT_GELU_ERF, wl.DT_F16, False, seed=23)
    ts = {k: wl.bits(v) for k, v in wl.generate(sq).items()}
    a = oracle.mlp(ts["X"], ts["W_up"], ts["W_down"], act=sq.act, dtype=sq.dtype)
    c = oracle.mlp(ts["X"], ts["W_up"], ts["W_down"], act=sq.act, dtype=sq.dtype, w_layout=1)
    assert not np.array_equal(a[0], c[0])


def test_residual_is_added_once_before_the_rounding():
    w = wl.custom(6, 16, 32, wl.ACT_GELU_TANH, wl.DT_F16, False, seed=24)
    t = wl.generate(w, residual=True)
    b = {k: wl.bits(v) for k, v in t.items()}
    H0, Yx0, _ = oracle.mlp(b["X"], b["W_up"], b["W_down"], act=w.act, dtype=w.dtype)
    H1, Yx1, Y1 = oracle.mlp(b["X"], b["W_up"], b["W_down"], act=w.act, dtype=w.dtype, R=b["R"])
    assert np.array_equal(H0, H1)
    r = _dec(b["R"], w.dtype)
    assert np.allclose(Yx1, Yx0 + r, rtol=1e-15, atol=0)
    # a residual that cancels the block's output leaves only the rounding residue
    Rneg = oracle.encode(-Yx0, w.dtype)
    _, Yx2, _ = oracle.mlp(b["X"], b["W_up"], b["W_down"], act=w.act, dtype=w.dtype, R=Rneg)
    assert np.max(np.abs(Yx2)) <= np.max(np.abs(Yx0)) * 2.0 ** -11


def test_mlp_rejects_bad_arguments():
    X = np.zeros((2, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.mlp(X, np.zeros((8, 5), np.uint16), np.zeros((6, 8), np.uint16), act=0, dtype=0)
    with pytest.raises(ValueError):
        oracle.mlp(X, np.zeros((8, 8), np.uint16), np.zeros((8, 8), np.uint16),
                   np.zeros(8, np.uint16), None, act=0, dtype=0)
    W = np.zeros((8, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.mlp(X, W, W, act=6, dtype=0)
    with pytest.raises(ValueError):
        oracle.mlp(X, W, W, act=0, dtype=0, R=np.zeros((3, 8), np.uint16))
    with pytest.raises(ValueError):
        oracle.mlp(X, W, W, act=0, dtype=0, ln=(np.zeros(7, np.uint16), np.zeros(8, np.uint16), 1e-5))
    with pytest.raises(ValueError):
        oracle.mlp(X, np.zeros((8, 16), np.uint16), np.zeros((8, 8), np.uint16), act=2, dtype=0, w_layout=1)
