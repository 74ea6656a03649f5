"""The GPU parity checks themselves (tests/parity.py), pinned on the CPU.

A mistake planted in the oracle's output must be caught by the same checks the GPU
tests apply: an H element two steps away where the fp32 arithmetic cannot move it by
half an ulp, or a Y element past the tolerance.  One step of H, and Y within the
tolerance, must pass.
"""
import numpy as np
import pytest

import oracle
import parity
from transformer_mlp_gemms_gb300 import workloads as wl


def _case(dtype):
    w = wl.custom(40, 64, 96, wl.ACT_GELU_TANH, dtype, True, seed=17)
    b = {k: wl.bits(v) for k, v in wl.generate(w).items()}
    Ho, Yx, Yb = oracle.mlp(b["X"], b["W_up"], b["W_down"], b["b_up"], b["b_down"], act=w.act, dtype=w.dtype)
    return w, b, Ho, Yx, Yb


def _step(bits, k):
    """Move a 16-bit pattern k steps along the ordered line (sign-magnitude)."""
    o = int(parity.ordered(np.asarray([bits], dtype=np.uint16))[0]) + k
    return np.uint16((0x8000 | -o) if o < 0 else o)


@pytest.mark.parametrize("dtype", [wl.DT_F16, wl.DT_BF16])
def test_check_h_accepts_one_step_and_rejects_two_in_the_strict_region(dtype):
    w, b, Ho, _, _ = _case(dtype)
    bound = parity.h_bound(w, b)
    stats = parity.check_h(Ho.copy(), Ho, bound, dtype)
    assert stats["beyond_1ulp"] == 0 and stats["max_dist"] == 0
    assert stats["strict"] > Ho.size // 2  # at K = 64 most elements are in the strict region
    fine = parity.ulp(np.abs(oracle.decode(Ho, dtype)) * (1 - 2.0 ** -12), dtype)
    strict = np.argwhere(bound < 0.5 * fine)
    i = tuple(strict[len(strict) // 2])
    one = Ho.copy()
    one[i] = _step(one[i], 1)
    assert parity.check_h(one, Ho, bound, dtype)["beyond_1ulp"] == 0
    two = Ho.copy()
    two[i] = _step(two[i], 2)
    with pytest.raises(AssertionError):
        parity.check_h(two, Ho, bound, dtype)


def test_check_h_relaxed_region_uses_the_accumulation_bound():
    w, b, Ho, _, _ = _case(wl.DT_F16)
    # a bound of many ulps everywhere: two steps are allowed, a thousand are not
    big = np.full(Ho.shape, 1e3)
    two = Ho.copy()
    two[3, 5] = _step(two[3, 5], 2)
    assert parity.check_h(two, Ho, big, wl.DT_F16)["beyond_1ulp"] == 1
    small = np.zeros(Ho.shape)
    with pytest.raises(AssertionError):
        parity.check_h(two, Ho, small, wl.DT_F16)


@pytest.mark.parametrize("dtype", [wl.DT_F16, wl.DT_BF16])
def test_check_y_tolerance(dtype):
    _, _, _, Yx, Yb = _case(dtype)
    parity.check_y(Yb, Yx, dtype)  # the oracle's own rounding is within the bar
    rms = float(np.sqrt(np.mean(Yx * Yx)))
    bad = oracle.decode(Yb, dtype).copy()
    bad[7, 11] += 5 * (1e-2 * rms + 1e-3)
    with pytest.raises(AssertionError):
        parity.check_y(oracle.encode(bad, dtype), Yx, dtype)
    nan = Yb.copy()
    nan[0, 0] = 0x7E00  # a NaN pattern in both formats' quiet-NaN range
    with pytest.raises(AssertionError):
        parity.check_y(nan, Yx, dtype)


@pytest.mark.parametrize("dtype,spacing", [(wl.DT_F16, 2.0 ** -24), (wl.DT_BF16, 2.0 ** -133)])
def test_ulp_at_zero_is_the_subnormal_spacing(dtype, spacing):
    # the dtype's spacing at zero (and throughout the subnormal range), not the spacing at 1
    u = parity.ulp(np.array([0.0, -0.0, spacing, 3 * spacing, 1.0]), dtype)
    assert list(u[:4]) == [spacing] * 4
    assert u[4] == (2.0 ** -10 if dtype == wl.DT_F16 else 2.0 ** -7)


def test_check_h_near_zero_uses_the_subnormal_ulp():
    # an oracle zero: a few subnormal steps off is within ulp + bound where the bound is an
    # accumulation error many subnormal steps wide, and rejected where the bound is tiny
    ho = np.zeros((4, 4), dtype=np.uint16)
    hg = ho.copy()
    hg[1, 2] = _step(hg[1, 2], -14)  # -14 subnormal steps (f16: -8.3e-7)
    stats = parity.check_h(hg, ho, np.full(ho.shape, 2e-4), wl.DT_F16)
    assert stats["beyond_1ulp"] == 1 and stats["max_dist"] == 14 and stats["counted"] == 0
    with pytest.raises(AssertionError):
        parity.check_h(hg, ho, np.full(ho.shape, 1e-9), wl.DT_F16)


def test_fraction_floor_counts_elements_away_from_zero_only():
    w, b, Ho, _, _ = _case(wl.DT_F16)
    o = oracle.decode(Ho, wl.DT_F16)
    u = parity.ulp(o, wl.DT_F16)
    # half the elements with a bound of 4 ulps, the other half of 100 ulps (near zero)
    bound = np.where(np.arange(Ho.size).reshape(Ho.shape) % 2 == 0, 4 * u, 100 * u)
    near_zero = np.argwhere(bound > parity.FRACTION_BOUND_ULPS * u)
    counted = np.argwhere(bound < parity.FRACTION_BOUND_ULPS * u)
    many = Ho.copy()
    for ij in near_zero[: Ho.size // 10]:  # 10 % of all elements three steps off, all near zero
        many[tuple(ij)] = _step(many[tuple(ij)], 3)
    stats = parity.check_h(many, Ho, bound, wl.DT_F16)
    assert stats["beyond_1ulp"] == Ho.size // 10 and stats["counted_beyond_1ulp"] == 0
    bad = Ho.copy()
    for ij in counted[: Ho.size // 20]:  # 10 % of the counted elements two steps off, each within ulp + bound
        bad[tuple(ij)] = _step(bad[tuple(ij)], 2)
    with pytest.raises(AssertionError, match="counted_beyond_1ulp"):
        parity.check_h(bad, Ho, bound, wl.DT_F16)
