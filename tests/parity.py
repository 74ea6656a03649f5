"""Comparison helpers for the GPU parity tests (CUDA path vs the float64 oracle).

Tolerances, derived from the arithmetic (and stated once more in the design notes):

* Y: ``|Y_gpu - Yx_oracle| <= 1e-2 * RMS(Yx_oracle) + 1e-3 + ulp_dt(Y)/2`` per element:
  the bar of the specification on the error of the computation, with RMS over the
  compared rows, plus the unavoidable final rounding of Y to the I/O dtype (half an
  ulp), which on its own exceeds 1e-2 * RMS for bf16 outputs beyond ~2.5 RMS.
* H: within 1 ulp of the I/O dtype (ordered bit distance <= 1) wherever the GPU's
  fp32 arithmetic cannot move the value by half an ulp, and within ``ulp + bound``
  elsewhere.  The GPU sums K products in fp32; the classical bound
  |fl(sum) - sum| <= gamma_K * sum |x_k w_k|, gamma_K = K u / (1 - K u), u = 2^-23
  (one ulp: covers truncating adders), is propagated through the activation
  (|gelu'| <= 1.15; GEGLU by the product rule), plus 2^-20 relative for the fp32
  activation itself.  Where that bound is below half an ulp (of the spacing just below
  |H|, the finer one at a power of two), the GPU's pre-rounding value lies within half
  an ulp of the exact one, so the two roundings can differ by one step at most: there
  the check is exact, with no relaxation and no tolerated fraction.
"""
from __future__ import annotations

import numpy as np

import oracle
from transformer_mlp_gemms_gb300 import workloads as wl

U32 = 2.0 ** -23
GELU_SLOPE_MAX = 1.15  # max |d gelu / dz| over the reals is ~1.129 (erf form, z = sqrt 2)


def ulp(x: np.ndarray, dtype: int) -> np.ndarray:
    """Spacing of the I/O dtype at |x| (subnormal spacing below the normal range)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    if dtype == wl.DT_F16:
        fbits, emin = 10, -14
    else:
        fbits, emin = 7, -126
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - fbits).astype(np.int64))


def ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def check_y(Y_gpu_bits: np.ndarray, Yx: np.ndarray, dtype: int, what: str = "Y"):
    y = oracle.decode(Y_gpu_bits, dtype)
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs (unwritten or overflowed)"
    rms = float(np.sqrt(np.mean(Yx * Yx)))
    tol = 1e-2 * rms + 1e-3
    tol_el = tol + 0.5 * ulp(np.abs(Yx) + tol, dtype)
    err = np.abs(y - Yx)
    excess = err - tol_el
    i = int(np.argmax(excess)) if err.size else 0
    assert err.size == 0 or excess.flat[i] <= 0, (
        f"{what}: |err| {err.flat[i]:.3e} > tol {tol_el.flat[i]:.3e} at {np.unravel_index(i, err.shape)} "
        f"(Yx {Yx.flat[i]:.4e}, rms {rms:.3e})")
    return float(err.max()) if err.size else 0.0, tol


def h_bound(w, t_bits: dict, rows=None) -> np.ndarray:
    """Per-element absolute bound of the fp32 accumulation error propagated to H."""
    x = oracle.decode(t_bits["X"], w.dtype)
    if rows is not None:
        x = x[rows]
    wu = oracle.decode(t_bits["W_up"], w.dtype)
    b = oracle.decode(t_bits["b_up"], w.dtype) if w.bias else None
    P = oracle.linear(x, wu, b)
    S = oracle.linear(np.abs(x), np.abs(wu), None if b is None else np.abs(b))
    K = w.D
    gamma = K * U32 / (1 - K * U32)
    E = gamma * S
    F = w.F
    if w.act == wl.ACT_GEGLU:
        v, g = P[:, :F], P[:, F:]
        Ev, Eg = E[:, :F], E[:, F:]
        gg = oracle.gelu(g, oracle.GELU_ERF)
        Hx = v * gg
        bound = np.abs(gg) * Ev + GELU_SLOPE_MAX * (np.abs(v) + Ev) * Eg
    elif w.act == wl.ACT_NONE:
        Hx = P
        bound = E
    else:
        Hx = oracle.gelu(P, oracle.GELU_TANH if w.act == wl.ACT_GELU_TANH else oracle.GELU_ERF)
        bound = GELU_SLOPE_MAX * E
    return bound + 2.0 ** -20 * np.abs(Hx)


def check_h(H_gpu_bits: np.ndarray, H_oracle_bits: np.ndarray, bound: np.ndarray, dtype: int,
            what: str = "H") -> dict:
    """Check H element by element (rule above); return the distance statistics.

    ``strict``: elements whose bound is below half an ulp (the rule allows them one
    step at most); ``beyond_1ulp``: elements more than one step from the oracle
    (each one in the relaxed region, within ulp + bound); ``max_dist``: the largest
    ordered-bit distance.
    """
    d = np.abs(ordered(H_gpu_bits) - ordered(H_oracle_bits))
    hg = oracle.decode(H_gpu_bits, dtype)
    ho = oracle.decode(H_oracle_bits, dtype)
    both_inf = np.isinf(hg) & np.isinf(ho) & (np.sign(hg) == np.sign(ho))
    err = np.where(both_inf, 0.0, np.abs(hg - ho))
    # spacing just below |H|: at a power of two the lower binade's (half as large)
    fine = ulp(np.abs(ho) * (1.0 - 2.0 ** -12), dtype)
    strict = bound < 0.5 * fine
    within1 = d <= 1
    ok = within1 | (~strict & (err <= ulp(ho, dtype) + bound))
    bad = np.argwhere(~ok)
    stats = {"elements": int(d.size), "strict": int(strict.sum()), "beyond_1ulp": int((~within1).sum()),
             "max_dist": int(d.max()) if d.size else 0, "frac_within_1ulp": float(within1.mean()) if d.size else 1.0}
    print(f"{what}: {stats}")
    assert bad.size == 0, (f"{what}: {bad.shape[0]} elements beyond the rule ({stats}); first "
                           f"{[(tuple(i), float(hg[tuple(i)]), float(ho[tuple(i)]), bool(strict[tuple(i)])) for i in bad[:5]]}")
    return stats
