"""Float64 CPU oracle for the fused transformer MLP (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it, and it
shares no code with the CUDA library: ``kt_mlp_oracle.c`` has its own fp16/bf16
codecs, plain loops in natural summation order, and the C library's ``erfc`` /
``exp`` in double precision.

What is computed (see the C file's header for the page citations):

* ``P = X @ W_up (+ b_up)`` in float64,
* ``H~ = gelu(P)`` (erf or tanh form) or, for GEGLU, ``P[:, :F] * gelu_erf(P[:, F:])``
  (value first half, gate second half; "SDXL as a requirements inventory",
  section 1.3 FeedForward),
* ``H = round_dt(H~)`` -- the single rounding of H to the I/O dtype,
* ``Yx = H @ W_down (+ b_down)`` in float64 and ``Y = round_dt(Yx)``.

Parity status of each function is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kt_mlp_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkt_mlp_oracle.so")

F16, BF16 = 0, 1
GELU_ERF, GELU_TANH, GEGLU, NONE, GELU_SIGMOID, SILU = 0, 1, 2, 3, 4, 5

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over rows, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_f16.restype = ctypes.c_uint16
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_decode.argtypes = [u16p, f64p, i64, ctypes.c_int]
        lib.oracle_encode.argtypes = [f64p, u16p, i64, ctypes.c_int]
        lib.oracle_gelu_erf.argtypes = [ctypes.c_double]
        lib.oracle_gelu_erf.restype = ctypes.c_double
        lib.oracle_gelu_tanh.argtypes = [ctypes.c_double]
        lib.oracle_gelu_tanh.restype = ctypes.c_double
        lib.oracle_gelu_vec.argtypes = [f64p, f64p, i64, ctypes.c_int]
        lib.oracle_linear.argtypes = [f64p, f64p, f64p, f64p, i64, i64, i64]
        lib.oracle_activation.argtypes = [f64p, f64p, i64, i64, ctypes.c_int]
        lib.oracle_mlp_rows.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        u16p, u16p, u16p, u16p, u16p,
                                        ctypes.POINTER(ctypes.c_int64), i64, u16p, f64p, u16p]
        lib.oracle_mlp_rows.restype = ctypes.c_int
        lib.oracle_mlp_rows_ex.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           u16p, u16p, u16p, u16p, u16p, u16p, u16p, u16p, ctypes.c_double,
                                           ctypes.c_int, ctypes.POINTER(ctypes.c_int64), i64, u16p, f64p, u16p]
        lib.oracle_mlp_rows_ex.restype = ctypes.c_int
        lib.oracle_layernorm_row.argtypes = [f64p, f64p, f64p, ctypes.c_double, f64p, i64]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bit patterns or float16, got {a.dtype}")
    return a


def num_threads() -> int:
    return _load().oracle_num_threads()


def decode(bits, dtype: int) -> np.ndarray:
    """16-bit patterns of fp16 (dtype=0) or bf16 (dtype=1) -> exact float64."""
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double), b.size, dtype)
    return out


def encode(x, dtype: int) -> np.ndarray:
    """float64 -> 16-bit patterns, IEEE round-to-nearest-even, one rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_encode(_ptr(x, ctypes.c_double), _ptr(out, ctypes.c_uint16), x.size, dtype)
    return out


def gelu(z, form: int) -> np.ndarray:
    """gelu_erf (0), gelu_tanh (1), gelu_sigmoid (4) or silu (5) in float64, elementwise."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    out = np.empty_like(z)
    _load().oracle_gelu_vec(_ptr(z, ctypes.c_double), _ptr(out, ctypes.c_double), z.size, form)
    return out


def linear(A, B, bias=None) -> np.ndarray:
    """float64 ``A[M,K] @ B[K,N] (+ bias[N])``, natural summation order."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    bb = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    if bb is not None and bb.shape != (N,):
        raise ValueError("bias must have shape [N]")
    C = np.empty((M, N), dtype=np.float64)
    _load().oracle_linear(_ptr(A, ctypes.c_double), _ptr(B, ctypes.c_double),
                          _ptr(bb, ctypes.c_double), _ptr(C, ctypes.c_double), M, K, N)
    return C


def activation(P, F: int, act: int) -> np.ndarray:
    """H~ from P: gelu / none (P is [M,F]) or GEGLU (P is [M,2F], gate = second half)."""
    P = np.ascontiguousarray(P, dtype=np.float64)
    M = P.shape[0]
    want = 2 * F if act == GEGLU else F
    if P.shape[1] != want:
        raise ValueError(f"P must be [M,{want}]")
    Hx = np.empty((M, F), dtype=np.float64)
    _load().oracle_activation(_ptr(P, ctypes.c_double), _ptr(Hx, ctypes.c_double), M, F, act)
    return Hx


def layernorm(x, gamma, beta, eps: float) -> np.ndarray:
    """float64 LayerNorm of each row of x (biased variance over the last axis)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(gamma, dtype=np.float64)
    b = np.ascontiguousarray(beta, dtype=np.float64)
    out = np.empty_like(x)
    D = x.shape[-1]
    for i in range(x.shape[0]):
        _load().oracle_layernorm_row(_ptr(x[i], ctypes.c_double), _ptr(g, ctypes.c_double), _ptr(b, ctypes.c_double),
                                     eps, _ptr(out[i], ctypes.c_double), D)
    return out


def mlp(X, W_up, W_down, b_up=None, b_down=None, *, act: int, dtype: int, rows=None,
        R=None, ln=None, w_layout: int = 0):
    """The whole MLP on 16-bit inputs.

    ``X[M,D]``, ``W_up[D,F_up]``, ``W_down[F,D]``, ``b_up[F_up]``, ``b_down[D]``
    are uint16 bit patterns (or float16 arrays for dtype=F16).  ``rows`` (optional)
    selects a subset of rows of X.  Options: ``R[M,D]`` residual added before the
    final rounding; ``ln=(gamma[D], beta[D], eps)`` LayerNorm of X first (rounded to
    the dtype); ``w_layout=1`` weights in [out][in] order (W_up[F_up,D],
    W_down[D,F]).  Returns ``(H_bits[R,F], Yx[R,D] float64, Y_bits[R,D])`` for the R
    selected rows.
    """
    X, W_up, W_down = _u16(X), _u16(W_up), _u16(W_down)
    M, D = X.shape
    F = W_down.shape[1] if w_layout == 1 else W_down.shape[0]
    F_up = 2 * F if act == GEGLU else F
    want_up, want_dn = ((F_up, D), (D, F)) if w_layout == 1 else ((D, F_up), (F, D))
    if W_up.shape != want_up or W_down.shape != want_dn:
        raise ValueError("weight shapes do not match X, act and w_layout")
    Rb = None if R is None else _u16(R)
    if Rb is not None and Rb.shape != (M, D):
        raise ValueError("R must be [M,D]")
    lg = lb = None
    eps = 0.0
    if ln is not None:
        lg, lb, eps = _u16(ln[0]), _u16(ln[1]), float(ln[2])
        if lg.shape != (D,) or lb.shape != (D,):
            raise ValueError("LayerNorm gamma / beta must be [D]")
    bias = b_up is not None or b_down is not None
    if bias:
        if b_up is None or b_down is None:
            raise ValueError("give both biases or neither")
        b_up, b_down = _u16(b_up), _u16(b_down)
        if b_up.shape != (F_up,) or b_down.shape != (D,):
            raise ValueError("bias shapes do not match")
    if rows is None:
        r = None
        NR = M
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        NR = r.size
    H = np.empty((NR, F), dtype=np.uint16)
    Yx = np.empty((NR, D), dtype=np.float64)
    Y = np.empty((NR, D), dtype=np.uint16)
    rc = _load().oracle_mlp_rows_ex(
        M, D, F, act, dtype, 1 if bias else 0,
        _ptr(X, ctypes.c_uint16), _ptr(W_up, ctypes.c_uint16), _ptr(W_down, ctypes.c_uint16),
        _ptr(b_up if bias else None, ctypes.c_uint16), _ptr(b_down if bias else None, ctypes.c_uint16),
        _ptr(Rb, ctypes.c_uint16), _ptr(lg, ctypes.c_uint16), _ptr(lb, ctypes.c_uint16), eps, w_layout,
        _ptr(r, ctypes.c_int64), NR,
        _ptr(H, ctypes.c_uint16), _ptr(Yx, ctypes.c_double), _ptr(Y, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle_mlp_rows rejected its arguments")
    return H, Yx, Y
