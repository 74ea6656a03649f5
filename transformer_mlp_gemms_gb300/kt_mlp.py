"""Thin ctypes binding of ``include/kt_mlp.h`` (argument marshalling only).

Every function here has the name of the C entry point it wraps and does no
arithmetic of its own: it converts torch tensors / ints to pointers, the
current torch CUDA stream to a ``cudaStream_t``, and non-OK statuses to
``KtError``.  The library is loaded from the package's in-tree ``_build``
directory; if it is missing the import of a compute entry point fails loudly
(there is no fallback of any kind).
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libkt_mlp.so")

KT_ACT_GELU_ERF, KT_ACT_GELU_TANH, KT_ACT_GEGLU, KT_ACT_NONE, KT_ACT_GELU_SIGMOID, KT_ACT_SILU = range(6)
KT_F16, KT_BF16 = 0, 1
KT_W_IN_OUT, KT_W_OUT_IN = 0, 1
KT_H_AUTO, KT_H_MEMORY, KT_H_ON_CHIP = 0, 1, 2
KT_LAUNCH_AUTO, KT_LAUNCH_ONE, KT_LAUNCH_TWO = 0, 1, 2
KT_ACTIVATION_SCALAR_FORM = 0x100  # kt_debug_activation: the scalar instruction form
KT_OK, KT_ERR_INVALID, KT_ERR_UNSUPPORTED, KT_ERR_CUDA, KT_ERR_TIMEOUT, KT_ERR_NOMEM = range(6)
STATUS_NAMES = {0: "KT_OK", 1: "KT_ERR_INVALID", 2: "KT_ERR_UNSUPPORTED", 3: "KT_ERR_CUDA",
                4: "KT_ERR_TIMEOUT", 5: "KT_ERR_NOMEM"}


class KtError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")


class kt_gemm_plan_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("BM", "BN", "BK", "stages", "split_k", "tiles_m", "tiles_n", "kblocks", "grid", "waves",
                 "smem_bytes", "tmem_cols", "cluster_sk", "b_kmajor")] + \
               [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("useful_over_padded", ctypes.c_double), ("est_us", ctypes.c_double)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class kt_plan_info(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("D", ctypes.c_int64), ("F", ctypes.c_int64),
                ("act", ctypes.c_int32), ("dtype", ctypes.c_int32), ("bias", ctypes.c_int32),
                ("num_sms", ctypes.c_int32),
                ("up", kt_gemm_plan_info), ("down", kt_gemm_plan_info),
                ("workspace_bytes", ctypes.c_int64),
                ("residual", ctypes.c_int32), ("layernorm", ctypes.c_int32), ("weight_layout", ctypes.c_int32),
                ("ln_eps", ctypes.c_float), ("h_on_chip", ctypes.c_int32), ("fused_grid", ctypes.c_int32),
                ("fused_stages", ctypes.c_int32), ("fused_smem_bytes", ctypes.c_int32), ("fused_est_us", ctypes.c_double),
                ("one_launch", ctypes.c_int32), ("one_launch_grid", ctypes.c_int32),
                ("one_launch_stages", ctypes.c_int32), ("one_launch_smem_bytes", ctypes.c_int32),
                ("one_launch_est_us", ctypes.c_double)]

    def as_dict(self):
        d = {n: getattr(self, n) for n, _ in self._fields_ if n not in ("up", "down")}
        d["up"] = self.up.as_dict()
        d["down"] = self.down.as_dict()
        return d


class kt_mlp_options(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("D", ctypes.c_int64), ("F", ctypes.c_int64),
                ("act", ctypes.c_int32), ("dtype", ctypes.c_int32), ("bias", ctypes.c_int32),
                ("residual", ctypes.c_int32), ("layernorm", ctypes.c_int32), ("weight_layout", ctypes.c_int32),
                ("ln_eps", ctypes.c_float), ("h_path", ctypes.c_int32), ("launches", ctypes.c_int32)]


class kt_mlp_tensors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("X", "W_up", "W_down", "b_up", "b_down", "R", "ln_gamma", "ln_beta", "Y", "H_out")]


def options(M, D, F, act, dtype, bias=False, residual=False, layernorm=False, weight_layout=KT_W_IN_OUT,
            ln_eps=1e-5, h_path=KT_H_MEMORY, launches=KT_LAUNCH_AUTO) -> kt_mlp_options:
    return kt_mlp_options(M, D, F, act, dtype, int(bias), int(residual), int(layernorm), weight_layout,
                          ln_eps if layernorm else 0.0, h_path, launches)


def tensors(X, W_up, W_down, Y, b_up=None, b_down=None, R=None, ln_gamma=None, ln_beta=None,
            H_out=None) -> kt_mlp_tensors:
    return kt_mlp_tensors(_ptr(X), _ptr(W_up), _ptr(W_down), _ptr(b_up), _ptr(b_down), _ptr(R), _ptr(ln_gamma),
                          _ptr(ln_beta), _ptr(Y), _ptr(H_out))


_lock = threading.Lock()
_lib = None

# every entry point declared in include/kt_mlp.h, with its ctypes signature
_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
SIGNATURES = {
    "kt_mlp_plan": ([_I64, _I64, _I64, _I32, _I32, _I32, ctypes.POINTER(_VP)], _I32),
    "kt_mlp_run": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], _I32),
    "kt_mlp_plan_ex": ([ctypes.POINTER(kt_mlp_options), ctypes.POINTER(_VP)], _I32),
    "kt_mlp_plan_info_ex": ([ctypes.POINTER(kt_mlp_options), _I32, ctypes.POINTER(kt_plan_info)], _I32),
    "kt_mlp_run_ex": ([_VP, ctypes.POINTER(kt_mlp_tensors), _VP], _I32),
    "kt_mlp_run_ex_timed": ([_VP, ctypes.POINTER(kt_mlp_tensors), _VP, ctypes.POINTER(ctypes.c_float)], _I32),
    "kt_mlp_run_with_h": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], _I32),
    "kt_mlp_run_host": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], _I32),
    "kt_mlp_run_timed": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.POINTER(ctypes.c_float),
                          ctypes.POINTER(ctypes.c_float)], _I32),
    "kt_mlp_status": ([_VP], _I32),
    "kt_mlp_destroy": ([_VP], _I32),
    "kt_mlp_describe": ([_VP, ctypes.c_char_p, ctypes.c_size_t], _I32),
    "kt_mlp_get_info": ([_VP, ctypes.POINTER(kt_plan_info)], _I32),
    "kt_mlp_plan_info": ([_I64, _I64, _I64, _I32, _I32, _I32, _I32, ctypes.POINTER(kt_plan_info)], _I32),
    "kt_mlp_debug_stall": ([_VP, _I32, _I64], _I32),
    "kt_mlp_debug_trace": ([_VP, _VP, _VP], _I32),
    "kt_debug_timestamp": ([_VP, _VP], _I32),
    "kt_debug_activation": ([_I32, _VP, _VP, _VP, _I64, _VP], _I32),
    "kt_down_proj_noalloc": ([_I64, _I64, _I64, _I32, _VP, _VP, _VP, _VP, _VP], _I32),
    "kt_last_error": ([], ctypes.c_char_p),
    "kt_mlp_abi_version": ([], _I32),
}


def load(path: str | None = None):
    """Load the shared library once (raises OSError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise OSError(f"{p} not found: build it with `python -m transformer_mlp_gemms_gb300.build`")
        lib = ctypes.CDLL(p)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != KT_OK:
        raise KtError(status, where, load().kt_last_error().decode(errors="replace"))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a tensor, an int address or None, got {type(x)}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kt_mlp_abi_version() -> int:
    return load().kt_mlp_abi_version()


def kt_last_error() -> str:
    return load().kt_last_error().decode(errors="replace")


def kt_mlp_plan(M: int, D: int, F: int, act: int, dtype: int, bias: bool) -> int:
    out = _VP()
    _check(load().kt_mlp_plan(M, D, F, act, dtype, int(bias), ctypes.byref(out)), "kt_mlp_plan")
    return out.value


def kt_mlp_plan_ex(opts: kt_mlp_options) -> int:
    out = _VP()
    _check(load().kt_mlp_plan_ex(ctypes.byref(opts), ctypes.byref(out)), "kt_mlp_plan_ex")
    return out.value


def kt_mlp_plan_info_ex(opts: kt_mlp_options, num_sms: int) -> dict:
    info = kt_plan_info()
    _check(load().kt_mlp_plan_info_ex(ctypes.byref(opts), num_sms, ctypes.byref(info)), "kt_mlp_plan_info_ex")
    return info.as_dict()


def kt_mlp_run_ex(plan: int, t: kt_mlp_tensors, stream=None) -> None:
    _check(load().kt_mlp_run_ex(plan, ctypes.byref(t), _stream(stream)), "kt_mlp_run_ex")


def kt_mlp_run_ex_timed(plan: int, t: kt_mlp_tensors, stream=None):
    """Returns (ms_layernorm, ms_up, ms_down): device time of each kernel (CUDA events)."""
    ms = (ctypes.c_float * 3)()
    _check(load().kt_mlp_run_ex_timed(plan, ctypes.byref(t), _stream(stream), ms), "kt_mlp_run_ex_timed")
    return ms[0], ms[1], ms[2]


def kt_mlp_run(plan: int, X, W_up, W_down, b_up, b_down, Y, stream=None) -> None:
    _check(load().kt_mlp_run(plan, _ptr(X), _ptr(W_up), _ptr(W_down), _ptr(b_up), _ptr(b_down), _ptr(Y),
                             _stream(stream)), "kt_mlp_run")


def kt_mlp_run_with_h(plan: int, X, W_up, W_down, b_up, b_down, Y, H_out, stream=None) -> None:
    _check(load().kt_mlp_run_with_h(plan, _ptr(X), _ptr(W_up), _ptr(W_down), _ptr(b_up), _ptr(b_down),
                                    _ptr(Y), _ptr(H_out), _stream(stream)), "kt_mlp_run_with_h")


def kt_mlp_run_host(plan: int, X_host, W_up, W_down, b_up, b_down, Y_host, stream=None) -> None:
    _check(load().kt_mlp_run_host(plan, _ptr(X_host), _ptr(W_up), _ptr(W_down), _ptr(b_up), _ptr(b_down),
                                  _ptr(Y_host), _stream(stream)), "kt_mlp_run_host")


def kt_mlp_run_timed(plan: int, X, W_up, W_down, b_up, b_down, Y, stream=None):
    """Returns (ms_up, ms_down): device time of each kernel, measured with CUDA events."""
    a, b = ctypes.c_float(), ctypes.c_float()
    _check(load().kt_mlp_run_timed(plan, _ptr(X), _ptr(W_up), _ptr(W_down), _ptr(b_up), _ptr(b_down),
                                   _ptr(Y), _stream(stream), ctypes.byref(a), ctypes.byref(b)),
           "kt_mlp_run_timed")
    return a.value, b.value


def kt_mlp_status(plan: int) -> int:
    """Returns the status code (does not raise on KT_ERR_TIMEOUT)."""
    return load().kt_mlp_status(plan)


def kt_mlp_destroy(plan: int) -> None:
    _check(load().kt_mlp_destroy(plan), "kt_mlp_destroy")


def kt_mlp_describe(plan: int) -> str:
    buf = ctypes.create_string_buffer(1024)
    _check(load().kt_mlp_describe(plan, buf, len(buf)), "kt_mlp_describe")
    return buf.value.decode()


def kt_mlp_get_info(plan: int) -> dict:
    info = kt_plan_info()
    _check(load().kt_mlp_get_info(plan, ctypes.byref(info)), "kt_mlp_get_info")
    return info.as_dict()


def kt_mlp_plan_info(M: int, D: int, F: int, act: int, dtype: int, bias: bool, num_sms: int) -> dict:
    info = kt_plan_info()
    _check(load().kt_mlp_plan_info(M, D, F, act, dtype, int(bias), num_sms, ctypes.byref(info)),
           "kt_mlp_plan_info")
    return info.as_dict()


def kt_mlp_debug_stall(plan: int, enable: bool, limit_us: int = 0) -> None:
    _check(load().kt_mlp_debug_stall(plan, int(bool(enable)), limit_us), "kt_mlp_debug_stall")


def kt_mlp_debug_trace(plan: int, trace_up=None, trace_down=None) -> None:
    _check(load().kt_mlp_debug_trace(plan, _ptr(trace_up), _ptr(trace_down)), "kt_mlp_debug_trace")


def kt_debug_activation(act: int, z, gate, out, n: int, stream=None) -> None:
    _check(load().kt_debug_activation(act, _ptr(z), _ptr(gate), _ptr(out), n, _stream(stream)),
           "kt_debug_activation")


def kt_down_proj_noalloc(M: int, F: int, D: int, dtype: int, H, W_down, b_down, Y, stream=None) -> None:
    """The down projection without any device allocation (static 16 MiB scratch per device)."""
    _check(load().kt_down_proj_noalloc(M, F, D, dtype, _ptr(H), _ptr(W_down), _ptr(b_down), _ptr(Y),
                                       _stream(stream)), "kt_down_proj_noalloc")


def kt_debug_timestamp(dst, stream=None) -> None:
    _check(load().kt_debug_timestamp(_ptr(dst), _stream(stream)), "kt_debug_timestamp")


class Plan:
    """Owning handle: ``Plan(M, D, F, act, dtype, bias)`` (kt_mlp_plan), or with any of
    ``residual``, ``layernorm``, ``weight_layout``, ``ln_eps``, ``h_path``, ``launches``
    (kt_mlp_plan_ex); destroyed with the object."""

    def __init__(self, M, D, F, act, dtype, bias, residual=False, layernorm=False, weight_layout=KT_W_IN_OUT,
                 ln_eps=1e-5, h_path=KT_H_MEMORY, launches=KT_LAUNCH_AUTO):
        self.M, self.D, self.F, self.act, self.dtype, self.bias = M, D, F, act, dtype, bool(bias)
        self.residual, self.layernorm, self.weight_layout = bool(residual), bool(layernorm), weight_layout
        if residual or layernorm or weight_layout != KT_W_IN_OUT or h_path != KT_H_MEMORY or launches:
            self.handle = kt_mlp_plan_ex(options(M, D, F, act, dtype, bias, residual, layernorm, weight_layout,
                                                 ln_eps, h_path, launches))
        else:
            self.handle = kt_mlp_plan(M, D, F, act, dtype, bias)

    def run_ex(self, X, W_up, W_down, Y, b_up=None, b_down=None, R=None, ln_gamma=None, ln_beta=None,
               H_out=None, stream=None):
        kt_mlp_run_ex(self.handle, tensors(X, W_up, W_down, Y, b_up, b_down, R, ln_gamma, ln_beta, H_out), stream)

    def run_ex_timed(self, X, W_up, W_down, Y, b_up=None, b_down=None, R=None, ln_gamma=None, ln_beta=None,
                     stream=None):
        return kt_mlp_run_ex_timed(self.handle, tensors(X, W_up, W_down, Y, b_up, b_down, R, ln_gamma, ln_beta),
                                   stream)

    def run(self, X, W_up, W_down, b_up, b_down, Y, stream=None):
        kt_mlp_run(self.handle, X, W_up, W_down, b_up, b_down, Y, stream)

    def run_with_h(self, X, W_up, W_down, b_up, b_down, Y, H, stream=None):
        kt_mlp_run_with_h(self.handle, X, W_up, W_down, b_up, b_down, Y, H, stream)

    def run_host(self, X_host, W_up, W_down, b_up, b_down, Y_host, stream=None):
        kt_mlp_run_host(self.handle, X_host, W_up, W_down, b_up, b_down, Y_host, stream)

    def run_timed(self, X, W_up, W_down, b_up, b_down, Y, stream=None):
        return kt_mlp_run_timed(self.handle, X, W_up, W_down, b_up, b_down, Y, stream)

    def status(self) -> int:
        return kt_mlp_status(self.handle)

    def describe(self) -> str:
        return kt_mlp_describe(self.handle)

    def info(self) -> dict:
        return kt_mlp_get_info(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            kt_mlp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
