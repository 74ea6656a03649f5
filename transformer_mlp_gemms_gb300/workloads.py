"""Seeded synthetic workloads for the fused MLP (inputs only, no arithmetic of the method).

This module is the one thing the CUDA path's tests and the float64 oracle share:
it draws the inputs.  It computes nothing of the MLP itself.

Shapes follow the pages' workloads:

* ``tiny``     -- a 33 x 64 -> 176 -> 64 GELU MLP (fp16, erf GELU), the small case.
* ``siglip``   -- the F16 SigLIP MLP ``[1,729,1152] -> [1,729,4304] -> [1,729,1152]``
  without biases, tanh GELU ("MLP layout sweep and remaining representation
  limits", opening paragraph and "ISA review").
* ``sdxl_l2`` / ``sdxl_l1`` -- SDXL's GEGLU FeedForward at the 32x32 (d=1280) and
  64x64 (d=640) transformer levels, batch 2 (cond + uncond), hidden 4*d, bf16,
  with biases ("SDXL as a requirements inventory", sections 1.2-1.4).
* ``sweep_M<m>`` -- the SigLIP MLP at M in {256, 729, 1000, 4096, 16384}.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; draw float32 ``randn`` in
the order X, W_up, [b_up], W_down, [b_down]; scale by sqrt(variance) with weight
variance 1/fan_in and bias variance 0.02; cast to the I/O dtype (round to
nearest even).  The same rounded tensors go to the GPU and to the oracle.
Options of the transformer block draw after those, in the order R (the
residual, variance 1, like the residual stream X), LayerNorm gamma
(1 + 0.2 * randn) and beta (0.1 * randn); they never change the tensors above.
Weights are drawn [in][out]; ``torch_order`` returns the [out][in] copies that
PyTorch's nn.Linear stores.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

ACT_GELU_ERF, ACT_GELU_TANH, ACT_GEGLU, ACT_NONE, ACT_GELU_SIGMOID, ACT_SILU = 0, 1, 2, 3, 4, 5
DT_F16, DT_BF16 = 0, 1
ACT_NAMES = {ACT_GELU_ERF: "gelu_erf", ACT_GELU_TANH: "gelu_tanh", ACT_GEGLU: "geglu", ACT_NONE: "none",
             ACT_GELU_SIGMOID: "gelu_sigmoid", ACT_SILU: "silu"}
DT_NAMES = {DT_F16: "f16", DT_BF16: "bf16"}
TORCH_DTYPES = {DT_F16: torch.float16, DT_BF16: torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int          # B of X[B, L, D]
    tokens: int         # L of X[B, L, D]
    D: int              # model dim
    F: int              # hidden dim (GEGLU: projection is 2F wide)
    act: int
    dtype: int
    bias: bool
    seed: int

    @property
    def M(self) -> int:
        return self.batch * self.tokens

    @property
    def F_up(self) -> int:
        return 2 * self.F if self.act == ACT_GEGLU else self.F

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs of one call: 2*M*D*F_up + 2*M*F*D (no padding)."""
        return 2 * self.M * self.D * self.F_up + 2 * self.M * self.F * self.D

    @property
    def io_bytes(self) -> int:
        """Bytes the call must move with H kept on chip: X, weights, biases, Y."""
        e = 2
        n = self.M * self.D + self.D * self.F_up + self.F * self.D + self.M * self.D
        if self.bias:
            n += self.F_up + self.D
        return n * e

    @property
    def h_bytes(self) -> int:
        """Bytes of the intermediate H[M, F] in the I/O dtype."""
        return 2 * self.M * self.F

    def describe(self) -> str:
        return (f"{self.name}: X[{self.batch},{self.tokens},{self.D}] M={self.M} D={self.D} "
                f"F={self.F} act={ACT_NAMES[self.act]} dtype={DT_NAMES[self.dtype]} "
                f"bias={int(self.bias)} seed={self.seed}")


def _sweep(i: int, m: int) -> Workload:
    return Workload(f"sweep_M{m}", 1, m, 1152, 4304, ACT_GELU_TANH, DT_F16, False, 4 + i)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 1, 33, 64, 176, ACT_GELU_ERF, DT_F16, False, 0),
        Workload("siglip", 1, 729, 1152, 4304, ACT_GELU_TANH, DT_F16, False, 1),
        Workload("sdxl_l2", 2, 1024, 1280, 5120, ACT_GEGLU, DT_BF16, True, 2),
        Workload("sdxl_l1", 2, 4096, 640, 2560, ACT_GEGLU, DT_BF16, True, 3),
    ] + [_sweep(i, m) for i, m in enumerate([256, 729, 1000, 4096, 16384])]
}


def custom(M: int, D: int, F: int, act: int, dtype: int, bias: bool, seed: int,
           name: str = "custom") -> Workload:
    return Workload(name, 1, M, D, F, act, dtype, bias, seed)


def generate(w: Workload, residual: bool = False, layernorm: bool = False) -> dict:
    """Seeded CPU tensors for one workload, already rounded to the I/O dtype.

    Returns a dict with X[M,D], W_up[D,F_up], W_down[F,D] and, when ``w.bias``,
    b_up[F_up], b_down[D] (torch tensors on the CPU); with ``residual`` also R[M,D],
    with ``layernorm`` also ln_gamma[D] and ln_beta[D].
    """
    g = torch.Generator("cpu").manual_seed(w.seed)
    dt = TORCH_DTYPES[w.dtype]

    def draw(shape, var):
        return (torch.randn(*shape, generator=g, dtype=torch.float32) * math.sqrt(var)).to(dt)

    out = {"X": draw((w.M, w.D), 1.0), "W_up": draw((w.D, w.F_up), 1.0 / w.D)}
    if w.bias:
        out["b_up"] = draw((w.F_up,), 0.02)
    out["W_down"] = draw((w.F, w.D), 1.0 / w.F)
    if w.bias:
        out["b_down"] = draw((w.D,), 0.02)
    if residual:
        out["R"] = draw((w.M, w.D), 1.0)
    if layernorm:
        out["ln_gamma"] = (1.0 + 0.2 * torch.randn(w.D, generator=g, dtype=torch.float32)).to(dt)
        out["ln_beta"] = draw((w.D,), 0.01)
    return out


def torch_order(t: dict) -> dict:
    """The same tensors with both weights in [out][in] order (contiguous copies)."""
    out = dict(t)
    out["W_up"] = t["W_up"].t().contiguous()
    out["W_down"] = t["W_down"].t().contiguous()
    return out


def bits(t: torch.Tensor) -> np.ndarray:
    """The 16-bit patterns of an fp16/bf16 CPU tensor, as a numpy uint16 array."""
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("expected fp16 or bf16")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(M: int, n: int, seed: int = 0) -> np.ndarray:
    """Row indices for sampled checks at full size: first, last, tile edges, random."""
    fixed = {0, M - 1}
    for edge in (127, 128, 255, 256, M - 128, M - 129):
        if 0 <= edge < M:
            fixed.add(edge)
    rng = np.random.default_rng(seed)
    extra = rng.choice(M, size=min(M, n), replace=False)
    return np.asarray(sorted(fixed | set(int(r) for r in extra)), dtype=np.int64)
