"""Seeded synthetic workloads for row-wise RMSNorm / fused residual Add + RMSNorm.

This module only draws random inputs. It contains none of the normalisation arithmetic, so
both the GPU path's tests/benchmark and the CPU oracle can take their inputs from it.

Every workload is drawn on the host with numpy's PCG64 generator, seeded per workload, in a
fixed order: x, residual, (outlier mask, outlier sign), w, b, dy, d_ro. Values are drawn in float32
and, for bf16 workloads, rounded to bf16 (round to nearest even) by torch's CPU cast. bf16
tensors are returned as ``uint16`` arrays holding the raw bit patterns; fp32 tensors as
``float32`` arrays.

The pages name benchmark suites for this op (Quack-suite, DeepSeek-V3/V4 norm workloads on the
KernelAgent page) whose shapes are not published there; the shapes below stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, Optional

import numpy as np

BF16 = "bf16"
F32 = "f32"


@dataclass(frozen=True)
class Workload:
    """One synthetic problem: op kind, shape, dtype, eps, seed and value distributions."""

    name: str
    op: str                      # rmsnorm_fwd | add_rmsnorm_fwd | rmsnorm_bwd | add_rmsnorm_bwd |
                                 # layernorm_fwd | add_layernorm_fwd | layernorm_bwd |
                                 # add_rmsnorm_fp8
    M: int
    N: int
    dtype: str                   # "bf16" | "f32"
    eps: float
    seed: int
    x_sigma: float = 1.0         # x ~ N(x_mean, x_sigma^2)
    x_mean: float = 0.0
    res_sigma: float = 1.0       # residual ~ N(0, res_sigma^2)
    outlier_frac: float = 0.0    # fraction of residual entries replaced by +/- outlier_value
    outlier_value: float = 50.0
    w_kind: str = "normal"       # "normal": 1 + 0.1*N(0,1); "uniform": U(0.5, 1.5)
    residual_grad: bool = True   # layernorm_bwd: a gradient arrives at residual_out (d_ro)
    meta: Dict[str, str] = field(default_factory=dict)

    def with_shape(self, M: int, N: Optional[int] = None) -> "Workload":
        return replace(self, M=M, N=self.N if N is None else N,
                       name=f"{self.name}@{M}x{self.N if N is None else N}")

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4


# The workloads. Names give op, shape and dtype.
WORKLOADS: Dict[str, Workload] = {}


def _add(w: Workload) -> None:
    WORKLOADS[w.name] = w


_add(Workload("rmsnorm_fwd_256x1024_bf16", "rmsnorm_fwd", 256, 1024, BF16, 1e-6, 0))
_add(Workload("add_rmsnorm_fwd_4096x4096_bf16", "add_rmsnorm_fwd", 4096, 4096, BF16, 1e-6, 1))
_add(Workload("add_rmsnorm_fwd_16384x4096_bf16", "add_rmsnorm_fwd", 16384, 4096, BF16, 1e-6, 1))
_add(Workload("add_rmsnorm_fwd_16384x7168_bf16", "add_rmsnorm_fwd", 16384, 7168, BF16, 1e-6, 2,
              res_sigma=2.0, outlier_frac=0.01, outlier_value=50.0, w_kind="uniform"))
for _dt in (BF16, F32):
    for _m in (1, 8, 32, 64):
        _add(Workload(f"rmsnorm_fwd_{_m}x8192_{_dt}", "rmsnorm_fwd", _m, 8192, _dt, 1e-5, 3))
    _add(Workload(f"rmsnorm_fwd_65536x2048_{_dt}", "rmsnorm_fwd", 65536, 2048, _dt, 1e-5, 3))
_add(Workload("rmsnorm_bwd_16384x4096_bf16", "rmsnorm_bwd", 16384, 4096, BF16, 1e-6, 4))
# The fused backward: x plays the stored residual_out; dy and d_ro are the gradients arriving at
# y and at residual_out.
_add(Workload("add_rmsnorm_bwd_16384x4096_bf16", "add_rmsnorm_bwd", 16384, 4096, BF16, 1e-6, 5))
# LayerNorm (mean-subtracting variant): x ~ N(0.5, 1), bias b ~ 0.1 N(0,1); the backward draws
# dy and the gradient at residual_out like the fused RMSNorm backward.
_add(Workload("add_layernorm_fwd_16384x4096_bf16", "add_layernorm_fwd", 16384, 4096, BF16, 1e-5, 6,
              x_mean=0.5))
_add(Workload("layernorm_bwd_16384x4096_bf16", "layernorm_bwd", 16384, 4096, BF16, 1e-5, 7,
              x_mean=0.5))
# The plain LayerNorm backward (no gradient at residual_out: two input rows, as RMSNorm's).
_add(Workload("layernorm_bwd_plain_16384x4096_bf16", "layernorm_bwd", 16384, 4096, BF16, 1e-5, 14,
              x_mean=0.5, residual_grad=False))
# The fused Add+RMSNorm feeding fp8 e4m3 codes with a per-row scale (inputs as the fused forward).
_add(Workload("add_rmsnorm_fp8_16384x4096_bf16", "add_rmsnorm_fp8", 16384, 4096, BF16, 1e-6, 8))
# Rows wider than one CTA holds in registers: split over a thread-block cluster (16384 wide: 4
# CTAs; 65536 wide: 8).
_add(Workload("add_rmsnorm_fwd_16384x16384_bf16", "add_rmsnorm_fwd", 16384, 16384, BF16, 1e-6, 9))
_add(Workload("add_rmsnorm_fwd_4096x65536_bf16", "add_rmsnorm_fwd", 4096, 65536, BF16, 1e-6, 9))
# The backward of rows too wide for one CTA's registers (each row split over a cluster).
_add(Workload("rmsnorm_bwd_8192x16384_bf16", "rmsnorm_bwd", 8192, 16384, BF16, 1e-6, 10))
_add(Workload("add_rmsnorm_bwd_8192x16384_bf16", "add_rmsnorm_bwd", 8192, 16384, BF16, 1e-6, 11))
_add(Workload("layernorm_bwd_8192x16384_bf16", "layernorm_bwd", 8192, 16384, BF16, 1e-5, 12,
              x_mean=0.5))
# The fp8 output of wide rows (split over a cluster).
_add(Workload("add_rmsnorm_fp8_16384x16384_bf16", "add_rmsnorm_fp8", 16384, 16384, BF16, 1e-6, 13))
# Short rows over many rows (one row per warp: the LayerNorm and fp8 forwards, the RMSNorm and
# LayerNorm backwards) and a LayerNorm forward of 8192 columns (a CTA of 4 vectors a thread).
_add(Workload("add_layernorm_fwd_65536x1024_bf16", "add_layernorm_fwd", 65536, 1024, BF16, 1e-5, 15,
              x_mean=0.5))
_add(Workload("add_layernorm_fwd_8192x8192_bf16", "add_layernorm_fwd", 8192, 8192, BF16, 1e-5, 16,
              x_mean=0.5))
_add(Workload("add_rmsnorm_fp8_65536x1024_bf16", "add_rmsnorm_fp8", 65536, 1024, BF16, 1e-6, 17))
_add(Workload("rmsnorm_bwd_131072x512_bf16", "rmsnorm_bwd", 131072, 512, BF16, 1e-6, 18))
_add(Workload("layernorm_bwd_plain_65536x1024_bf16", "layernorm_bwd", 65536, 1024, BF16, 1e-5, 19,
              x_mean=0.5, residual_grad=False))


def get(name: str) -> Workload:
    return WORKLOADS[name]


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even) with torch's CPU cast; return the bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _store(a: np.ndarray, dtype: str) -> np.ndarray:
    return to_bf16_bits(a) if dtype == BF16 else np.ascontiguousarray(a, dtype=np.float32)


def make(w: Workload) -> Dict[str, np.ndarray]:
    """Draw the host inputs of ``w``: x, w and, per op, residual or dy.

    The result maps tensor names to host arrays in the workload's storage encoding (uint16
    bf16 bits or float32). For the fused op it also holds ``outliers``, the number of
    residual entries replaced by outliers.
    """
    rng = np.random.default_rng(w.seed)
    shape = (w.M, w.N)
    out: Dict[str, np.ndarray] = {}
    x = rng.standard_normal(shape, dtype=np.float32)
    if w.x_sigma != 1.0:
        x *= np.float32(w.x_sigma)
    if w.x_mean != 0.0:
        x += np.float32(w.x_mean)
    out["x"] = _store(x, w.dtype)
    del x
    if w.op in ("add_rmsnorm_fwd", "add_layernorm_fwd", "add_rmsnorm_fp8"):
        res = rng.standard_normal(shape, dtype=np.float32)
        if w.res_sigma != 1.0:
            res *= np.float32(w.res_sigma)
        if w.outlier_frac > 0.0:
            mask = rng.random(shape, dtype=np.float32) < w.outlier_frac
            sign = rng.integers(0, 2, size=shape, dtype=np.int8)
            res[mask] = np.where(sign[mask] == 1, w.outlier_value, -w.outlier_value)
            out["outliers"] = np.array(int(mask.sum()))
            del mask, sign
        out["residual"] = _store(res, w.dtype)
        del res
    if w.w_kind == "uniform":
        wt = rng.uniform(0.5, 1.5, size=w.N).astype(np.float32)
    else:
        wt = (np.float32(1.0) + np.float32(0.1) * rng.standard_normal(w.N, dtype=np.float32))
    out["w"] = _store(wt, w.dtype)
    if w.op.startswith(("layernorm", "add_layernorm")):
        out["b"] = _store(np.float32(0.1) * rng.standard_normal(w.N, dtype=np.float32), w.dtype)
    if w.op in ("rmsnorm_bwd", "add_rmsnorm_bwd", "layernorm_bwd"):
        out["dy"] = _store(rng.standard_normal(shape, dtype=np.float32), w.dtype)
    if w.op == "add_rmsnorm_bwd" or (w.op == "layernorm_bwd" and w.residual_grad):
        out["d_ro"] = _store(rng.standard_normal(shape, dtype=np.float32), w.dtype)
    return out


def min_bytes(w: Workload) -> int:
    """Minimum HBM bytes one call moves: every input read once, every output written once.

    rmsnorm_fwd: x, y (M*N each), w (N), rstd (M, fp32).
    add_rmsnorm_fwd: x, residual, residual_out, y (M*N each), w (N), rstd (M, fp32).
    rmsnorm_bwd: x, dy, dx (M*N each), w (N), rstd (M, fp32), dw (N, fp32).
    add_rmsnorm_bwd: residual_out, dy, d_residual_out, d_r (M*N each), w, rstd, dw.
    add_layernorm_fwd: x, residual, residual_out, y (M*N each), w, b (N), mean, rstd (M, fp32).
    layernorm_bwd: x, dy, d_residual_out (when residual_grad), dx (M*N each), w (N), mean, rstd
    (M), dw, db (N, fp32).
    add_rmsnorm_fp8: x, residual, residual_out (M*N each), the codes (M*N bytes), w (N),
    scale (M, fp32).
    """
    e = w.elem_bytes
    if w.op == "rmsnorm_fwd":
        return 2 * w.M * w.N * e + w.N * e + 4 * w.M
    if w.op == "add_rmsnorm_fwd":
        return 4 * w.M * w.N * e + w.N * e + 4 * w.M
    if w.op == "rmsnorm_bwd":
        return 3 * w.M * w.N * e + w.N * e + 4 * w.M + 4 * w.N
    if w.op == "add_rmsnorm_bwd":
        return 4 * w.M * w.N * e + w.N * e + 4 * w.M + 4 * w.N
    if w.op == "add_layernorm_fwd":
        return 4 * w.M * w.N * e + 2 * w.N * e + 8 * w.M
    if w.op == "layernorm_bwd":
        return (4 if w.residual_grad else 3) * w.M * w.N * e + w.N * e + 8 * w.M + 8 * w.N
    if w.op == "add_rmsnorm_fp8":
        return 3 * w.M * w.N * e + w.M * w.N + w.N * e + 4 * w.M
    raise ValueError(w.op)


__all__ = ["Workload", "WORKLOADS", "get", "make", "min_bytes", "to_bf16_bits", "BF16", "F32"]
