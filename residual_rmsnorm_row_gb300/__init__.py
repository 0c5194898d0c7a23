"""Row-wise RMSNorm and fused residual Add + RMSNorm for GB300 (sm_103a), forward and backward.

The computation runs in ``librrn.so`` (hand-written CUDA kernels behind the C ABI of
``include/rrn.h``); this package is its Python binding. PyTorch supplies device memory and
streams only.

Two layers:
  * the C entry points under their own names (``rmsnorm_fwd``, ``add_rmsnorm_fwd``,
    ``rmsnorm_bwd`` ...), writing into tensors the caller provides;
  * allocating conveniences (``rms_norm``, ``add_rms_norm``, ``rms_norm_backward``) that
    create the outputs with torch and call the same entry points.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from ._binding import (  # noqa: F401  (re-exported API)
    BF16,
    F32,
    LIBRARY_PATH,
    VARIANT_AUTO,
    VARIANT_NAMES,
    VARIANT_ROW_CLUSTER,
    VARIANT_ROW_CTA,
    VARIANT_ROW_TMA,
    VARIANT_ROW_WARP,
    VARIANT_STREAM,
    Launch,
    RRNError,
    add_rmsnorm_bwd,
    add_rmsnorm_fwd,
    add_rmsnorm_fwd_ex,
    device_faults,
    layernorm_bwd,
    layernorm_bwd_workspace_bytes,
    layernorm_fwd,
    load_library,
    plan_bwd,
    plan_fwd,
    plan_fwd_fp8,
    plan_layernorm_bwd,
    plan_layernorm_fwd,
    rmsnorm_bwd,
    rmsnorm_bwd_ex,
    rmsnorm_bwd_noalloc,
    rmsnorm_bwd_workspace_bytes,
    rmsnorm_fwd,
    rmsnorm_fwd_fp8,
    selftest_wait_timeout,
)


def rms_norm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6,
             stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Return ``(y, rstd)`` for y = x * rstd * w over the last dimension of ``x``."""
    M = x.numel() // x.shape[-1]
    y = torch.empty_like(x)
    rstd = torch.empty(M, device=x.device, dtype=torch.float32)
    rmsnorm_fwd(x, w, y, rstd, eps, stream)
    return y, rstd


def add_rms_norm(x: torch.Tensor, residual: torch.Tensor, w: torch.Tensor, eps: float = 1e-6,
                 inplace: bool = False,
                 stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Return ``(y, residual_out, rstd)``; ``inplace`` writes residual_out into ``residual``."""
    M = x.numel() // x.shape[-1]
    y = torch.empty_like(x)
    residual_out = residual if inplace else torch.empty_like(x)
    rstd = torch.empty(M, device=x.device, dtype=torch.float32)
    add_rmsnorm_fwd(x, residual, residual_out, w, y, rstd, eps, stream)
    return y, residual_out, rstd


def _workspace(M: int, N: int, like: torch.Tensor) -> torch.Tensor:
    nbytes = rmsnorm_bwd_workspace_bytes(M, N, like.dtype)
    return torch.empty(max(nbytes, 16) // 4, device=like.device, dtype=torch.float32)


def rms_norm_backward(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, rstd: torch.Tensor,
                      eps: float = 1e-6, workspace: Optional[torch.Tensor] = None,
                      stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Return ``(dx, dw)``; allocates the dw workspace unless one is given."""
    M, N = x.numel() // x.shape[-1], x.shape[-1]
    dx = torch.empty_like(x)
    dw = torch.empty(N, device=x.device, dtype=torch.float32)
    if workspace is None:
        workspace = _workspace(M, N, x)
    rmsnorm_bwd(dy, x, w, rstd, dx, dw, workspace, eps, stream)
    return dx, dw


def add_rms_norm_backward(dy: torch.Tensor, d_residual_out: Optional[torch.Tensor],
                          residual_out: torch.Tensor, w: torch.Tensor, rstd: torch.Tensor,
                          eps: float = 1e-6, workspace: Optional[torch.Tensor] = None,
                          stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Return ``(d_r, dw)``: the gradient w.r.t. x + residual (both inputs) and w."""
    M, N = residual_out.numel() // residual_out.shape[-1], residual_out.shape[-1]
    d_r = torch.empty_like(residual_out)
    dw = torch.empty(N, device=residual_out.device, dtype=torch.float32)
    if workspace is None:
        workspace = _workspace(M, N, residual_out)
    add_rmsnorm_bwd(dy, d_residual_out, residual_out, w, rstd, d_r, dw, workspace, eps,
                    stream=stream)
    return d_r, dw


def layer_norm(x: torch.Tensor, w: torch.Tensor, b: Optional[torch.Tensor] = None,
               eps: float = 1e-5, residual: Optional[torch.Tensor] = None, stream=None):
    """Return ``(y, mean, rstd)``, or ``(y, residual_out, mean, rstd)`` with ``residual``."""
    M = x.numel() // x.shape[-1]
    y = torch.empty_like(x)
    mean = torch.empty(M, device=x.device, dtype=torch.float32)
    rstd = torch.empty(M, device=x.device, dtype=torch.float32)
    if residual is None:
        layernorm_fwd(x, w, b, y, mean, rstd, eps, stream=stream)
        return y, mean, rstd
    residual_out = torch.empty_like(x)
    layernorm_fwd(x, w, b, y, mean, rstd, eps, residual=residual, residual_out=residual_out,
                  stream=stream)
    return y, residual_out, mean, rstd


def layer_norm_backward(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, mean: torch.Tensor,
                        rstd: torch.Tensor, eps: float = 1e-5,
                        d_residual_out: Optional[torch.Tensor] = None, stream=None):
    """Return ``(dx, dw, db)`` (dx is the gradient w.r.t. x + residual when fused)."""
    M, N = x.numel() // x.shape[-1], x.shape[-1]
    dx = torch.empty_like(x)
    dw = torch.empty(N, device=x.device, dtype=torch.float32)
    db = torch.empty(N, device=x.device, dtype=torch.float32)
    nbytes = layernorm_bwd_workspace_bytes(M, N, x.dtype)
    ws = torch.empty(max(nbytes, 16) // 4, device=x.device, dtype=torch.float32)
    layernorm_bwd(dy, d_residual_out, x, w, mean, rstd, dx, dw, db, ws, eps, stream=stream)
    return dx, dw, db


def rms_norm_fp8(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6,
                 residual: Optional[torch.Tensor] = None, stream=None):
    """Return ``(q, scale)`` (q as torch.float8_e4m3fn) or, with ``residual``,
    ``(q, scale, residual_out)``: RMSNorm(x (+ residual)) * w quantised per row."""
    M = x.numel() // x.shape[-1]
    q = torch.empty(x.shape, device=x.device, dtype=torch.float8_e4m3fn)
    scale = torch.empty(M, device=x.device, dtype=torch.float32)
    ro = torch.empty_like(x) if residual is not None else None
    rmsnorm_fwd_fp8(x, residual, ro, w, q, scale, None, eps, stream=stream)
    return (q, scale) if residual is None else (q, scale, ro)


class RMSNormFunction(torch.autograd.Function):
    """y = RMSNorm(x) * w with the library's forward and backward kernels."""

    @staticmethod
    def forward(ctx, x, w, eps):
        xc = x.contiguous()
        y, rstd = rms_norm(xc, w, eps)
        ctx.save_for_backward(xc, w, rstd)
        ctx.eps = eps
        return y

    @staticmethod
    def backward(ctx, dy):
        x, w, rstd = ctx.saved_tensors
        dx, dw = rms_norm_backward(dy.contiguous(), x, w, rstd, ctx.eps)
        return dx, dw.to(w.dtype), None


class AddRMSNormFunction(torch.autograd.Function):
    """(y, residual_out) = (RMSNorm(x + residual) * w, x + residual) with the library's kernels.

    The backward evaluates the gradient at the stored residual_out (rounded to the storage
    type) with the forward's rstd, as a training framework saves them.
    """

    @staticmethod
    def forward(ctx, x, residual, w, eps):
        y, residual_out, rstd = add_rms_norm(x.contiguous(), residual.contiguous(), w, eps)
        ctx.save_for_backward(residual_out, w, rstd)
        ctx.eps = eps
        return y, residual_out

    @staticmethod
    def backward(ctx, dy, d_residual_out):
        residual_out, w, rstd = ctx.saved_tensors
        if dy is None:
            dy = torch.zeros_like(residual_out)
        d_r, dw = add_rms_norm_backward(
            dy.contiguous(), None if d_residual_out is None else d_residual_out.contiguous(),
            residual_out, w, rstd, ctx.eps)
        return d_r, d_r, dw.to(w.dtype), None


class RMSNorm(torch.nn.Module):
    """RMSNorm over the last dimension; with ``residual`` it is the fused Add + RMSNorm and
    returns ``(y, residual_out)``."""

    def __init__(self, hidden: int, eps: float = 1e-6, dtype=torch.bfloat16, device="cuda"):
        super().__init__()
        self.eps = eps
        self.weight = torch.nn.Parameter(torch.ones(hidden, dtype=dtype, device=device))

    def forward(self, x, residual=None):
        if residual is None:
            return RMSNormFunction.apply(x, self.weight, self.eps)
        return AddRMSNormFunction.apply(x, residual, self.weight, self.eps)


__all__ = [
    "rmsnorm_fwd", "add_rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_workspace_bytes",
    "add_rmsnorm_fwd_ex", "rmsnorm_bwd_ex", "plan_fwd", "plan_bwd", "Launch", "RRNError",
    "load_library", "rms_norm", "add_rms_norm", "rms_norm_backward", "device_faults",
    "add_rmsnorm_bwd", "add_rms_norm_backward", "RMSNormFunction", "AddRMSNormFunction", "RMSNorm",
    "layernorm_fwd", "layernorm_bwd", "layernorm_bwd_workspace_bytes", "layer_norm",
    "layer_norm_backward", "rmsnorm_fwd_fp8", "rms_norm_fp8", "rmsnorm_bwd_noalloc",
    "plan_layernorm_fwd", "plan_layernorm_bwd", "plan_fwd_fp8",
]
