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
    VARIANT_ROW_CTA,
    VARIANT_ROW_WARP,
    VARIANT_STREAM,
    Launch,
    RRNError,
    add_rmsnorm_fwd,
    add_rmsnorm_fwd_ex,
    load_library,
    plan_bwd,
    plan_fwd,
    rmsnorm_bwd,
    rmsnorm_bwd_ex,
    rmsnorm_bwd_workspace_bytes,
    rmsnorm_fwd,
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


def rms_norm_backward(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, rstd: torch.Tensor,
                      eps: float = 1e-6, workspace: Optional[torch.Tensor] = None,
                      stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Return ``(dx, dw)``; allocates the dw workspace unless one is given."""
    M, N = x.numel() // x.shape[-1], x.shape[-1]
    dx = torch.empty_like(x)
    dw = torch.empty(N, device=x.device, dtype=torch.float32)
    if workspace is None:
        nbytes = rmsnorm_bwd_workspace_bytes(M, N, x.dtype)
        workspace = torch.empty(max(nbytes, 16) // 4, device=x.device, dtype=torch.float32)
    rmsnorm_bwd(dy, x, w, rstd, dx, dw, workspace, eps, stream)
    return dx, dw


__all__ = [
    "rmsnorm_fwd", "add_rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_workspace_bytes",
    "add_rmsnorm_fwd_ex", "rmsnorm_bwd_ex", "plan_fwd", "plan_bwd", "Launch", "RRNError",
    "load_library", "rms_norm", "add_rms_norm", "rms_norm_backward",
]
