"""ctypes binding of ``librrn.so`` (C ABI in ``include/rrn.h``): argument marshalling only.

Each function here has the name of the C entry point it calls, takes torch CUDA tensors,
passes their device pointers, sizes and the stream to the library, and raises ``RRNError``
on a nonzero status. No arithmetic of the operation happens in Python; there is no CPU
fallback - if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "librrn.so")

BF16, F32 = 0, 1
_DTYPES = {torch.bfloat16: BF16, torch.float32: F32}

(VARIANT_AUTO, VARIANT_ROW_CTA, VARIANT_ROW_WARP, VARIANT_STREAM, VARIANT_ROW_TMA,
 VARIANT_ROW_CLUSTER) = range(6)
VARIANT_NAMES = {VARIANT_ROW_CTA: "row_cta", VARIANT_ROW_WARP: "row_warp",
                 VARIANT_STREAM: "stream", VARIANT_ROW_TMA: "row_tma",
                 VARIANT_ROW_CLUSTER: "row_cluster"}

STATUS_NAMES = {0: "RRN_OK", 1: "RRN_ERR_NULL", 2: "RRN_ERR_SHAPE", 3: "RRN_ERR_EPS",
                4: "RRN_ERR_DTYPE", 5: "RRN_ERR_ALIGN", 6: "RRN_ERR_WORKSPACE",
                7: "RRN_ERR_CUDA", 8: "RRN_ERR_CONFIG", 9: "RRN_ERR_SCRATCH"}


class RRNError(RuntimeError):
    """A nonzero rrn_status from the library."""

    def __init__(self, status: int, message: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        extra = f" (cudaError {cuda_error})" if status == 7 else ""
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}{extra}")


class rrn_launch(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("vpt", ctypes.c_int), ("threads", ctypes.c_int),
                ("ctas", ctypes.c_int), ("stages", ctypes.c_int), ("cluster", ctypes.c_int),
                ("vec", ctypes.c_int)]


@dataclass(frozen=True)
class Launch:
    """A launch configuration (0 = automatic), mirroring ``rrn_launch``."""

    variant: int = 0
    vpt: int = 0
    threads: int = 0
    ctas: int = 0
    stages: int = 0
    cluster: int = 0
    vec: int = 0

    def to_c(self) -> rrn_launch:
        return rrn_launch(self.variant, self.vpt, self.threads, self.ctas, self.stages,
                          self.cluster, self.vec)

    @staticmethod
    def from_c(c: rrn_launch) -> "Launch":
        return Launch(c.variant, c.vpt, c.threads, c.ctas, c.stages, c.cluster, c.vec)

    @property
    def name(self) -> str:
        base = VARIANT_NAMES.get(self.variant, "auto")
        st = f",stages={self.stages}" if self.variant == VARIANT_ROW_TMA else ""
        st += f",cluster={self.cluster}" if self.cluster > 1 else ""
        return f"{base}(vpt={self.vpt},threads={self.threads},ctas={self.ctas}{st},vec={self.vec})"


_LIB: Optional[ctypes.CDLL] = None

_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_size_t)
_SIGNATURES = {
    "rmsnorm_fwd": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32, _vp]),
    "add_rmsnorm_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32, _vp]),
    "rmsnorm_bwd_workspace_bytes": (_i32, [_i64, _i64, _i32, ctypes.POINTER(_sz)]),
    "rmsnorm_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _f32, _i32, _vp]),
    "rrn_status_string": (ctypes.c_char_p, [_i32]),
    "rmsnorm_bwd_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32, _vp]),
    "rrn_last_cuda_error": (_i32, []),
    "rrn_device_faults": (_i32, [ctypes.POINTER(ctypes.c_uint), _i32]),
    "rrn_selftest_wait_timeout": (_i32, [ctypes.c_uint64, _vp]),
    "rrn_plan_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, ctypes.POINTER(rrn_launch)]),
    "rrn_plan_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, ctypes.POINTER(rrn_launch)]),
    "rrn_plan_layernorm_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32,
                                      ctypes.POINTER(rrn_launch)]),
    "rrn_plan_layernorm_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, ctypes.POINTER(rrn_launch)]),
    "rrn_plan_fwd_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, ctypes.POINTER(rrn_launch)]),
    "add_rmsnorm_fwd_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32,
                                  ctypes.POINTER(rrn_launch), _vp]),
    "rmsnorm_bwd_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _f32, _i32,
                              ctypes.POINTER(rrn_launch), _vp]),
    "add_rmsnorm_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _f32, _i32,
                               _vp]),
    "rmsnorm_fwd_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32, _vp]),
    "rmsnorm_fwd_fp8_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32,
                                  ctypes.POINTER(rrn_launch), _vp]),
    "layernorm_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32, _vp]),
    "add_layernorm_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32,
                                 _vp]),
    "add_layernorm_fwd_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32,
                                    ctypes.POINTER(rrn_launch), _vp]),
    "layernorm_bwd_workspace_bytes": (_i32, [_i64, _i64, _i32, ctypes.POINTER(_sz)]),
    "layernorm_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64,
                             _f32, _i32, _vp]),
    "layernorm_bwd_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64,
                                _f32, _i32, ctypes.POINTER(rrn_launch), _vp]),
    "add_rmsnorm_bwd_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _f32,
                                  _i32, ctypes.POINTER(rrn_launch), _vp]),
}


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load ``librrn.so`` (once) and declare the C signatures. Raises if it is missing."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIBRARY_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"the GPU library {p} is not built: run `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (or residual_rmsnorm_row_gb300/build.py) first")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        lib = load_library()
        msg = lib.rrn_status_string(status).decode()
        raise RRNError(status, msg, lib.rrn_last_cuda_error() if status == 7 else 0)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"dtype {t.dtype} is not supported (bfloat16 or float32)") from None


def _mat(t: torch.Tensor, name: str, N: Optional[int] = None) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")
    if N is not None and (t.dim() == 0 or t.shape[-1] != N):
        raise ValueError(f"{name} must have last dimension {N}")
    return t.data_ptr()


def _same(a: torch.Tensor, b: torch.Tensor, name: str) -> None:
    if b.shape != a.shape or b.dtype != a.dtype:
        raise ValueError(f"{name} must have the shape and dtype of x")


def _rows(x: torch.Tensor):
    N = int(x.shape[-1])
    return (x.numel() // N if N else 0), N


def _vec(t: Optional[torch.Tensor], name: str) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    return t.data_ptr()


def rmsnorm_fwd(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, rstd: Optional[torch.Tensor],
                eps: float, stream=None) -> None:
    """C ``rmsnorm_fwd``: y = x * rstd * w per row of x ([..., N]); rstd optional ([M] fp32)."""
    M, N = _rows(x)
    _same(x, y, "y")
    if w.shape != (N,) or w.dtype != x.dtype:
        raise ValueError("w must have shape (N,) and the dtype of x")
    if rstd is not None and rstd.numel() != M:
        raise ValueError("rstd must hold M values")
    _check(load_library().rmsnorm_fwd(_mat(x, "x", N), _mat(w, "w"), _mat(y, "y"),
                                      _vec(rstd, "rstd"), M, N, float(eps), _dtype(x),
                                      _stream(stream)))


def add_rmsnorm_fwd(x: torch.Tensor, residual: torch.Tensor, residual_out: torch.Tensor,
                    w: torch.Tensor, y: torch.Tensor, rstd: Optional[torch.Tensor], eps: float,
                    stream=None) -> None:
    """C ``add_rmsnorm_fwd``: residual_out = x + residual, y = RMSNorm(x + residual) * w."""
    M, N = _rows(x)
    _same(x, residual, "residual")
    _same(x, residual_out, "residual_out")
    _same(x, y, "y")
    if w.shape != (N,) or w.dtype != x.dtype:
        raise ValueError("w must have shape (N,) and the dtype of x")
    if rstd is not None and rstd.numel() != M:
        raise ValueError("rstd must hold M values")
    _check(load_library().add_rmsnorm_fwd(
        _mat(x, "x", N), _mat(residual, "residual"), _mat(residual_out, "residual_out"),
        _mat(w, "w"), _mat(y, "y"), _vec(rstd, "rstd"), M, N, float(eps), _dtype(x),
        _stream(stream)))


def add_rmsnorm_fwd_ex(x: torch.Tensor, residual: Optional[torch.Tensor],
                       residual_out: Optional[torch.Tensor], w: torch.Tensor, y: torch.Tensor,
                       rstd: Optional[torch.Tensor], eps: float, launch: Optional[Launch] = None,
                       stream=None) -> None:
    """C ``add_rmsnorm_fwd_ex``: either forward with an explicit launch configuration."""
    M, N = _rows(x)
    _same(x, y, "y")
    if residual is not None:
        _same(x, residual, "residual")
        _same(x, residual_out, "residual_out")
    if w.shape != (N,) or w.dtype != x.dtype:
        raise ValueError("w must have shape (N,) and the dtype of x")
    cfg = ctypes.byref(launch.to_c()) if launch is not None else None
    _check(load_library().add_rmsnorm_fwd_ex(
        _mat(x, "x", N), None if residual is None else _mat(residual, "residual"),
        None if residual is None else _mat(residual_out, "residual_out"), _mat(w, "w"),
        _mat(y, "y"), _vec(rstd, "rstd"), M, N, float(eps), _dtype(x), cfg, _stream(stream)))


def rmsnorm_bwd_workspace_bytes(M: int, N: int, dtype: torch.dtype) -> int:
    """C ``rmsnorm_bwd_workspace_bytes`` for the current device."""
    out = ctypes.c_size_t(0)
    _check(load_library().rmsnorm_bwd_workspace_bytes(int(M), int(N), _DTYPES[dtype],
                                                      ctypes.byref(out)))
    return int(out.value)


def rmsnorm_bwd(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, rstd: torch.Tensor,
                dx: torch.Tensor, dw: torch.Tensor, workspace: torch.Tensor, eps: float,
                stream=None) -> None:
    """C ``rmsnorm_bwd``: dx (dtype of x) and dw ([N] fp32, overwritten)."""
    M, N = _rows(x)
    _same(x, dy, "dy")
    _same(x, dx, "dx")
    if w.shape != (N,) or w.dtype != x.dtype:
        raise ValueError("w must have shape (N,) and the dtype of x")
    if rstd.numel() != M or dw.numel() != N:
        raise ValueError("rstd must hold M values and dw N values")
    _check(load_library().rmsnorm_bwd(
        _mat(dy, "dy", N), _mat(x, "x"), _mat(w, "w"), _vec(rstd, "rstd"), _mat(dx, "dx"),
        _vec(dw, "dw"), _mat(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        M, N, float(eps), _dtype(x), _stream(stream)))


def rmsnorm_bwd_noalloc(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, rstd: torch.Tensor,
                        dx: torch.Tensor, dw: torch.Tensor, eps: float, stream=None) -> None:
    """C ``rmsnorm_bwd_noalloc``: ``rmsnorm_bwd`` for callers that cannot allocate device memory
    (the partial sums live in the library's own fixed 8 MiB device array; calls that overlap on
    the GPU race on it, so order them on one stream)."""
    M, N = _rows(x)
    _same(x, dy, "dy")
    _same(x, dx, "dx")
    if w.shape != (N,) or w.dtype != x.dtype:
        raise ValueError("w must have shape (N,) and the dtype of x")
    if rstd.numel() != M or dw.numel() != N:
        raise ValueError("rstd must hold M values and dw N values")
    _check(load_library().rmsnorm_bwd_noalloc(
        _mat(dy, "dy", N), _mat(x, "x"), _mat(w, "w"), _vec(rstd, "rstd"), _mat(dx, "dx"),
        _vec(dw, "dw"), M, N, float(eps), _dtype(x), _stream(stream)))


def rmsnorm_bwd_ex(dy, x, w, rstd, dx, dw, workspace, eps, launch: Optional[Launch] = None,
                   stream=None) -> None:
    """C ``rmsnorm_bwd_ex``: backward with an explicit stage-1 launch configuration."""
    M, N = _rows(x)
    _same(x, dy, "dy")
    _same(x, dx, "dx")
    cfg = ctypes.byref(launch.to_c()) if launch is not None else None
    _check(load_library().rmsnorm_bwd_ex(
        _mat(dy, "dy", N), _mat(x, "x"), _mat(w, "w"), _vec(rstd, "rstd"), _mat(dx, "dx"),
        _vec(dw, "dw"), _mat(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        M, N, float(eps), _dtype(x), cfg, _stream(stream)))


def add_rmsnorm_bwd(dy: torch.Tensor, d_residual_out: Optional[torch.Tensor],
                    residual_out: torch.Tensor, w: torch.Tensor, rstd: torch.Tensor,
                    d_r: torch.Tensor, dw: torch.Tensor, workspace: torch.Tensor, eps: float,
                    launch: Optional[Launch] = None, stream=None) -> None:
    """C ``add_rmsnorm_bwd`` (``_ex`` with ``launch``): d_r w.r.t. x + residual, and dw."""
    M, N = _rows(residual_out)
    _same(residual_out, dy, "dy")
    _same(residual_out, d_r, "d_r")
    if d_residual_out is not None:
        _same(residual_out, d_residual_out, "d_residual_out")
    if w.shape != (N,) or w.dtype != residual_out.dtype:
        raise ValueError("w must have shape (N,) and the dtype of residual_out")
    if rstd.numel() != M or dw.numel() != N:
        raise ValueError("rstd must hold M values and dw N values")
    args = [_mat(dy, "dy", N), None if d_residual_out is None else _mat(d_residual_out, "d_residual_out"),
            _mat(residual_out, "residual_out"), _mat(w, "w"), _vec(rstd, "rstd"), _mat(d_r, "d_r"),
            _vec(dw, "dw"), _mat(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), M, N, float(eps), _dtype(residual_out)]
    lib = load_library()
    if launch is None:
        _check(lib.add_rmsnorm_bwd(*args, _stream(stream)))
    else:
        _check(lib.add_rmsnorm_bwd_ex(*args, ctypes.byref(launch.to_c()), _stream(stream)))


def _opt(t: Optional[torch.Tensor], name: str) -> Optional[int]:
    return None if t is None else _mat(t, name)


def layernorm_fwd(x: torch.Tensor, w: torch.Tensor, b: Optional[torch.Tensor], y: torch.Tensor,
                  mean: Optional[torch.Tensor], rstd: Optional[torch.Tensor], eps: float,
                  residual: Optional[torch.Tensor] = None,
                  residual_out: Optional[torch.Tensor] = None, launch: Optional[Launch] = None,
                  stream=None) -> None:
    """C ``layernorm_fwd`` / ``add_layernorm_fwd`` (with ``residual``) / ``add_layernorm_fwd_ex``
    (with ``launch``): y = (r - mean) * rstd * w + b for r = x (+ residual)."""
    M, N = _rows(x)
    _same(x, y, "y")
    if residual is not None:
        _same(x, residual, "residual")
        _same(x, residual_out, "residual_out")
    for t, n in ((w, "w"), (b, "b")):
        if t is not None and (t.shape != (N,) or t.dtype != x.dtype):
            raise ValueError(f"{n} must have shape (N,) and the dtype of x")
    for t, n in ((mean, "mean"), (rstd, "rstd")):
        if t is not None and t.numel() != M:
            raise ValueError(f"{n} must hold M values")
    lib = load_library()
    px, pw, pb, py = _mat(x, "x", N), _mat(w, "w"), _opt(b, "b"), _mat(y, "y")
    pm, pr = _vec(mean, "mean"), _vec(rstd, "rstd")
    if launch is not None:
        _check(lib.add_layernorm_fwd_ex(px, _opt(residual, "residual"), _opt(residual_out, "residual_out"),
                                        pw, pb, py, pm, pr, M, N, float(eps), _dtype(x),
                                        ctypes.byref(launch.to_c()), _stream(stream)))
    elif residual is not None:
        _check(lib.add_layernorm_fwd(px, _mat(residual, "residual"), _mat(residual_out, "residual_out"),
                                     pw, pb, py, pm, pr, M, N, float(eps), _dtype(x), _stream(stream)))
    else:
        _check(lib.layernorm_fwd(px, pw, pb, py, pm, pr, M, N, float(eps), _dtype(x), _stream(stream)))


def rmsnorm_fwd_fp8(x: torch.Tensor, residual: Optional[torch.Tensor],
                    residual_out: Optional[torch.Tensor], w: torch.Tensor, q: torch.Tensor,
                    scale: torch.Tensor, rstd: Optional[torch.Tensor], eps: float,
                    launch: Optional[Launch] = None, stream=None) -> None:
    """C ``rmsnorm_fwd_fp8`` (``_ex`` with ``launch``): e4m3 codes ``q`` (uint8 or
    float8_e4m3fn, [M, N]) and per-row ``scale`` of RMSNorm(x (+ residual)) * w."""
    M, N = _rows(x)
    if residual is not None:
        _same(x, residual, "residual")
        _same(x, residual_out, "residual_out")
    if q.shape != x.shape or q.element_size() != 1:
        raise ValueError("q must be a one-byte tensor of the shape of x")
    if w.shape != (N,) or w.dtype != x.dtype:
        raise ValueError("w must have shape (N,) and the dtype of x")
    if scale.numel() != M or (rstd is not None and rstd.numel() != M):
        raise ValueError("scale and rstd must hold M values")
    args = [_mat(x, "x", N), _opt(residual, "residual"), _opt(residual_out, "residual_out"),
            _mat(w, "w"), _mat(q, "q"), _vec(scale, "scale"), _vec(rstd, "rstd"), M, N,
            float(eps), _dtype(x)]
    lib = load_library()
    if launch is None:
        _check(lib.rmsnorm_fwd_fp8(*args, _stream(stream)))
    else:
        _check(lib.rmsnorm_fwd_fp8_ex(*args, ctypes.byref(launch.to_c()), _stream(stream)))


def layernorm_bwd_workspace_bytes(M: int, N: int, dtype: torch.dtype) -> int:
    """C ``layernorm_bwd_workspace_bytes`` for the current device."""
    out = ctypes.c_size_t(0)
    _check(load_library().layernorm_bwd_workspace_bytes(int(M), int(N), _DTYPES[dtype],
                                                        ctypes.byref(out)))
    return int(out.value)


def layernorm_bwd(dy: torch.Tensor, d_residual_out: Optional[torch.Tensor], x: torch.Tensor,
                  w: torch.Tensor, mean: torch.Tensor, rstd: torch.Tensor, dx: torch.Tensor,
                  dw: torch.Tensor, db: Optional[torch.Tensor], workspace: torch.Tensor,
                  eps: float, launch: Optional[Launch] = None, stream=None) -> None:
    """C ``layernorm_bwd`` (``_ex`` with ``launch``)."""
    M, N = _rows(x)
    _same(x, dy, "dy")
    _same(x, dx, "dx")
    if d_residual_out is not None:
        _same(x, d_residual_out, "d_residual_out")
    if w.shape != (N,) or w.dtype != x.dtype:
        raise ValueError("w must have shape (N,) and the dtype of x")
    if mean.numel() != M or rstd.numel() != M or dw.numel() != N or (db is not None and db.numel() != N):
        raise ValueError("mean/rstd must hold M values, dw/db N values")
    args = [_mat(dy, "dy", N), _opt(d_residual_out, "d_residual_out"), _mat(x, "x"), _mat(w, "w"),
            _vec(mean, "mean"), _vec(rstd, "rstd"), _mat(dx, "dx"), _vec(dw, "dw"), _vec(db, "db"),
            _mat(workspace, "workspace"), workspace.numel() * workspace.element_size(), M, N,
            float(eps), _dtype(x)]
    lib = load_library()
    if launch is None:
        _check(lib.layernorm_bwd(*args, _stream(stream)))
    else:
        _check(lib.layernorm_bwd_ex(*args, ctypes.byref(launch.to_c()), _stream(stream)))


def plan_fwd(x: torch.Tensor, residual: Optional[torch.Tensor] = None,
             residual_out: Optional[torch.Tensor] = None, w: Optional[torch.Tensor] = None,
             y: Optional[torch.Tensor] = None) -> Launch:
    """C ``rrn_plan_fwd``: the launch the automatic forward would use for these tensors."""
    M, N = _rows(x)
    out = rrn_launch()
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    _check(load_library().rrn_plan_fwd(ptr(x), ptr(residual), ptr(residual_out),
                                       ptr(w if w is not None else x), ptr(y if y is not None else x),
                                       M, N, _dtype(x), ctypes.byref(out)))
    return Launch.from_c(out)


def plan_layernorm_fwd(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, b: Optional[torch.Tensor] = None,
                       residual: Optional[torch.Tensor] = None,
                       residual_out: Optional[torch.Tensor] = None) -> Launch:
    """C ``rrn_plan_layernorm_fwd``: the launch the automatic LayerNorm forward would use."""
    M, N = _rows(x)
    out = rrn_launch()
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    _check(load_library().rrn_plan_layernorm_fwd(ptr(x), ptr(residual), ptr(residual_out), ptr(w), ptr(b),
                                                 ptr(y), M, N, _dtype(x), ctypes.byref(out)))
    return Launch.from_c(out)


def plan_layernorm_bwd(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, dx: torch.Tensor,
                       d_residual_out: Optional[torch.Tensor] = None) -> Launch:
    """C ``rrn_plan_layernorm_bwd``: the stage-1 launch the automatic LayerNorm backward would use."""
    M, N = _rows(x)
    out = rrn_launch()
    dro = None if d_residual_out is None else d_residual_out.data_ptr()
    _check(load_library().rrn_plan_layernorm_bwd(dy.data_ptr(), dro, x.data_ptr(), w.data_ptr(),
                                                 dx.data_ptr(), M, N, _dtype(x), ctypes.byref(out)))
    return Launch.from_c(out)


def plan_fwd_fp8(x: torch.Tensor, w: torch.Tensor, q: torch.Tensor, residual: Optional[torch.Tensor] = None,
                 residual_out: Optional[torch.Tensor] = None) -> Launch:
    """C ``rrn_plan_fwd_fp8``: the launch the automatic fp8 forward would use."""
    M, N = _rows(x)
    out = rrn_launch()
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    _check(load_library().rrn_plan_fwd_fp8(ptr(x), ptr(residual), ptr(residual_out), ptr(w), ptr(q),
                                           M, N, _dtype(x), ctypes.byref(out)))
    return Launch.from_c(out)


def device_faults(clear: bool = True) -> int:
    """C ``rrn_device_faults``: the device fault word (bit 0: a bounded wait ran out)."""
    out = ctypes.c_uint(0)
    _check(load_library().rrn_device_faults(ctypes.byref(out), 1 if clear else 0))
    return int(out.value)


def selftest_wait_timeout(limit_ns: int = 50_000_000, stream=None) -> None:
    """C ``rrn_selftest_wait_timeout``: make one bounded wait run out on purpose."""
    _check(load_library().rrn_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def plan_bwd(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, dx: torch.Tensor,
             d_residual_out: Optional[torch.Tensor] = None) -> Launch:
    """C ``rrn_plan_bwd``: the stage-1 launch the automatic backward would use
    (``d_residual_out`` given: the fused backward's)."""
    M, N = _rows(x)
    out = rrn_launch()
    dro = None if d_residual_out is None else d_residual_out.data_ptr()
    _check(load_library().rrn_plan_bwd(dy.data_ptr(), dro, x.data_ptr(), w.data_ptr(),
                                       dx.data_ptr(), M, N, _dtype(x), ctypes.byref(out)))
    return Launch.from_c(out)
