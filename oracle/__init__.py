"""CPU fp64 oracle for row-wise RMSNorm and fused residual Add + RMSNorm (forward, backward).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU-baseline
leg may import this package; the product path (the GPU library and its Python binding) never
does, and this package imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, single-threaded); this module only
loads it with ctypes and marshals numpy arrays. Input encodings are taken from the numpy
dtype: ``uint16`` arrays hold raw bf16 bit patterns, ``float32`` and ``float64`` arrays hold
values. Every output is a float64 array.

What each function computes, with the passage it follows, is stated in ``oracle.c``:
  rmsnorm_fwd      y = x * rstd * w, rstd = 1/sqrt(mean(x^2) + eps)  (Machete, "Built-In Areas")
  add_rmsnorm_fwd  the same on r = x + residual, also returning r  (KernelAgent page, Oink)
  rmsnorm_bwd      dx and dw, the exact derivative of rmsnorm_fwd
  add_rmsnorm_bwd  d_r (gradient w.r.t. x + residual) and dw, the derivative of add_rmsnorm_fwd
  add_layernorm_fwd / add_layernorm_bwd   the LayerNorm variant (mean subtracted, bias added)
  rmsnorm_quant_fp8  RMSNorm (+ residual add) feeding fp8 e4m3 codes with a per-row scale
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import numpy as np

from . import libbuild as _build

BF16, F32, F64 = 0, 1, 2
_CODES = {np.dtype(np.uint16): BF16, np.dtype(np.float32): F32, np.dtype(np.float64): F64}

_dbl_p = ctypes.POINTER(ctypes.c_double)


def _code(a: np.ndarray) -> int:
    try:
        return _CODES[a.dtype]
    except KeyError:
        raise TypeError(f"oracle input dtype {a.dtype} is not uint16 (bf16 bits), float32 or float64")


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _out(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_dbl_p)


class Oracle:
    """ctypes handle on one compiled copy of ``oracle.c`` (the default build, or a test's)."""

    def __init__(self, path: Optional[str] = None):
        self.path = path or _build.build()
        lib = ctypes.CDLL(self.path)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_decode.argtypes = [vp, i32, i64, _dbl_p]
        lib.oracle_add_rmsnorm_fwd.argtypes = [vp, i32, vp, i32, vp, i32, i64, i64, dbl,
                                               _dbl_p, _dbl_p, _dbl_p]
        lib.oracle_rmsnorm_fwd.argtypes = [vp, i32, vp, i32, i64, i64, dbl, _dbl_p, _dbl_p]
        lib.oracle_rmsnorm_bwd.argtypes = [vp, i32, vp, i32, vp, i32, i64, i64, dbl,
                                           _dbl_p, _dbl_p]
        lib.oracle_add_rmsnorm_bwd.argtypes = [vp, i32, vp, i32, vp, i32, vp, i32, i64, i64, dbl,
                                               _dbl_p, _dbl_p]
        lib.oracle_add_layernorm_fwd.argtypes = [vp, i32, vp, i32, vp, i32, vp, i32, i64, i64, dbl,
                                                 _dbl_p, _dbl_p, _dbl_p, _dbl_p]
        lib.oracle_add_layernorm_bwd.argtypes = [vp, i32, vp, i32, vp, i32, vp, i32, i64, i64, dbl,
                                                 _dbl_p, _dbl_p, _dbl_p]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = dbl
        lib.oracle_e4m3_encode.argtypes = [dbl]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_rmsnorm_quant_fp8.argtypes = [vp, i32, vp, i32, vp, i32, i64, i64, dbl, _dbl_p,
                                                 _dbl_p, vp, _dbl_p, _dbl_p]
        lib.oracle_rmsnorm_quant_fp8.restype = i32
        for name in ("oracle_decode", "oracle_add_rmsnorm_fwd", "oracle_rmsnorm_fwd",
                     "oracle_rmsnorm_bwd", "oracle_add_rmsnorm_bwd", "oracle_add_layernorm_fwd",
                     "oracle_add_layernorm_bwd"):
            getattr(lib, name).restype = i32
        self.lib = lib

    @staticmethod
    def _check(status: int, what: str) -> None:
        if status != 0:
            raise RuntimeError(f"{what}: oracle returned status {status}")

    def decode(self, a: np.ndarray) -> np.ndarray:
        """Exact fp64 values of ``a`` (bf16 bit patterns, float32 or float64)."""
        a = np.ascontiguousarray(a)
        out = np.empty(a.shape, dtype=np.float64)
        self._check(self.lib.oracle_decode(_ptr(a), _code(a), a.size, _out(out)), "decode")
        return out

    def add_rmsnorm_fwd(self, x: np.ndarray, residual: Optional[np.ndarray], w: np.ndarray,
                        eps: float) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
        """Return ``(r, y, rstd)`` for r = x + residual (residual None: r = x)."""
        x = np.ascontiguousarray(x)
        w = np.ascontiguousarray(w)
        M, N = x.shape
        if w.shape != (N,):
            raise ValueError("w must have shape (N,)")
        if residual is not None:
            residual = np.ascontiguousarray(residual)
            if residual.shape != x.shape:
                raise ValueError("residual must have the shape of x")
        r = np.empty((M, N), dtype=np.float64)
        y = np.empty((M, N), dtype=np.float64)
        rstd = np.empty((M,), dtype=np.float64)
        self._check(self.lib.oracle_add_rmsnorm_fwd(
            _ptr(x), _code(x), _ptr(residual), 0 if residual is None else _code(residual),
            _ptr(w), _code(w), M, N, float(eps), _out(r), _out(y), _out(rstd)),
            "add_rmsnorm_fwd")
        return r, y, rstd

    def rmsnorm_fwd(self, x: np.ndarray, w: np.ndarray, eps: float) -> Tuple[np.ndarray, np.ndarray]:
        """Return ``(y, rstd)``."""
        x = np.ascontiguousarray(x)
        w = np.ascontiguousarray(w)
        M, N = x.shape
        if w.shape != (N,):
            raise ValueError("w must have shape (N,)")
        y = np.empty((M, N), dtype=np.float64)
        rstd = np.empty((M,), dtype=np.float64)
        self._check(self.lib.oracle_rmsnorm_fwd(_ptr(x), _code(x), _ptr(w), _code(w), M, N,
                                                float(eps), _out(y), _out(rstd)), "rmsnorm_fwd")
        return y, rstd

    def rmsnorm_bwd(self, dy: np.ndarray, x: np.ndarray, w: np.ndarray, eps: float,
                    want_dx: bool = True) -> Tuple[Optional[np.ndarray], np.ndarray]:
        """Return ``(dx, dw)``; ``dx`` is None when ``want_dx`` is False (dw alone)."""
        dy = np.ascontiguousarray(dy)
        x = np.ascontiguousarray(x)
        w = np.ascontiguousarray(w)
        M, N = x.shape
        if dy.shape != x.shape or w.shape != (N,):
            raise ValueError("dy must have the shape of x and w shape (N,)")
        dx = np.empty((M, N), dtype=np.float64) if want_dx else None
        dw = np.empty((N,), dtype=np.float64)
        self._check(self.lib.oracle_rmsnorm_bwd(_ptr(dy), _code(dy), _ptr(x), _code(x), _ptr(w),
                                                _code(w), M, N, float(eps), _out(dx), _out(dw)),
                    "rmsnorm_bwd")
        return dx, dw


    def add_rmsnorm_bwd(self, dy: np.ndarray, d_residual_out: Optional[np.ndarray],
                        residual_out: np.ndarray, w: np.ndarray, eps: float,
                        want_dr: bool = True) -> Tuple[Optional[np.ndarray], np.ndarray]:
        """Return ``(d_r, dw)``: the gradient w.r.t. r = x + residual and w."""
        dy = np.ascontiguousarray(dy)
        r = np.ascontiguousarray(residual_out)
        w = np.ascontiguousarray(w)
        M, N = r.shape
        if dy.shape != r.shape or w.shape != (N,):
            raise ValueError("dy must have the shape of residual_out and w shape (N,)")
        if d_residual_out is not None:
            d_residual_out = np.ascontiguousarray(d_residual_out)
            if d_residual_out.shape != r.shape:
                raise ValueError("d_residual_out must have the shape of residual_out")
        d_r = np.empty((M, N), dtype=np.float64) if want_dr else None
        dw = np.empty((N,), dtype=np.float64)
        self._check(self.lib.oracle_add_rmsnorm_bwd(
            _ptr(dy), _code(dy), _ptr(d_residual_out),
            0 if d_residual_out is None else _code(d_residual_out), _ptr(r), _code(r), _ptr(w),
            _code(w), M, N, float(eps), _out(d_r), _out(dw)), "add_rmsnorm_bwd")
        return d_r, dw

    def add_layernorm_fwd(self, x: np.ndarray, residual: Optional[np.ndarray], w: np.ndarray,
                          b: Optional[np.ndarray], eps: float):
        """Return ``(r, y, mean, rstd)`` of LayerNorm on r = x (+ residual); b may be None."""
        x = np.ascontiguousarray(x)
        w = np.ascontiguousarray(w)
        M, N = x.shape
        if w.shape != (N,) or (b is not None and np.shape(b) != (N,)):
            raise ValueError("w and b must have shape (N,)")
        if residual is not None:
            residual = np.ascontiguousarray(residual)
            if residual.shape != x.shape:
                raise ValueError("residual must have the shape of x")
        if b is not None:
            b = np.ascontiguousarray(b)
        r = np.empty((M, N))
        y = np.empty((M, N))
        mean = np.empty(M)
        rstd = np.empty(M)
        self._check(self.lib.oracle_add_layernorm_fwd(
            _ptr(x), _code(x), _ptr(residual), 0 if residual is None else _code(residual),
            _ptr(w), _code(w), _ptr(b), 0 if b is None else _code(b), M, N, float(eps),
            _out(r), _out(y), _out(mean), _out(rstd)), "add_layernorm_fwd")
        return r, y, mean, rstd

    def add_layernorm_bwd(self, dy: np.ndarray, d_residual_out: Optional[np.ndarray],
                          x: np.ndarray, w: np.ndarray, eps: float):
        """Return ``(dx, dw, db)`` of LayerNorm at x (the stored residual_out when fused)."""
        dy = np.ascontiguousarray(dy)
        x = np.ascontiguousarray(x)
        w = np.ascontiguousarray(w)
        M, N = x.shape
        if dy.shape != x.shape or w.shape != (N,):
            raise ValueError("dy must have the shape of x and w shape (N,)")
        if d_residual_out is not None:
            d_residual_out = np.ascontiguousarray(d_residual_out)
        dx = np.empty((M, N))
        dw = np.empty(N)
        db = np.empty(N)
        self._check(self.lib.oracle_add_layernorm_bwd(
            _ptr(dy), _code(dy), _ptr(d_residual_out),
            0 if d_residual_out is None else _code(d_residual_out), _ptr(x), _code(x), _ptr(w),
            _code(w), M, N, float(eps), _out(dx), _out(dw), _out(db)), "add_layernorm_bwd")
        return dx, dw, db

    def e4m3_decode(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_decode(int(code)))

    def e4m3_encode(self, v: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(v)))

    def rmsnorm_quant_fp8(self, x: np.ndarray, residual: Optional[np.ndarray], w: np.ndarray,
                          eps: float):
        """Return ``(r, v, q, scale, rstd)``: v = y / scale (fp64), q its e4m3 codes (uint8)."""
        x = np.ascontiguousarray(x)
        w = np.ascontiguousarray(w)
        M, N = x.shape
        if residual is not None:
            residual = np.ascontiguousarray(residual)
        r = np.empty((M, N))
        v = np.empty((M, N))
        q = np.empty((M, N), dtype=np.uint8)
        scale = np.empty(M)
        rstd = np.empty(M)
        self._check(self.lib.oracle_rmsnorm_quant_fp8(
            _ptr(x), _code(x), _ptr(residual), 0 if residual is None else _code(residual), _ptr(w),
            _code(w), M, N, float(eps), _out(r), _out(v), q.ctypes.data_as(ctypes.c_void_p),
            _out(scale), _out(rstd)), "rmsnorm_quant_fp8")
        return r, v, q, scale, rstd


_DEFAULT: Optional[Oracle] = None


def default() -> Oracle:
    """The oracle built from this directory's ``oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


def decode(a):
    return default().decode(a)


def add_rmsnorm_fwd(x, residual, w, eps):
    return default().add_rmsnorm_fwd(x, residual, w, eps)


def rmsnorm_fwd(x, w, eps):
    return default().rmsnorm_fwd(x, w, eps)


def rmsnorm_bwd(dy, x, w, eps, want_dx=True):
    return default().rmsnorm_bwd(dy, x, w, eps, want_dx)


def add_rmsnorm_bwd(dy, d_residual_out, residual_out, w, eps, want_dr=True):
    return default().add_rmsnorm_bwd(dy, d_residual_out, residual_out, w, eps, want_dr)


def add_layernorm_fwd(x, residual, w, b, eps):
    return default().add_layernorm_fwd(x, residual, w, b, eps)


def add_layernorm_bwd(dy, d_residual_out, x, w, eps):
    return default().add_layernorm_bwd(dy, d_residual_out, x, w, eps)


def rmsnorm_quant_fp8(x, residual, w, eps):
    return default().rmsnorm_quant_fp8(x, residual, w, eps)


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` (used by the package's build step)."""
    return _build.build(force)


__all__ = ["Oracle", "default", "decode", "add_rmsnorm_fwd", "rmsnorm_fwd", "rmsnorm_bwd",
           "add_rmsnorm_bwd", "add_layernorm_fwd", "add_layernorm_bwd", "rmsnorm_quant_fp8",
           "build", "BF16", "F32", "F64"]
