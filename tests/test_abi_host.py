"""The C ABI on a host without a GPU: the library builds, loads, exports every symbol that
include/rrn.h declares, and rejects bad arguments with the documented codes before it touches
the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rrn.h")

OK, ERR_NULL, ERR_SHAPE, ERR_EPS, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA, ERR_CONFIG = range(9)
BF16, F32 = 0, 1
A = 0x10000  # a 16-byte-aligned address that is never dereferenced (every call below fails
             # validation or has M == 0, so nothing is launched)


@pytest.fixture(scope="module")
def lib():
    from residual_rmsnorm_row_gb300 import build

    build.build()
    import residual_rmsnorm_row_gb300 as rrn

    return rrn.load_library()


def declared_symbols():
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"RRN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    assert {"rmsnorm_fwd", "add_rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_workspace_bytes",
            "rrn_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"librrn.so does not export {name}"


def test_library_exports_nothing_else():
    import subprocess

    from residual_rmsnorm_row_gb300 import build

    out = subprocess.run(["nm", "-D", "--defined-only", build.LIBRARY], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_symbols())


def test_status_strings(lib):
    for s in range(10):
        assert b"unknown" not in lib.rrn_status_string(s)
    assert b"unknown" in lib.rrn_status_string(99)


def fwd(lib, x=A, w=A, y=A, rstd=None, M=4, N=64, eps=1e-6, dtype=BF16):
    return lib.rmsnorm_fwd(x, w, y, rstd, M, N, eps, dtype, None)


def add_fwd(lib, x=A, res=A, ro=A, w=A, y=A, rstd=None, M=4, N=64, eps=1e-6, dtype=BF16):
    return lib.add_rmsnorm_fwd(x, res, ro, w, y, rstd, M, N, eps, dtype, None)


def bwd(lib, dy=A, x=A, w=A, rstd=A, dx=A, dw=A, ws=A, wsb=1 << 30, M=4, N=64, eps=1e-6,
        dtype=BF16):
    return lib.rmsnorm_bwd(dy, x, w, rstd, dx, dw, ws, wsb, M, N, eps, dtype, None)


def test_null_pointers(lib):
    assert fwd(lib, x=None) == ERR_NULL
    assert fwd(lib, w=None) == ERR_NULL
    assert fwd(lib, y=None) == ERR_NULL
    assert add_fwd(lib, res=None) == ERR_NULL
    assert add_fwd(lib, ro=None) == ERR_NULL
    for k in ("dy", "x", "w", "rstd", "dx", "dw"):
        assert bwd(lib, **{k: None}) == ERR_NULL, k


def test_bad_shapes(lib):
    assert fwd(lib, M=-1) == ERR_SHAPE
    assert fwd(lib, N=0) == ERR_SHAPE
    assert fwd(lib, N=-5) == ERR_SHAPE
    assert fwd(lib, N=1 << 31) == ERR_SHAPE
    assert fwd(lib, M=1 << 60, N=1 << 20) == ERR_SHAPE
    assert bwd(lib, M=-3) == ERR_SHAPE


def test_bad_eps(lib):
    for eps in (-1e-6, float("nan"), float("inf")):
        assert fwd(lib, eps=eps) == ERR_EPS
        assert add_fwd(lib, eps=eps) == ERR_EPS
        assert bwd(lib, eps=eps) == ERR_EPS


def test_bad_dtype(lib):
    for dt in (-1, 2, 7):
        assert fwd(lib, dtype=dt) == ERR_DTYPE
        assert bwd(lib, dtype=dt) == ERR_DTYPE


def test_misaligned_elements(lib):
    assert fwd(lib, x=A + 1) == ERR_ALIGN
    assert fwd(lib, x=A + 2, dtype=F32) == ERR_ALIGN
    assert fwd(lib, rstd=A + 2) == ERR_ALIGN
    assert add_fwd(lib, ro=A + 1) == ERR_ALIGN
    assert bwd(lib, dw=A + 1) == ERR_ALIGN


def test_empty_problem_launches_nothing(lib):
    # A forward with M == 0 returns before any CUDA call, so it succeeds even without a GPU.
    assert fwd(lib, M=0) == OK
    assert add_fwd(lib, M=0) == OK
    # A backward with M == 0 sets dw (a sum over no rows) to zero on the stream, so dw is
    # checked even then; the row pointers and the workspace are not (the zeroing itself is a
    # GPU test).
    assert bwd(lib, M=0, dy=None, x=None, w=None, rstd=None, dx=None, dw=None, ws=None,
               wsb=0) == ERR_NULL
    assert bwd(lib, M=0, dw=A + 2, ws=None, wsb=0) == ERR_ALIGN
    n = ctypes.c_size_t(123)
    assert lib.rmsnorm_bwd_workspace_bytes(0, 4096, BF16, ctypes.byref(n)) == OK
    assert n.value == 0


def test_workspace_query_checks_arguments(lib):
    n = ctypes.c_size_t(0)
    assert lib.rmsnorm_bwd_workspace_bytes(4, 4096, BF16, None) == ERR_NULL
    assert lib.rmsnorm_bwd_workspace_bytes(-1, 4096, BF16, ctypes.byref(n)) == ERR_SHAPE
    assert lib.rmsnorm_bwd_workspace_bytes(4, 4096, 9, ctypes.byref(n)) == ERR_DTYPE


def test_python_binding_rejects_host_tensors():
    import torch

    import residual_rmsnorm_row_gb300 as rrn

    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    w = torch.zeros(64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        rrn.rmsnorm_fwd(x, w, x, None, 1e-6)
