"""rmsnorm_bwd_noalloc, the backward entry point for callers that cannot allocate device memory,
against the fp64 oracle and the regular rmsnorm_bwd.

Some callers cannot hand the library a workspace: plugins inside an engine that owns every
device allocation and passes a plugin only its inputs and outputs, and C callers without a
caching allocator, for whom a cudaMalloc/cudaFree pair per call would synchronise the device.
They call rmsnorm_bwd_noalloc, which keeps its partial sums in a fixed array inside the library.
Here it is called through the C ABI several times in a row (the array keeps the previous call's
contents) and its dx and dw must match the oracle within the bounds the other GPU tests use, and
the regular entry point's results on the same inputs within the same bounds. The file name makes
pytest collect it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import residual_rmsnorm_row_gb300 as rrn
import synth
from gpu_util import bwd_cond, check_dw, check_out, to_dev, values

pytestmark = pytest.mark.gpu

RRN_ERR_SCRATCH = 9
SCRATCH_FLOATS = 1 << 21


def _both(M: int, N: int, dtype: str, seed: int):
    wl = synth.Workload("noalloc", "rmsnorm_bwd", M, N, dtype, 1e-6, seed)
    h = synth.make(wl)
    x, w, dy = to_dev(h["x"], dtype), to_dev(h["w"], dtype), to_dev(h["dy"], dtype)
    _, rstd = rrn.rms_norm(x, w, wl.eps)
    dx0, dw0 = rrn.rms_norm_backward(dy, x, w, rstd, wl.eps)        # the regular entry point
    dx1 = torch.full_like(x, float("nan"))
    dw1 = torch.full((N,), float("nan"), device="cuda")
    lib = rrn.load_library()
    st = lib.rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), w.data_ptr(), rstd.data_ptr(),
                                 dx1.data_ptr(), dw1.data_ptr(), M, N, ctypes.c_float(wl.eps),
                                 0 if dtype == "bf16" else 1,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.rrn_status_string(st)
    torch.cuda.synchronize()
    return h, wl, dx0, dw0, dx1, dw1


def _check(M: int, N: int, dtype: str, seed: int):
    h, wl, dx0, dw0, dx1, dw1 = _both(M, N, dtype, seed)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(h["dy"], h["x"], h["w"], wl.eps)
    cond = None if dtype == "bf16" else bwd_cond(h["x"], h["dy"], h["w"], wl.eps)
    # against the oracle
    check_out(values(dx1), dx_ref, dtype, f"noalloc dx {M}x{N} {dtype}", cond=cond)
    check_dw(dw1.cpu().numpy().astype(np.float64), dw_ref, f"noalloc dw {M}x{N} {dtype}")
    # against the regular entry point: dx is computed row by row the same way (bit for bit);
    # dw within the dw bound (its partial sums may be added in another order)
    assert torch.equal(dx1, dx0), "noalloc dx differs from rmsnorm_bwd's"
    check_dw(dw1.cpu().numpy().astype(np.float64), dw0.cpu().numpy().astype(np.float64),
             "noalloc dw vs rmsnorm_bwd")
    return dx1, dw1


def test_noalloc_matches_oracle_and_regular_backward_on_calls_in_a_row():
    # 16384 x 4096: the array holds 512 rows of partial sums, fewer than the regular plan's
    # stage-1 CTAs, so the CTA count is lowered; the second call has another shape and dtype;
    # the third repeats the first and must give the same bits (the array kept the second call's
    # contents in between).
    first = _check(16384, 4096, "bf16", 4)
    _check(1000, 1024, "f32", 5)
    third = _check(16384, 4096, "bf16", 4)
    assert torch.equal(first[0], third[0]) and torch.equal(first[1], third[1])


def test_noalloc_short_rows_one_per_warp():
    # rows of 512 columns over many rows: the regular plan takes a row per warp (one row of
    # partial sums per CTA); the array holds 4096 such rows, more than that plan's CTAs
    M, N = 16384, 512
    x = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    w = torch.empty(N, device="cuda", dtype=torch.bfloat16)
    assert rrn.plan_bwd(x, x, w, x).variant == rrn.VARIANT_ROW_WARP
    _check(M, N, "bf16", 7)


def test_noalloc_wide_rows_split_over_clusters():
    # rows of 24576 columns are split over clusters of 8 CTAs, one row of partial sums per
    # cluster: the array holds 85 such rows (2^21 // 24576), more than this GPU runs at once,
    # so the regular launch is kept
    _check(400, 24576, "bf16", 6)


def test_noalloc_rejects_rows_wider_than_its_array_and_zeroes_dw_when_empty():
    lib = rrn.load_library()
    n_too_wide = SCRATCH_FLOATS + 8
    dy = torch.zeros(1, n_too_wide, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(n_too_wide, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(1, device="cuda")
    dw = torch.zeros(n_too_wide, device="cuda")
    st = lib.rmsnorm_bwd_noalloc(dy.data_ptr(), dy.data_ptr(), w.data_ptr(), rstd.data_ptr(),
                                 dy.data_ptr(), dw.data_ptr(), 1, n_too_wide,
                                 ctypes.c_float(1e-6), 0, None)
    assert st == RRN_ERR_SCRATCH
    # argument errors are reported as such, even for rows too wide for the array
    assert lib.rmsnorm_bwd_noalloc(None, None, None, None, None, None, 4, n_too_wide,
                                   ctypes.c_float(1e-6), 0, None) == 1      # RRN_ERR_NULL
    # M == 0: dw is a sum over no rows, zero as in the oracle, for any width
    empty = np.zeros((0, 4096), dtype=np.uint16)
    _, dw_ref = oracle.rmsnorm_bwd(empty, empty, np.zeros(4096, np.uint16), 1e-6)
    dw0 = torch.full((4096,), 7.0, device="cuda")
    assert lib.rmsnorm_bwd_noalloc(None, None, None, None, None, dw0.data_ptr(), 0, 4096,
                                   ctypes.c_float(1e-6), 0, None) == 0
    torch.cuda.synchronize()
    check_dw(dw0.cpu().numpy().astype(np.float64), dw_ref, "noalloc dw, M == 0")
    assert not torch.any(dw0 != 0)
