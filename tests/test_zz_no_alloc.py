"""rmsnorm_bwd_noalloc, the backward entry point for callers that cannot allocate device memory,
against the regular rmsnorm_bwd.

Callers that cannot hand the library a workspace - code running during CUDA graph capture,
plugins inside an engine that owns every device allocation, C callers without a caching
allocator - call rmsnorm_bwd_noalloc, which keeps its partial sums in a fixed array inside the
library. Both entry points are called here through the C ABI on the same inputs, several calls in
a row (the array keeps the previous call's contents), and must agree within the bounds the other
GPU tests use. The file name makes pytest collect it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import residual_rmsnorm_row_gb300 as rrn
import synth

pytestmark = pytest.mark.gpu

RRN_ERR_SCRATCH = 9


def _dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.float32:
        return torch.from_numpy(a).cuda()
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def _values(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def _both(M: int, N: int, dtype: str, seed: int):
    wl = synth.Workload("noalloc", "rmsnorm_bwd", M, N, dtype, 1e-6, seed)
    h = synth.make(wl)
    x, w, dy = _dev(h["x"]), _dev(h["w"]), _dev(h["dy"])
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
    return dx0, dw0, dx1, dw1, dtype


def _agree(dx0, dw0, dx1, dw1, dtype):
    ref, got = _values(dx0), _values(dx1)
    rel = 2.0 ** -8 if dtype == "bf16" else 1e-5
    assert np.all(np.abs(got - ref) <= rel * np.abs(ref) + 1e-6), "dx differs"
    r, g = _values(dw0), _values(dw1)
    assert np.all(np.abs(g - r) <= 1e-3 * np.maximum(np.abs(r), 1.0)), "dw differs"


def test_noalloc_matches_the_regular_backward_on_calls_in_a_row():
    # 16384 x 4096 needs fewer stage-1 CTAs than the regular plan (the array holds 2^21 floats);
    # the second call has another shape and dtype; the third repeats the first.
    for M, N, dtype, seed in ((16384, 4096, "bf16", 4), (1000, 1024, "f32", 5), (16384, 4096, "bf16", 4)):
        _agree(*_both(M, N, dtype, seed))


def test_noalloc_wide_rows_split_over_clusters():
    # rows of 24576 columns: each row is split over a cluster of 8 CTAs, and the array holds
    # partial sums for 85 CTAs - lowered to 80, whole clusters
    _agree(*_both(400, 24576, "bf16", 6))


def test_noalloc_rejects_rows_wider_than_its_array_and_allows_empty():
    lib = rrn.load_library()
    n_too_wide = (1 << 21) + 8
    # rejected from the width alone, before anything is read
    assert lib.rmsnorm_bwd_noalloc(None, None, None, None, None, None, 4, n_too_wide,
                                   ctypes.c_float(1e-6), 0, None) == RRN_ERR_SCRATCH
    assert lib.rmsnorm_bwd_noalloc(None, None, None, None, None, None, 0, 4096,
                                   ctypes.c_float(1e-6), 0, None) == 0
