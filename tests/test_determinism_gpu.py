"""Bitwise reproducibility: the same call on the same inputs gives the same bits, every output.

The reductions run in a fixed order (no atomics): the dw (and db) sums of the backward kernels,
the per-row sums and maxima of the forward kernels. Each case runs twice on the same device
buffers and compares the raw bits, on a shape that spans many CTAs per SM.
"""
from __future__ import annotations

import pytest
import torch

import residual_rmsnorm_row_gb300 as rrn
import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32) if t.element_size() == 4 else t


def _same(a, b):
    return all(torch.equal(_bits(x), _bits(y)) for x, y in zip(a, b))


@pytest.mark.parametrize("launch", [None, rrn.Launch(rrn.VARIANT_ROW_CTA, 2, 256, 0, 0, 8)],
                         ids=["auto", "dw-over-clusters-of-8"])
def test_fused_backward_is_bitwise_reproducible(launch):
    wl = synth.get("add_rmsnorm_bwd_16384x4096_bf16").with_shape(4096)
    h = synth.make(wl)
    x, w = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16")
    dy, dro = to_dev(h["dy"], "bf16"), to_dev(h["d_ro"], "bf16")
    _, rstd = rrn.rms_norm(x, w, wl.eps)
    ws = torch.empty(wl.M * wl.N, device="cuda")

    def run():
        dr = torch.empty_like(x)
        dw = torch.empty(wl.N, device="cuda")
        rrn.add_rmsnorm_bwd(dy, dro, x, w, rstd, dr, dw, ws, wl.eps, launch=launch)
        torch.cuda.synchronize()
        return dr, dw

    assert _same(run(), run())


@pytest.mark.parametrize("with_dro", [True, False])
def test_short_row_backward_is_bitwise_reproducible(with_dro):
    # 512 columns over many rows: one row per warp, the CTA's warps adding their dw sums in order
    wl = synth.get("add_rmsnorm_bwd_16384x4096_bf16").with_shape(16384, 512)
    h = synth.make(wl)
    x, w = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16")
    dy = to_dev(h["dy"], "bf16")
    dro = to_dev(h["d_ro"], "bf16") if with_dro else None
    _, rstd = rrn.rms_norm(x, w, wl.eps)
    assert rrn.plan_bwd(dy, x, w, x, dro).variant == rrn.VARIANT_ROW_WARP
    ws = torch.empty(wl.M * wl.N, device="cuda")

    def run():
        dr = torch.empty_like(x)
        dw = torch.empty(wl.N, device="cuda")
        rrn.add_rmsnorm_bwd(dy, dro, x, w, rstd, dr, dw, ws, wl.eps)
        torch.cuda.synchronize()
        return dr, dw

    assert _same(run(), run())


@pytest.mark.parametrize("with_dro", [True, False])
def test_short_row_layernorm_backward_is_bitwise_reproducible(with_dro):
    # 1024 columns over many rows: one row per warp, the warps adding dw and db in order
    wl = synth.get("layernorm_bwd_16384x4096_bf16").with_shape(16384, 1024)
    h = synth.make(wl)
    x, w = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16")
    dy = to_dev(h["dy"], "bf16")
    dro = to_dev(h["d_ro"], "bf16") if with_dro else None
    _, mean, rstd = rrn.layer_norm(x, w, None, wl.eps)
    assert rrn.plan_layernorm_bwd(dy, x, w, x, dro).variant == rrn.VARIANT_ROW_WARP
    ws = torch.empty(wl.M * wl.N * 2, device="cuda")

    def run():
        dx = torch.empty_like(x)
        dw = torch.empty(wl.N, device="cuda")
        db = torch.empty(wl.N, device="cuda")
        rrn.layernorm_bwd(dy, dro, x, w, mean, rstd, dx, dw, db, ws, wl.eps)
        torch.cuda.synchronize()
        return dx, dw, db

    assert _same(run(), run())


@pytest.mark.parametrize("with_dro", [True, False])
def test_layernorm_backward_is_bitwise_reproducible(with_dro):
    wl = synth.get("layernorm_bwd_16384x4096_bf16").with_shape(4096)
    h = synth.make(wl)
    x, w, b = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16"), to_dev(h["b"], "bf16")
    dy = to_dev(h["dy"], "bf16")
    dro = to_dev(h["d_ro"], "bf16") if with_dro else None
    _, mean, rstd = rrn.layer_norm(x, w, b, wl.eps)
    ws = torch.empty(wl.M * wl.N * 2, device="cuda")

    def run():
        dx = torch.empty_like(x)
        dw = torch.empty(wl.N, device="cuda")
        db = torch.empty(wl.N, device="cuda")
        rrn.layernorm_bwd(dy, dro, x, w, mean, rstd, dx, dw, db, ws, wl.eps)
        torch.cuda.synchronize()
        return dx, dw, db

    assert _same(run(), run())


def test_fp8_and_layernorm_forward_are_bitwise_reproducible():
    wl = synth.get("add_rmsnorm_fwd_16384x4096_bf16").with_shape(4096)
    h = synth.make(wl)
    x, res, w = to_dev(h["x"], "bf16"), to_dev(h["residual"], "bf16"), to_dev(h["w"], "bf16")

    def run():
        q, scale, ro = rrn.rms_norm_fp8(x, w, wl.eps, residual=res)
        y, mean, rstd = rrn.layer_norm(x, w, None, wl.eps)
        torch.cuda.synchronize()
        return q.view(torch.uint8), scale, ro, y, mean, rstd

    assert _same(run(), run())


def test_split_row_kernels_are_bitwise_reproducible():
    # rows split over thread-block clusters: the CTAs' partial sums meet through distributed
    # shared memory (asynchronous remote stores counted on mbarriers) and are added in rank order
    M, N = 2048, 16384
    wl = synth.Workload("split-det", "layernorm_bwd", M, N, "bf16", 1e-5, 61, x_mean=0.5)
    h = synth.make(wl)
    x, w = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16")
    dy, dro = to_dev(h["dy"], "bf16"), to_dev(h["d_ro"], "bf16")
    _, rstd = rrn.rms_norm(x, w, wl.eps)
    _, mean, lrstd = rrn.layer_norm(x, w, None, wl.eps)
    ws = torch.empty(2 * M * N, device="cuda")
    for d in (dro, None):
        plan = rrn.plan_bwd(dy, x, w, x, d)
        assert plan.variant == rrn.VARIANT_ROW_CLUSTER, plan.name
        lplan = rrn.plan_layernorm_bwd(dy, x, w, x, d)
        assert lplan.variant == rrn.VARIANT_ROW_CLUSTER, lplan.name

    def run():
        out = []
        for d in (dro, None):
            dr = torch.empty_like(x)
            dw = torch.empty(N, device="cuda")
            rrn.add_rmsnorm_bwd(dy, d, x, w, rstd, dr, dw, ws, wl.eps)
            dx = torch.empty_like(x)
            lw = torch.empty(N, device="cuda")
            lb = torch.empty(N, device="cuda")
            rrn.layernorm_bwd(dy, d, x, w, mean, lrstd, dx, lw, lb, ws, wl.eps)
            out += [dr, dw, dx, lw, lb]
        y, ro, rs = rrn.add_rms_norm(x, dy, w, wl.eps)
        q, scale, ro2 = rrn.rms_norm_fp8(x, w, wl.eps, residual=dy)
        torch.cuda.synchronize()
        return out + [y, ro, rs, q.view(torch.uint8), scale, ro2]

    assert rrn.plan_fwd(x, dy, x, w, x).variant == rrn.VARIANT_ROW_CLUSTER
    assert _same(run(), run())
