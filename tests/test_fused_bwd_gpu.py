"""GPU parity of the fused Add + RMSNorm backward and of the autograd wrappers.

The oracle evaluates the gradient at the stored residual_out r (its input) with rstd recomputed
from r in fp64; the GPU call gets rstd from the GPU forward of that same r, so both sides
differentiate at the same point.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import residual_rmsnorm_row_gb300 as rrn
import synth
from gpu_util import bwd_cond, check_dw, check_out, to_dev, values

pytestmark = pytest.mark.gpu


def run_fused_bwd(h, dtype, eps, launch=None, with_dro=True):
    r = to_dev(h["x"], dtype)
    w = to_dev(h["w"], dtype)
    dy = to_dev(h["dy"], dtype)
    dro = to_dev(h["d_ro"], dtype) if with_dro else None
    _, rstd = rrn.rms_norm(r, w, eps)
    M, N = r.shape
    d_r = torch.full_like(r, float("nan"))
    dw = torch.full((N,), float("nan"), device="cuda")
    ws = torch.empty(max(rrn.rmsnorm_bwd_workspace_bytes(M, N, r.dtype), 4 * r.numel()) // 4,
                     device="cuda")
    rrn.add_rmsnorm_bwd(dy, dro, r, w, rstd, d_r, dw, ws, eps, launch=launch)
    torch.cuda.synchronize()
    return d_r, dw


def test_fused_backward_full_size():
    wl = synth.get("add_rmsnorm_bwd_16384x4096_bf16")
    h = synth.make(wl)
    d_r, dw = run_fused_bwd(h, "bf16", wl.eps)
    ref_dr, ref_dw = oracle.add_rmsnorm_bwd(h["dy"], h["d_ro"], h["x"], h["w"], wl.eps)
    a = check_out(values(d_r), ref_dr, "bf16", "d_r")
    b = check_dw(dw.cpu().numpy().astype(np.float64), ref_dw)
    print(f"fused bwd 16384x4096: d_r max err/bound {a:.3f}, dw {b:.3f}")


def _launches(dtype, N):
    V = 8 if dtype == "bf16" else 4
    out = [None, rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0), rrn.Launch(rrn.VARIANT_STREAM, 0, 64, 9)]
    if N % V == 0:
        nvec = N // V
        for vpt in (1, 2, 4):
            thr = -(-(-(-nvec // vpt)) // 32) * 32
            if thr <= (256 if vpt == 4 else 512):
                out += [rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 0),
                        rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 0, 0, 8),   # dw over clusters
                        rrn.Launch(rrn.VARIANT_ROW_CLUSTER, vpt, 0, 0, 0, 2),  # rows split
                        rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 0, 0),
                        rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 0, 2, 4),
                        rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 11, 2)]
        if nvec <= 256:  # one row per warp (the planner's grid; 3 CTAs of 2 warps walking rows)
            vpt = next(v for v in (1, 2, 4, 8) if 32 * v >= nvec)
            out += [rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 128, 0), rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 64, 3)]
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1, 9, 1000, 2048, 4095, 4096, 7168, 8192])
@pytest.mark.parametrize("with_dro", [True, False])
def test_fused_backward_variants(dtype, N, with_dro):
    M = 131
    wl = synth.Workload("fused-bwd", "add_rmsnorm_bwd", M, N, dtype, 1e-6, 81)
    h = synth.make(wl)
    ref_dr, ref_dw = oracle.add_rmsnorm_bwd(h["dy"], h["d_ro"] if with_dro else None, h["x"],
                                            h["w"], wl.eps)
    cond = bwd_cond(h["x"], h["dy"], h["w"], wl.eps)
    if with_dro:
        cond = cond + np.abs(oracle.decode(h["d_ro"]))
    for launch in _launches(dtype, N):
        d_r, dw = run_fused_bwd(h, dtype, wl.eps, launch, with_dro)
        check_out(values(d_r), ref_dr, dtype, f"d_r {launch}", cond)
        check_dw(dw.cpu().numpy().astype(np.float64), ref_dw, f"dw {launch}")


@pytest.mark.parametrize("N,launch", [(4096, None), (512, rrn.Launch(rrn.VARIANT_ROW_WARP, 0, 128, 0))],
                         ids=["auto", "row-per-warp"])
def test_fused_backward_in_place(N, launch):
    M = 64
    wl = synth.Workload("fused-bwd-alias", "add_rmsnorm_bwd", M, N, "bf16", 1e-6, 82)
    h = synth.make(wl)
    ref_dr, _ = oracle.add_rmsnorm_bwd(h["dy"], h["d_ro"], h["x"], h["w"], wl.eps)
    r, w = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16")
    _, rstd = rrn.rms_norm(r, w, wl.eps)
    dw = torch.empty(N, device="cuda")
    ws = torch.empty(max(rrn.rmsnorm_bwd_workspace_bytes(M, N, r.dtype), 4 * M * N) // 4, device="cuda")
    for target in ("dy", "d_ro", "r"):
        dy, dro, rr = to_dev(h["dy"], "bf16"), to_dev(h["d_ro"], "bf16"), r.clone()
        out = {"dy": dy, "d_ro": dro, "r": rr}[target]
        rrn.add_rmsnorm_bwd(dy, dro, rr, w, rstd, out, dw, ws, wl.eps, launch=launch)
        torch.cuda.synchronize()
        check_out(values(out), ref_dr, "bf16", f"d_r written over {target}")


def test_autograd_wrappers_match_the_c_calls():
    torch.manual_seed(0)
    M, N, eps = 256, 2048, 1e-6
    x = torch.randn(M, N, device="cuda").to(torch.bfloat16).requires_grad_(True)
    res = torch.randn(M, N, device="cuda").to(torch.bfloat16).requires_grad_(True)
    norm = rrn.RMSNorm(N, eps)
    with torch.no_grad():
        norm.weight.copy_(1.0 + 0.1 * torch.randn(N, device="cuda"))
    y, ro = norm(x, res)
    dy = torch.randn_like(y)
    dro = torch.randn_like(ro)
    torch.autograd.backward([y, ro], [dy, dro])
    # the same through the C entry points
    y2, ro2, rstd = rrn.add_rms_norm(x.detach(), res.detach(), norm.weight.detach(), eps)
    d_r, dw = rrn.add_rms_norm_backward(dy, dro, ro2, norm.weight.detach(), rstd, eps)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(ro, ro2)
    assert torch.equal(x.grad, d_r) and torch.equal(res.grad, d_r)
    assert torch.equal(norm.weight.grad, dw.to(torch.bfloat16))
    # plain RMSNorm through autograd
    x.grad = None
    norm.weight.grad = None
    y3 = norm(x)
    y3.backward(dy)
    y4, rstd4 = rrn.rms_norm(x.detach(), norm.weight.detach(), eps)
    dx4, dw4 = rrn.rms_norm_backward(dy, x.detach(), norm.weight.detach(), rstd4, eps)
    assert torch.equal(y3, y4) and torch.equal(x.grad, dx4)
    assert torch.equal(norm.weight.grad, dw4.to(torch.bfloat16))
