"""GPU parity of the LayerNorm variant (forward with residual and bias, backward with dw, db)
against the CPU fp64 oracle, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import residual_rmsnorm_row_gb300 as rrn
import synth
from gpu_util import (bits_of, bwd_cond, check_dw, check_mean, check_out, check_rstd, to_dev,
                      to_host, values)

pytestmark = pytest.mark.gpu
CHUNK = 2048


def ln_fwd(h, dtype, eps, fused, bias, launch=None):
    x = to_dev(h["x"], dtype)
    w = to_dev(h["w"], dtype)
    b = to_dev(h["b"], dtype) if bias else None
    M = x.shape[0]
    y = torch.full_like(x, float("nan"))
    mean = torch.full((M,), float("nan"), device="cuda")
    rstd = torch.full((M,), float("nan"), device="cuda")
    res = to_dev(h["residual"], dtype) if fused else None
    ro = torch.full_like(x, float("nan")) if fused else None
    rrn.layernorm_fwd(x, w, b, y, mean, rstd, eps, residual=res, residual_out=ro, launch=launch)
    torch.cuda.synchronize()
    return y, ro, mean, rstd


def compare(h, dtype, eps, fused, bias, y, ro, mean, rstd):
    M = h["x"].shape[0]
    for s in range(0, M, CHUNK):
        idx = np.arange(s, min(M, s + CHUNK))
        r_ref, y_ref, m_ref, rs_ref = oracle.add_layernorm_fwd(
            h["x"][idx], h["residual"][idx] if fused else None, h["w"], h["b"] if bias else None, eps)
        ti = torch.from_numpy(idx).cuda()
        check_out(values(y.index_select(0, ti)), y_ref, dtype, "LN y")
        check_rstd(rstd.index_select(0, ti).cpu().numpy().astype(np.float64), rs_ref, "LN rstd")
        check_mean(mean.index_select(0, ti).cpu().numpy().astype(np.float64), m_ref, rs_ref)
        if fused:
            assert np.array_equal(to_host(ro.index_select(0, ti)), bits_of(r_ref.astype(np.float32), dtype))


def test_layernorm_forward_full_size():
    wl = synth.get("add_layernorm_fwd_16384x4096_bf16")
    h = synth.make(wl)
    y, ro, mean, rstd = ln_fwd(h, "bf16", wl.eps, True, True)
    compare(h, "bf16", wl.eps, True, True, y, ro, mean, rstd)


def test_layernorm_backward_full_size():
    wl = synth.get("layernorm_bwd_16384x4096_bf16")
    h = synth.make(wl)
    x, w = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16")
    _, mean, rstd = rrn.layer_norm(x, w, to_dev(h["b"], "bf16"), wl.eps)
    dx, dw, db = rrn.layer_norm_backward(to_dev(h["dy"], "bf16"), x, w, mean, rstd, wl.eps,
                                         d_residual_out=to_dev(h["d_ro"], "bf16"))
    torch.cuda.synchronize()
    ref_dx, ref_dw, ref_db = oracle.add_layernorm_bwd(h["dy"], h["d_ro"], h["x"], h["w"], wl.eps)
    check_out(values(dx), ref_dx, "bf16", "LN dx")
    check_dw(dw.cpu().numpy().astype(np.float64), ref_dw, "LN dw")
    check_dw(db.cpu().numpy().astype(np.float64), ref_db, "LN db")


def test_layernorm_backward_plain_full_size():
    # no gradient at residual_out: the two-input-row backward, in the layout the benchmark times
    wl = synth.get("layernorm_bwd_plain_16384x4096_bf16")
    h = synth.make(wl)
    x, w = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16")
    _, mean, rstd = rrn.layer_norm(x, w, to_dev(h["b"], "bf16"), wl.eps)
    dx, dw, db = rrn.layer_norm_backward(to_dev(h["dy"], "bf16"), x, w, mean, rstd, wl.eps)
    torch.cuda.synchronize()
    ref_dx, ref_dw, ref_db = oracle.add_layernorm_bwd(h["dy"], None, h["x"], h["w"], wl.eps)
    check_out(values(dx), ref_dx, "bf16", "LN dx")
    check_dw(dw.cpu().numpy().astype(np.float64), ref_dw, "LN dw")
    check_dw(db.cpu().numpy().astype(np.float64), ref_db, "LN db")


def _fwd_launches(dtype, N):
    V = 8 if dtype == "bf16" else 4
    out = [None, rrn.Launch(rrn.VARIANT_STREAM, 0, 128, 0), rrn.Launch(rrn.VARIANT_STREAM, 0, 1024, 7)]
    if N % V == 0:
        nvec = N // V
        for vpt in (1, 2, 4, 8):
            thr = -(-(-(-nvec // vpt)) // 32) * 32
            if thr <= (256 if vpt == 8 else 512 if vpt == 4 else 1024):
                out += [rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 0), rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 9)]
        if nvec <= 256:  # one row per warp: a grid for every row, and 5 CTAs of 2 warps walking rows
            vpt = next(v for v in (1, 2, 4, 8) if 32 * v >= nvec)
            out += [rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 128, 0), rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 64, 5)]
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1, 7, 8, 256, 1000, 1024, 2048, 4095, 4096, 7168, 8192, 20000])
def test_layernorm_forward_variants(dtype, N):
    M = 67
    for fused in (False, True):
        wl = synth.Workload("ln", "add_layernorm_fwd" if fused else "layernorm_fwd", M, N, dtype,
                            1e-5, 91, x_mean=0.5)
        h = synth.make(wl)
        for bias in (True, False):
            for launch in _fwd_launches(dtype, N):
                y, ro, mean, rstd = ln_fwd(h, dtype, wl.eps, fused, bias, launch)
                compare(h, dtype, wl.eps, fused, bias, y, ro, mean, rstd)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [4, 8, 1000, 4096, 8192])
def test_layernorm_forward_in_place(dtype, N):
    """residual_out written over residual, and over x; y written over x (the plain op)."""
    M = 300
    wl = synth.Workload("ln-alias", "add_layernorm_fwd", M, N, dtype, 1e-5, 93, x_mean=0.5)
    h = synth.make(wl)
    r_ref, y_ref, m_ref, rs_ref = oracle.add_layernorm_fwd(h["x"], h["residual"], h["w"], h["b"], wl.eps)
    y2_ref = oracle.add_layernorm_fwd(h["x"], None, h["w"], h["b"], wl.eps)[1]
    w, b = to_dev(h["w"], dtype), to_dev(h["b"], dtype)
    r_bits = bits_of(r_ref.astype(np.float32), dtype)
    for launch in _fwd_launches(dtype, N):
        for target in ("residual", "x"):
            x, res = to_dev(h["x"], dtype), to_dev(h["residual"], dtype)
            y = torch.empty_like(x)
            mean, rstd = torch.empty(M, device="cuda"), torch.empty(M, device="cuda")
            ro = res if target == "residual" else x
            rrn.layernorm_fwd(x, w, b, y, mean, rstd, wl.eps, residual=res, residual_out=ro, launch=launch)
            torch.cuda.synchronize()
            assert np.array_equal(to_host(ro), r_bits), f"residual_out over {target}, {launch}"
            check_out(values(y), y_ref, dtype, f"LN y (residual_out over {target}), {launch}")
            check_rstd(rstd.cpu().numpy().astype(np.float64), rs_ref, "LN rstd")
            check_mean(mean.cpu().numpy().astype(np.float64), m_ref, rs_ref)
        x = to_dev(h["x"], dtype)
        mean, rstd = torch.empty(M, device="cuda"), torch.empty(M, device="cuda")
        rrn.layernorm_fwd(x, w, b, x, mean, rstd, wl.eps, launch=launch)
        torch.cuda.synchronize()
        check_out(values(x), y2_ref, dtype, f"LN y over x, {launch}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1, 8, 9, 256, 512, 1000, 1024, 4095, 4096, 7168, 8192])
def test_layernorm_backward_variants(dtype, N):
    M = 75
    wl = synth.Workload("ln-bwd", "layernorm_bwd", M, N, dtype, 1e-5, 92, x_mean=0.5)
    h = synth.make(wl)
    x, w = to_dev(h["x"], dtype), to_dev(h["w"], dtype)
    _, mean, rstd = rrn.layer_norm(x, w, None, wl.eps)
    V = 8 if dtype == "bf16" else 4
    launches = [None, rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0), rrn.Launch(rrn.VARIANT_STREAM, 0, 64, 5)]
    if N % V == 0:
        nvec = N // V
        for vpt in (1, 2, 4):
            thr = -(-(-(-nvec // vpt)) // 32) * 32
            if thr <= (256 if vpt == 4 else 512):
                launches += [rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 0), rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 6),
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 0, 0),     # ring depth planned
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 7, 2),     # one row in flight,
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 5, 4),     # 10-15 rows a CTA
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 0, 3)]
    if N % V == 0 and N // V >= 512:
        # each row split over a cluster (CTA q owning a column slice); 3 x C CTAs: ragged rows
        for C in (2, 4, 8):
            if -(-(N // V) // C) <= 1024:
                launches += [rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 0, 0, C),
                             rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 3 * C, 0, C)]
    if N % V == 0 and N // V <= 128:
        # one row per warp: the planner's grid, and 4 CTAs of 2 warps walking rows
        vpt = next(v for v in (1, 2, 4) if 32 * v >= N // V)
        launches += [rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 128, 0), rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 64, 4)]
    cond0 = bwd_cond(h["x"], h["dy"], h["w"], wl.eps, layernorm=True)
    for with_dro in (True, False):
        ref_dx, ref_dw, ref_db = oracle.add_layernorm_bwd(h["dy"], h["d_ro"] if with_dro else None,
                                                          h["x"], h["w"], wl.eps)
        cond = cond0 + (np.abs(oracle.decode(h["d_ro"])) if with_dro else 0.0)
        for launch in launches:
            dx = torch.full_like(x, float("nan"))
            dw = torch.full((N,), float("nan"), device="cuda")
            db = torch.full((N,), float("nan"), device="cuda")
            ws = torch.empty(max(rrn.layernorm_bwd_workspace_bytes(M, N, x.dtype), 8 * x.numel()) // 4,
                             device="cuda")
            rrn.layernorm_bwd(to_dev(h["dy"], dtype), to_dev(h["d_ro"], dtype) if with_dro else None,
                              x, w, mean, rstd, dx, dw, db, ws, wl.eps, launch=launch)
            torch.cuda.synchronize()
            check_out(values(dx), ref_dx, dtype, f"LN dx {launch}", cond)
            check_dw(dw.cpu().numpy().astype(np.float64), ref_dw, f"LN dw {launch}")
            check_dw(db.cpu().numpy().astype(np.float64), ref_db, f"LN db {launch}")


@pytest.mark.parametrize("N,launch", [(4096, None), (1024, rrn.Launch(rrn.VARIANT_ROW_WARP, 0, 128, 0))],
                         ids=["auto", "row-per-warp"])
def test_layernorm_backward_in_place(N, launch):
    """dx written over dy, over the gradient at residual_out, and over x."""
    M = 70
    wl = synth.Workload("ln-bwd-alias", "layernorm_bwd", M, N, "bf16", 1e-5, 94, x_mean=0.5)
    h = synth.make(wl)
    ref_dx, ref_dw, ref_db = oracle.add_layernorm_bwd(h["dy"], h["d_ro"], h["x"], h["w"], wl.eps)
    cond = bwd_cond(h["x"], h["dy"], h["w"], wl.eps, layernorm=True) + np.abs(oracle.decode(h["d_ro"]))
    w = to_dev(h["w"], "bf16")
    x0 = to_dev(h["x"], "bf16")
    _, mean, rstd = rrn.layer_norm(x0, w, None, wl.eps)
    ws = torch.empty(max(rrn.layernorm_bwd_workspace_bytes(M, N, x0.dtype), 8 * M * N) // 4, device="cuda")
    for target in ("dy", "d_ro", "x"):
        x, dy, dro = x0.clone(), to_dev(h["dy"], "bf16"), to_dev(h["d_ro"], "bf16")
        out = {"dy": dy, "d_ro": dro, "x": x}[target]
        dw = torch.empty(N, device="cuda")
        db = torch.empty(N, device="cuda")
        rrn.layernorm_bwd(dy, dro, x, w, mean, rstd, out, dw, db, ws, wl.eps, launch=launch)
        torch.cuda.synchronize()
        check_out(values(out), ref_dx, "bf16", f"LN dx written over {target}, {launch}", cond)
        check_dw(dw.cpu().numpy().astype(np.float64), ref_dw, f"LN dw ({target})")
        check_dw(db.cpu().numpy().astype(np.float64), ref_db, f"LN db ({target})")


def test_layernorm_backward_ring_needs_two_stages():
    """The backward's ring refills a slot one row late: one stage is refused before any launch."""
    M, N = 64, 4096
    x = torch.zeros(M, N, device="cuda", dtype=torch.bfloat16)
    w = torch.ones(N, device="cuda", dtype=torch.bfloat16)
    mean, rstd = torch.zeros(M, device="cuda"), torch.ones(M, device="cuda")
    dx, dw, db = torch.empty_like(x), torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    ws = torch.empty(rrn.layernorm_bwd_workspace_bytes(M, N, x.dtype) // 4, device="cuda")
    with pytest.raises(rrn.RRNError):
        rrn.layernorm_bwd(x, None, x, w, mean, rstd, dx, dw, db, ws, 1e-5,
                          launch=rrn.Launch(rrn.VARIANT_ROW_TMA, 2, 256, 0, 1))
    # the rows of a CTA fewer than the stages, and a single CTA walking every row
    for launch in (rrn.Launch(rrn.VARIANT_ROW_TMA, 2, 256, 0, 4), rrn.Launch(rrn.VARIANT_ROW_TMA, 4, 128, 1, 3)):
        rrn.layernorm_bwd(x, x, x, w, mean, rstd, dx, dw, db, ws, 1e-5, launch=launch)
        torch.cuda.synchronize()
        assert torch.equal(dx, x) and float(dw.abs().max()) == 0.0 and float(db.abs().max()) == 0.0
    assert rrn.device_faults() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1024, 4096, 20000])
def test_layernorm_extreme_rows(dtype, N):
    rng = np.random.default_rng(93)
    base = rng.standard_normal((6, N)).astype(np.float32)
    # The statistics are taken relative to the mean of the row's first 8 values; first values
    # far from the mean compared with the spread send the row to the two-pass path, first
    # values 3.5 sigma away keep it on the one-step path with about four bits of cancellation.
    first_outlier = base[1].copy()
    first_outlier[:8] = 50.0
    first_far = base[2].copy()
    first_far[:8] = 3.5
    rows = np.stack([
        base[0] * 1e36 + 3e36,           # sum and squared deviations overflow fp32
        np.full(N, 3.0, np.float32),     # constant row: xhat = 0, y = b
        np.zeros(N, np.float32),
        base[3] * 1e-30,                 # tiny deviations
        base[4] + 100.0,                 # large offset relative to the spread
        base[5],
        first_outlier,
        first_far,
        base[5] * 0.01 + 1e4,            # offset a million times the spread
    ]).astype(np.float32)
    h = {"x": bits_of(rows, dtype), "w": bits_of((1 + 0.1 * rng.standard_normal(N)).astype(np.float32), dtype),
         "b": bits_of((0.1 * rng.standard_normal(N)).astype(np.float32), dtype)}
    for launch in (None, rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0)):
        y, _, mean, rstd = ln_fwd(h, dtype, 1e-5, False, True, launch)
        compare(h, dtype, 1e-5, False, True, y, None, mean, rstd)


@pytest.mark.parametrize("dtype,N", [("bf16", 16384), ("bf16", 32768), ("f32", 16384)])
def test_layernorm_backward_wide_rows(dtype, N):
    # rows too wide for one CTA's dw and db registers: the automatic plan splits each row over
    # a thread-block cluster
    M = 300
    wl = synth.Workload("ln-bwd-wide", "layernorm_bwd", M, N, dtype, 1e-5, 400 + N, x_mean=0.5)
    h = synth.make(wl)
    x, w = to_dev(h["x"], dtype), to_dev(h["w"], dtype)
    _, mean, rstd = rrn.layer_norm(x, w, None, wl.eps)
    cond0 = bwd_cond(h["x"], h["dy"], h["w"], wl.eps, layernorm=True)
    for with_dro in (True, False):
        ref_dx, ref_dw, ref_db = oracle.add_layernorm_bwd(h["dy"], h["d_ro"] if with_dro else None,
                                                          h["x"], h["w"], wl.eps)
        cond = cond0 + (np.abs(oracle.decode(h["d_ro"])) if with_dro else 0.0)
        dx = torch.full_like(x, float("nan"))
        dw = torch.full((N,), float("nan"), device="cuda")
        db = torch.full((N,), float("nan"), device="cuda")
        ws = torch.empty(rrn.layernorm_bwd_workspace_bytes(M, N, x.dtype) // 4, device="cuda")
        rrn.layernorm_bwd(to_dev(h["dy"], dtype), to_dev(h["d_ro"], dtype) if with_dro else None,
                          x, w, mean, rstd, dx, dw, db, ws, wl.eps)
        torch.cuda.synchronize()
        check_out(values(dx), ref_dx, dtype, "LN dx", cond)
        check_dw(dw.cpu().numpy().astype(np.float64), ref_dw, "LN dw")
        check_dw(db.cpu().numpy().astype(np.float64), ref_db, "LN db")


def test_layernorm_plans():
    """The automatic layouts the measurements chose (vectors per thread, ring or registers, ring
    slots, cluster split), through the C plan queries (tensors never read)."""
    def bwd(M, N, fused):
        x = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        w = torch.empty(N, device="cuda", dtype=torch.bfloat16)
        return rrn.plan_layernorm_bwd(x, x, w, x, x if fused else None)

    p = bwd(16384, 4096, True)
    assert (p.variant, p.vpt, p.threads, p.stages) == (rrn.VARIANT_ROW_TMA, 2, 256, 2), p
    p = bwd(16384, 4096, False)
    assert (p.variant, p.vpt, p.threads, p.stages) == (rrn.VARIANT_ROW_TMA, 4, 128, 2), p
    p = bwd(32768, 2048, False)
    assert (p.variant, p.vpt, p.threads) == (rrn.VARIANT_ROW_TMA, 4, 64), p
    p = bwd(65536, 1024, False)  # short rows over many rows: one row per warp
    assert (p.variant, p.vpt, p.threads) == (rrn.VARIANT_ROW_WARP, 4, 128), p
    p = bwd(131072, 512, True)
    assert (p.variant, p.vpt, p.threads) == (rrn.VARIANT_ROW_WARP, 2, 128), p
    p = bwd(8192, 8192, True)
    assert (p.variant, p.vpt, p.threads) == (rrn.VARIANT_ROW_TMA, 4, 256) and p.stages >= 2, p
    p = bwd(8192, 16384, True)
    assert (p.variant, p.cluster, p.vpt, p.threads) == (rrn.VARIANT_ROW_CLUSTER, 8, 2, 128), p
    p = bwd(8192, 16384, False)
    assert (p.variant, p.cluster, p.vpt, p.threads) == (rrn.VARIANT_ROW_CLUSTER, 8, 2, 128), p
    p = bwd(4096, 32768, True)
    assert (p.variant, p.cluster, p.vpt, p.threads) == (rrn.VARIANT_ROW_CLUSTER, 8, 2, 256), p
    p = bwd(64, 4095, False)
    assert p.variant == rrn.VARIANT_STREAM and p.vec == 0, p
    x = torch.empty(16384, 4096, device="cuda", dtype=torch.bfloat16)
    w = torch.empty(4096, device="cuda", dtype=torch.bfloat16)
    p = rrn.plan_layernorm_fwd(x, w, x, w, x, x)
    assert (p.variant, p.vpt, p.threads) == (rrn.VARIANT_ROW_CTA, 4, 128), p
    # wider rows: at most 4 vectors a thread, more threads instead
    for N, thr in ((2048, 64), (6144, 192), (8192, 256), (12288, 384), (16384, 512)):
        x = torch.empty(4096, N, device="cuda", dtype=torch.bfloat16)
        w = torch.empty(N, device="cuda", dtype=torch.bfloat16)
        p = rrn.plan_layernorm_fwd(x, w, x, w, x, x)
        assert (p.variant, p.vpt, p.threads) == (rrn.VARIANT_ROW_CTA, 4, thr), (N, p)
    # short rows over many rows: one row per warp
    for N, vpt in ((512, 2), (768, 4), (1024, 4)):
        x = torch.empty(65536, N, device="cuda", dtype=torch.bfloat16)
        w = torch.empty(N, device="cuda", dtype=torch.bfloat16)
        p = rrn.plan_layernorm_fwd(x, w, x, w, x, x)
        assert (p.variant, p.vpt, p.threads, p.ctas) == (rrn.VARIANT_ROW_WARP, vpt, 128, 65536 // 4), (N, p)
