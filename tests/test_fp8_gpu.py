"""GPU parity of RMSNorm (+ residual add) feeding fp8 e4m3 codes with a per-row scale.

The codes are integers decided by rounding: where the exact target y / scale is farther than
a small relative margin from every e4m3 rounding midpoint, the GPU code must equal the oracle's;
within that margin (fp32 arithmetic can land on either side) either neighbouring code is valid,
and the dequantised value must still be within half a step. scale and rstd are checked with the
rstd bound; residual_out bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import residual_rmsnorm_row_gb300 as rrn
import synth
from gpu_util import bits_of, check_rstd, to_dev, to_host

pytestmark = pytest.mark.gpu

# relative distance to a midpoint below which both neighbouring codes are accepted: well above
# the fp32 error of y * (448 / amax) (a few ulps, ~1e-6)
MARGIN = 1e-5


def e4m3_table():
    codes = np.arange(256, dtype=np.uint8)
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def check_codes(q_gpu: np.ndarray, v_ref: np.ndarray, q_ref: np.ndarray, what: str):
    table = e4m3_table()
    pos = np.sort(table[:0x7F])                      # non-negative finite values
    mids = (pos[:-1] + pos[1:]) / 2
    a = np.abs(v_ref)
    k = np.clip(np.searchsorted(mids, a), 0, len(mids) - 1)
    near = np.minimum(np.abs(a - mids[k]), np.abs(a - mids[np.clip(k - 1, 0, len(mids) - 1)]))
    ambiguous = near <= MARGIN * np.maximum(a, 2.0 ** -9)
    exact_ok = (q_gpu == q_ref) | ambiguous
    assert exact_ok.all(), (f"{what}: {int((~exact_ok).sum())} codes differ away from a midpoint; "
                            f"first at {np.argwhere(~exact_ok)[0].tolist()}")
    # ambiguous ones: a neighbour of the same sign, within half a step of the target
    gv = table[q_gpu]
    assert not np.isnan(gv).any(), f"{what}: NaN code"
    # every such code is checked: its sign, and its distance to the target against half the
    # step between the two codes that bracket the target
    sel = ambiguous & (q_gpu != q_ref)
    t = v_ref[sel]
    g = gv[sel]
    j = np.searchsorted(pos, np.abs(t))
    step = pos[np.minimum(j, len(pos) - 1)] - pos[np.maximum(j - 1, 0)]
    bad = (np.abs(g - t) > step / 2 * (1 + 1e-3)) | ((g != 0) & (np.sign(g) != np.sign(t)))
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {t.size} codes near a midpoint are not a "
                           f"neighbour within half a step")


def run(h, dtype, eps, fused, launch=None):
    x = to_dev(h["x"], dtype)
    w = to_dev(h["w"], dtype)
    M, N = x.shape
    res = to_dev(h["residual"], dtype) if fused else None
    ro = torch.full_like(x, float("nan")) if fused else None
    q = torch.full((M, N), 0x7F, dtype=torch.uint8, device="cuda")
    scale = torch.full((M,), float("nan"), device="cuda")
    rstd = torch.full((M,), float("nan"), device="cuda")
    rrn.rmsnorm_fwd_fp8(x, res, ro, w, q, scale, rstd, eps, launch=launch)
    torch.cuda.synchronize()
    return q, scale, rstd, ro


def compare(h, dtype, eps, fused, q, scale, rstd, ro, what=""):
    r_ref, v_ref, q_ref, s_ref, rs_ref = oracle.rmsnorm_quant_fp8(
        h["x"], h["residual"] if fused else None, h["w"], eps)
    check_codes(q.cpu().numpy(), v_ref, q_ref, f"codes {what}")
    check_rstd(rstd.cpu().numpy().astype(np.float64), rs_ref, "rstd")
    s = scale.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(s - s_ref) <= 1e-5 * s_ref), f"scale {what}"
    if fused:
        assert np.array_equal(to_host(ro), bits_of(r_ref.astype(np.float32), dtype))


def test_fp8_fused_full_size():
    wl = synth.get("add_rmsnorm_fwd_16384x4096_bf16")
    h = synth.make(wl)
    q, scale, rstd, ro = run(h, "bf16", wl.eps, True)
    for s in range(0, wl.M, 2048):
        sl = slice(s, s + 2048)
        hh = {k: h[k][sl] for k in ("x", "residual")}
        hh["w"] = h["w"]
        compare(hh, "bf16", wl.eps, True, q[sl], scale[sl], rstd[sl], ro[sl], f"rows {s}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1, 7, 1000, 1024, 2048, 4095, 4096, 7168, 8192, 20000])
def test_fp8_variants(dtype, N):
    M = 61
    for fused in (False, True):
        wl = synth.Workload("fp8", "add_rmsnorm_fwd" if fused else "rmsnorm_fwd", M, N, dtype,
                            1e-6, 101, res_sigma=2.0)
        h = synth.make(wl)
        V = 8 if dtype == "bf16" else 4
        launches = [None, rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0), rrn.Launch(rrn.VARIANT_STREAM, 0, 64, 5)]
        if N % V == 0:
            nvec = N // V
            for vpt in (1, 2, 4, 8):
                thr = -(-(-(-nvec // vpt)) // 32) * 32
                if thr <= (256 if vpt == 8 else 512 if vpt == 4 else 1024):
                    launches += [rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 0),
                                 rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 7)]
            # rows split over clusters (a CTA's slice may be empty; at most 8 x 256 vectors a CTA)
            if 2 <= nvec <= 2 * 2048:
                launches += [rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 0, 0, 2)]
                if -(-nvec // 2) <= 1024:
                    launches += [rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 1, 0, 6, 0, 2)]
            if 8 <= nvec <= 8 * 2048:
                launches += [rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 0, 0, 8)]
            if nvec <= 256:  # one row per warp: a grid for every row, and 3 CTAs of 2 warps walking rows
                vpt = next(v for v in (1, 2, 4, 8) if 32 * v >= nvec)
                launches += [rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 128, 0), rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 64, 3)]
        for launch in launches:
            q, scale, rstd, ro = run(h, dtype, wl.eps, fused, launch)
            compare(h, dtype, wl.eps, fused, q, scale, rstd, ro, str(launch))


def _warp_launch(N):
    # one row per warp where a warp holds the row (bf16: 8 values a vector, 8 vectors a lane)
    return [rrn.Launch(rrn.VARIANT_ROW_WARP, 0, 64, 0)] if N <= 2048 else []


@pytest.mark.parametrize("N", [4096, 1024])
def test_fp8_zero_and_extreme_rows(N):
    rng = np.random.default_rng(102)
    rows = np.stack([np.zeros(N, np.float32), rng.standard_normal(N).astype(np.float32) * 1e30,
                     np.full(N, 2.0, np.float32), rng.standard_normal(N).astype(np.float32)])
    h = {"x": bits_of(rows, "bf16"), "w": bits_of(np.ones(N, np.float32), "bf16")}
    for launch in [None, rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0),
                   rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 0, 0, 4)] + _warp_launch(N):
        q, scale, rstd, _ = run(h, "bf16", 1e-6, False, launch)
        compare(h, "bf16", 1e-6, False, q, scale, rstd, None, str(launch))
        assert float(scale[0]) == 0.0 and int(q[0].max()) == 0


@pytest.mark.parametrize("N", [4096, 1024])
def test_fp8_row_whose_r_times_w_overflows(N):
    # |r| near 1e38 with w = 8: r * w is beyond fp32 although y = r * rstd * w is about 8
    rng = np.random.default_rng(103)
    z = np.clip(rng.standard_normal(N), -3.0, 3.0).astype(np.float32)  # |r| <= 3e38 stays finite
    rows = np.stack([z * np.float32(1e38), rng.standard_normal(N).astype(np.float32)])
    h = {"x": bits_of(rows, "bf16"), "w": bits_of(np.full(N, 8.0, np.float32), "bf16")}
    for launch in [None, rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0),
                   rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 0, 0, 4)] + _warp_launch(N):
        q, scale, rstd, _ = run(h, "bf16", 1e-6, False, launch)
        compare(h, "bf16", 1e-6, False, q, scale, rstd, None, str(launch))


@pytest.mark.parametrize("dtype,N", [("bf16", 16384), ("bf16", 32768), ("bf16", 65536), ("bf16", 131072),
                                     ("f32", 16384)])
def test_fp8_wide_rows(dtype, N):
    """Rows wider than one CTA holds: split over clusters (automatic up to 8 CTAs of 2048
    vectors), the 128-bit two-pass kernel beyond."""
    M = 40
    for fused in (False, True):
        wl = synth.Workload("fp8-wide", "add_rmsnorm_fwd" if fused else "rmsnorm_fwd", M, N, dtype,
                            1e-6, 104, res_sigma=2.0)
        h = synth.make(wl)
        for launch in (None, rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 0, 0, 8),
                       rrn.Launch(rrn.VARIANT_STREAM, 0, 1024, 0)):
            q, scale, rstd, ro = run(h, dtype, wl.eps, fused, launch)
            compare(h, dtype, wl.eps, fused, q, scale, rstd, ro, f"{N} {launch}")


@pytest.mark.parametrize("dtype,N", [("bf16", 4096), ("f32", 4096), ("bf16", 4095), ("bf16", 32768), ("bf16", 1024)])
def test_fp8_in_place(dtype, N):
    """residual_out written over residual, and over x."""
    M = 96
    wl = synth.Workload("fp8-alias", "add_rmsnorm_fwd", M, N, dtype, 1e-6, 105, res_sigma=2.0)
    h = synth.make(wl)
    r_ref, v_ref, q_ref, s_ref, rs_ref = oracle.rmsnorm_quant_fp8(h["x"], h["residual"], h["w"], wl.eps)
    r_bits = bits_of(r_ref.astype(np.float32), dtype)
    w = to_dev(h["w"], dtype)
    V = 8 if dtype == "bf16" else 4
    launches = [None, rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0)]
    if N % V == 0:
        launches += [rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 0, 0, 4)]
        if N // V <= 1024:
            launches += [rrn.Launch(rrn.VARIANT_ROW_CTA, 0, 0, 0)]
        if N // V <= 256:
            launches += [rrn.Launch(rrn.VARIANT_ROW_WARP, 0, 128, 0)]
    for launch in launches:
        for target in ("residual", "x"):
            x, res = to_dev(h["x"], dtype), to_dev(h["residual"], dtype)
            ro = res if target == "residual" else x
            q = torch.full((M, N), 0x7F, dtype=torch.uint8, device="cuda")
            scale = torch.full((M,), float("nan"), device="cuda")
            rstd = torch.full((M,), float("nan"), device="cuda")
            rrn.rmsnorm_fwd_fp8(x, res, ro, w, q, scale, rstd, wl.eps, launch=launch)
            torch.cuda.synchronize()
            assert np.array_equal(to_host(ro), r_bits), f"residual_out over {target}, {launch}"
            check_codes(q.cpu().numpy(), v_ref, q_ref, f"codes (residual_out over {target}), {launch}")
            check_rstd(rstd.cpu().numpy().astype(np.float64), rs_ref, "rstd")
            s = scale.cpu().numpy().astype(np.float64)
            assert np.all(np.abs(s - s_ref) <= 1e-5 * s_ref), f"scale {launch}"


def test_fp8_plans():
    """The forward's layouts: one row per warp for short rows over many rows, one row per CTA, cluster split for wide rows with a residual (and
    beyond 2048 vectors without one; 256-thread CTAs for chunks above 512 vectors), the 128-bit
    two-pass kernel beyond 16384 vectors."""
    def plan(M, N, fused):
        x = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        w = torch.empty(N, device="cuda", dtype=torch.bfloat16)
        q = torch.empty(M, N, device="cuda", dtype=torch.uint8)
        return rrn.plan_fwd_fp8(x, w, q, x if fused else None, x if fused else None)

    p = plan(16384, 4096, True)
    assert (p.variant, p.vpt, p.threads) == (rrn.VARIANT_ROW_CTA, 4, 128), p
    p = plan(65536, 1024, True)  # short rows over many rows: one row per warp
    assert (p.variant, p.vpt, p.threads, p.ctas) == (rrn.VARIANT_ROW_WARP, 4, 128, 65536 // 4), p
    p = plan(32768, 2048, False)
    assert (p.variant, p.vpt, p.threads) == (rrn.VARIANT_ROW_WARP, 8, 128), p
    p = plan(16384, 16384, True)
    assert (p.variant, p.cluster) == (rrn.VARIANT_ROW_CLUSTER, 4), p
    p = plan(16384, 16384, False)
    assert (p.variant, p.vpt) == (rrn.VARIANT_ROW_CTA, 8), p
    p = plan(4096, 65536, True)
    assert (p.variant, p.cluster, p.vpt, p.threads) == (rrn.VARIANT_ROW_CLUSTER, 8, 4, 256), p
    p = plan(2048, 131072, True)
    assert (p.variant, p.cluster, p.vpt, p.threads) == (rrn.VARIANT_ROW_CLUSTER, 8, 4, 512), p
    p = plan(1024, 262144, True)
    assert (p.variant, p.threads, p.vec) == (rrn.VARIANT_STREAM, 1024, 1), p
    p = plan(64, 4095, False)
    assert p.variant == rrn.VARIANT_STREAM and p.vec == 0, p
