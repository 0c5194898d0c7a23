"""GPU parity: the CUDA path, called through the C ABI, against the CPU fp64 oracle.

Every comparison is element by element on the same seeded host inputs, with the bounds of
``gpu_util``. The named workloads run at their full sizes in the automatic launch
configuration (the one the benchmark times); the full-size forward outputs are compared in row
chunks against the oracle, so every element is checked.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import residual_rmsnorm_row_gb300 as rrn
import synth
from gpu_util import (bwd_cond, check_dw, check_out, check_rstd, to_dev, to_host, values, bits_of,
                      TORCH)

pytestmark = pytest.mark.gpu

CHUNK_ROWS = 2048


def fwd_case(x_h, res_h, w_h, dtype, eps, launch=None, inplace=None):
    """Run one forward on the GPU; return device tensors (y, residual_out or None, rstd)."""
    x = to_dev(x_h, dtype)
    w = to_dev(w_h, dtype)
    M = x.shape[0]
    y = torch.full_like(x, float("nan"))
    rstd = torch.full((M,), float("nan"), device="cuda")
    if res_h is None:
        rrn.add_rmsnorm_fwd_ex(x, None, None, w, y, rstd, eps, launch)
        ro = None
    else:
        res = to_dev(res_h, dtype)
        ro = torch.full_like(x, float("nan"))
        rrn.add_rmsnorm_fwd_ex(x, res, ro, w, y, rstd, eps, launch)
    torch.cuda.synchronize()
    return y, ro, rstd


def compare_fwd(x_h, res_h, w_h, dtype, eps, y, ro, rstd, rows=None):
    """Compare GPU outputs with the oracle over all rows (in chunks) or the given rows."""
    M = x_h.shape[0]
    worst = 0.0
    starts = range(0, M, CHUNK_ROWS) if rows is None else [None]
    for s in starts:
        idx = np.arange(s, min(M, s + CHUNK_ROWS)) if rows is None else np.asarray(rows)
        r_ref, y_ref, rs_ref = oracle.add_rmsnorm_fwd(x_h[idx], None if res_h is None else res_h[idx],
                                                      w_h, eps)
        ti = torch.from_numpy(idx).cuda()
        worst = max(worst, check_out(values(y.index_select(0, ti)), y_ref, dtype, "y"))
        worst = max(worst, check_rstd(rstd.index_select(0, ti).cpu().numpy().astype(np.float64), rs_ref))
        if res_h is not None:
            got_r = values(ro.index_select(0, ti))
            worst = max(worst, check_out(got_r, r_ref, dtype, "residual_out"))
            # residual_out is the sum rounded once: it must equal the correctly rounded sum.
            # The fp64 sum of two bf16/fp32 values is exact here, so rounding it to fp32 gives
            # the kernel's fp32 r bit for bit, and rounding that to bf16 its residual_out.
            want = bits_of(r_ref.astype(np.float32), dtype)
            assert np.array_equal(to_host(ro.index_select(0, ti)), want), \
                "residual_out is not the sum rounded once to the storage type"
    return worst


# ------------------------------------------------------------------ the named workloads
FWD_WORKLOADS = [n for n, w in synth.WORKLOADS.items() if w.op in ("rmsnorm_fwd", "add_rmsnorm_fwd")]


@pytest.mark.parametrize("name", FWD_WORKLOADS)
def test_forward_workload_full_size(name):
    wl = synth.get(name)
    h = synth.make(wl)
    res_h = h.get("residual")
    y, ro, rstd = fwd_case(h["x"], res_h, h["w"], wl.dtype, wl.eps)
    worst = compare_fwd(h["x"], res_h, h["w"], wl.dtype, wl.eps, y, ro, rstd)
    print(f"{name}: max err/bound {worst:.3f}")


def test_backward_workload_full_size():
    wl = synth.get("rmsnorm_bwd_16384x4096_bf16")
    h = synth.make(wl)
    x, w, dy = to_dev(h["x"], "bf16"), to_dev(h["w"], "bf16"), to_dev(h["dy"], "bf16")
    _, rstd = rrn.rms_norm(x, w, wl.eps)          # rstd from the GPU forward, as in training
    dx, dw = rrn.rms_norm_backward(dy, x, w, rstd, wl.eps)
    torch.cuda.synchronize()
    dx_ref, dw_ref = oracle.rmsnorm_bwd(h["dy"], h["x"], h["w"], wl.eps)
    a = check_out(values(dx), dx_ref, "bf16", "dx")
    b = check_dw(dw.cpu().numpy().astype(np.float64), dw_ref)
    print(f"bwd 16384x4096: dx max err/bound {a:.3f}, dw max err/bound {b:.3f}")


# ------------------------------------------------------------------ every kernel variant
def _variants(dtype, N, M):
    V = 8 if dtype == "bf16" else 4
    nvec = N // V
    out = []
    for vpt in (1, 2, 4, 8):
        lim = 256 if vpt == 8 else 512 if vpt == 4 else 1024
        thr = -(-nvec // vpt)
        thr = -(-thr // 32) * 32
        if N % V == 0 and thr <= lim:
            out.append(rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 0))
            out.append(rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 37))     # persistent, ragged
            for stages, ctas in ((0, 0), (1, 0), (2, 37), (3, 5)):
                out.append(rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, ctas, stages))
        if N % V == 0 and nvec <= 32 * vpt:
            out.append(rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 128, 0))
            out.append(rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 64, 5))
    if N % V == 0:
        for C in (2, 4, 8):
            chunk = -(-nvec // C)
            for vpt in (1, 4):
                thr = -(-(-(-chunk // vpt)) // 32) * 32
                if thr <= (512 if vpt == 4 else 1024):
                    out.append(rrn.Launch(rrn.VARIANT_ROW_CLUSTER, vpt, thr, 0, 0, C))
                    out.append(rrn.Launch(rrn.VARIANT_ROW_CLUSTER, vpt, thr, 3 * C, 0, C))
    out.append(rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0))
    out.append(rrn.Launch(rrn.VARIANT_STREAM, 0, 1024, 11))
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1024, 2048, 4096, 7168])
@pytest.mark.parametrize("fused", [False, True])
def test_every_variant(dtype, N, fused):
    M = 333
    wl = synth.Workload("variants", "add_rmsnorm_fwd" if fused else "rmsnorm_fwd", M, N, dtype,
                        1e-6, 7, res_sigma=2.0)
    h = synth.make(wl)
    for launch in _variants(dtype, N, M):
        y, ro, rstd = fwd_case(h["x"], h.get("residual"), h["w"], dtype, wl.eps, launch)
        compare_fwd(h["x"], h.get("residual"), h["w"], dtype, wl.eps, y, ro, rstd)


# ------------------------------------------------------------------ edge shapes
EDGE_N = [1, 7, 8, 9, 1000, 1024, 4095, 7168, 8192, 16384, 20000, 65536]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", EDGE_N)
@pytest.mark.parametrize("M", [1, 3, 130])
def test_edge_shapes_forward(dtype, N, M):
    for fused in (False, True):
        wl = synth.Workload("edge", "add_rmsnorm_fwd" if fused else "rmsnorm_fwd", M, N, dtype,
                            1e-5, 100 + N)
        h = synth.make(wl)
        y, ro, rstd = fwd_case(h["x"], h.get("residual"), h["w"], dtype, wl.eps)
        compare_fwd(h["x"], h.get("residual"), h["w"], dtype, wl.eps, y, ro, rstd)


# The automatic plan for wide rows when rows are not few (M >= 2 x SMs). Fused (two input
# rows): one row per CTA up to 1024 vectors, a cluster split of at most 512 vectors per CTA up
# to 4096 vectors, then clusters of 8 up to 8192. Plain (one input row, so twice the vectors for
# the same bytes in flight): one row per CTA up to 2048 vectors, cluster chunks of at most 1024
# up to 8192. Wider: the two-pass kernel (1024 threads from 8192 vectors or elements), as for
# unaligned rows.
R, C, S = rrn.VARIANT_ROW_CTA, rrn.VARIANT_ROW_CLUSTER, rrn.VARIANT_STREAM
WIDE_PLANS = [  # (dtype, N, fused, variant, cluster size or threads)
    ("bf16", 8192, True, R, None), ("bf16", 8192, False, R, None),
    ("bf16", 16384, True, C, 4), ("bf16", 16384, False, R, None),
    ("bf16", 24576, True, C, 8), ("bf16", 24576, False, C, 4),
    ("bf16", 32768, True, C, 8), ("bf16", 32768, False, C, 4),
    ("bf16", 40000, True, C, 8), ("bf16", 40000, False, C, 8),
    ("bf16", 65536, True, C, 8), ("bf16", 65536, False, C, 8),
    ("bf16", 80000, False, S, 1024),
    ("bf16", 9001, True, S, 1024), ("bf16", 9001, False, S, 1024),   # unaligned: element-wise
    ("f32", 16384, True, C, 8), ("f32", 16384, False, C, 4),
    ("f32", 32768, True, C, 8), ("f32", 32768, False, C, 8),
]


@pytest.mark.parametrize("dtype,N,fused,variant,extra", WIDE_PLANS)
def test_wide_rows_automatic_plan(dtype, N, fused, variant, extra):
    M = 400
    wl = synth.Workload("wide-plan", "add_rmsnorm_fwd" if fused else "rmsnorm_fwd", M, N, dtype,
                        1e-6, 200 + N, res_sigma=2.0)
    h = synth.make(wl)
    x, w = to_dev(h["x"], dtype), to_dev(h["w"], dtype)
    res = to_dev(h["residual"], dtype) if fused else None
    plan = rrn.plan_fwd(x, res, torch.empty_like(x) if fused else None, w, torch.empty_like(x))
    assert plan.variant == variant, plan.name
    if variant == rrn.VARIANT_ROW_CLUSTER:
        assert plan.cluster == extra and plan.ctas % extra == 0, plan.name
    if variant == rrn.VARIANT_STREAM:
        assert plan.threads == extra, plan.name
    y, ro, rstd = fwd_case(h["x"], h.get("residual"), h["w"], dtype, wl.eps)
    compare_fwd(h["x"], h.get("residual"), h["w"], dtype, wl.eps, y, ro, rstd)


def test_short_rows_forward_plan():
    """Many short rows: a row per warp up to 256 vectors plain, up to 128 fused (from 129 to 256
    vectors the fused forward takes a row per CTA)."""
    for N, fused, variant in ((1024, True, rrn.VARIANT_ROW_WARP), (1024, False, rrn.VARIANT_ROW_WARP),
                              (2048, True, rrn.VARIANT_ROW_CTA), (2048, False, rrn.VARIANT_ROW_WARP),
                              (1536, True, rrn.VARIANT_ROW_CTA)):
        x = torch.empty(32768, N, device="cuda", dtype=torch.bfloat16)
        w = torch.empty(N, device="cuda", dtype=torch.bfloat16)
        p = rrn.plan_fwd(x, x if fused else None, x if fused else None, w, x)
        assert p.variant == variant, (N, fused, p)


def test_empty_matrix():
    # M == 0: the forward writes nothing; the backward's dw (and LayerNorm's db) are sums over
    # no rows, which the oracle's definition makes zero - the GPU calls must overwrite them so.
    N = 4096
    x = torch.zeros(0, N, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    rstd = torch.full((1,), 5.0, device="cuda")
    rrn.rmsnorm_fwd(x, w, x, rstd[:0], 1e-6)
    rrn.add_rmsnorm_fwd(x, x, x, w, x, rstd[:0], 1e-6)
    empty = np.zeros((0, N), dtype=np.uint16)
    _, dw_ref = oracle.rmsnorm_bwd(empty, empty, to_host(w), 1e-6)
    _, dwf_ref = oracle.add_rmsnorm_bwd(empty, empty, empty, to_host(w), 1e-6)
    _, dwl_ref, db_ref = oracle.add_layernorm_bwd(empty, None, empty, to_host(w), 1e-5)
    assert dw_ref.shape == (N,)
    ws = torch.zeros(4, device="cuda")
    dw = torch.full((N,), 7.0, device="cuda")
    rrn.rmsnorm_bwd(x, x, w, rstd[:0], x, dw, ws, 1e-6)
    dwf = torch.full((N,), 7.0, device="cuda")
    rrn.add_rmsnorm_bwd(x, x, x, w, rstd[:0], x, dwf, ws, 1e-6)
    dwl = torch.full((N,), 7.0, device="cuda")
    db = torch.full((N,), 7.0, device="cuda")
    rrn.layernorm_bwd(x, None, x, w, rstd[:0], rstd[:0], x, dwl, db, ws, 1e-5)
    torch.cuda.synchronize()
    assert float(rstd[0]) == 5.0, "a forward with M == 0 wrote"
    for got, ref, what in ((dw, dw_ref, "rmsnorm_bwd dw"), (dwf, dwf_ref, "add_rmsnorm_bwd dw"),
                           (dwl, dwl_ref, "layernorm_bwd dw"), (db, db_ref, "layernorm_bwd db")):
        check_dw(got.cpu().numpy().astype(np.float64), ref, what)
        assert np.array_equal(got.cpu().numpy(), np.zeros(N, np.float32)), what


# ------------------------------------------------------------------ alignment and aliasing
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unaligned_base_pointers(dtype):
    M, N = 65, 4096
    wl = synth.Workload("unaligned", "add_rmsnorm_fwd", M, N, dtype, 1e-6, 21)
    h = synth.make(wl)
    t = TORCH[dtype]
    big = [torch.empty(M * N + 1, dtype=t, device="cuda") for _ in range(5)]
    x, res, ro, y = (b[1:].view(M, N) for b in big[:4])
    wbuf = torch.empty(N + 1, dtype=t, device="cuda")
    w = wbuf[1:]
    x.copy_(to_dev(h["x"], dtype))
    res.copy_(to_dev(h["residual"], dtype))
    w.copy_(to_dev(h["w"], dtype))
    rstd = torch.empty(M, device="cuda")
    plan = rrn.plan_fwd(x, res, ro, w, y)
    assert plan.vec == 0, "an unaligned base must take the element-wise path"
    rrn.add_rmsnorm_fwd(x, res, ro, w, y, rstd, wl.eps)
    torch.cuda.synchronize()
    compare_fwd(h["x"], h["residual"], h["w"], dtype, wl.eps, y, ro, rstd)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [2048, 4096, 20000, 4095])
def test_in_place_forms(dtype, N):
    M = 77
    wl = synth.Workload("alias", "add_rmsnorm_fwd", M, N, dtype, 1e-6, 31)
    h = synth.make(wl)
    r_ref, y_ref, rs_ref = oracle.add_rmsnorm_fwd(h["x"], h["residual"], h["w"], wl.eps)
    w = to_dev(h["w"], dtype)
    # residual_out written over residual
    x, res = to_dev(h["x"], dtype), to_dev(h["residual"], dtype)
    y = torch.empty_like(x)
    rstd = torch.empty(M, device="cuda")
    rrn.add_rmsnorm_fwd(x, res, res, w, y, rstd, wl.eps)
    torch.cuda.synchronize()
    check_out(values(res), r_ref, dtype, "residual_out==residual")
    check_out(values(y), y_ref, dtype, "y (residual_out==residual)")
    # residual_out written over x, y over residual
    x, res = to_dev(h["x"], dtype), to_dev(h["residual"], dtype)
    rrn.add_rmsnorm_fwd(x, res, x, w, res, rstd, wl.eps)
    torch.cuda.synchronize()
    check_out(values(x), r_ref, dtype, "residual_out==x")
    check_out(values(res), y_ref, dtype, "y==residual")
    # plain forward in place
    y_ref2, _ = oracle.rmsnorm_fwd(h["x"], h["w"], wl.eps)
    x = to_dev(h["x"], dtype)
    rrn.rmsnorm_fwd(x, w, x, None, wl.eps)
    torch.cuda.synchronize()
    check_out(values(x), y_ref2, dtype, "y==x")


# ------------------------------------------------------------------ bounds: guard bands
SENTINEL = 0x5A


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [7, 1024, 2048, 4096, 7168, 20000])
def test_outputs_stay_in_bounds(dtype, N):
    M, G = 37, 4096  # G guard bytes before and after every output
    wl = synth.Workload("guard", "add_rmsnorm_fwd", M, N, dtype, 1e-6, 41)
    h = synth.make(wl)
    es = 2 if dtype == "bf16" else 4
    t = TORCH[dtype]

    def guarded(nbytes):
        buf = torch.full((G + nbytes + G,), SENTINEL, dtype=torch.uint8, device="cuda")
        return buf, buf[G:G + nbytes]

    bufs = {}
    for name in ("ro", "y"):
        bufs[name] = guarded(M * N * es)
    bufs["rstd"] = guarded(M * 4)
    ro = bufs["ro"][1].view(t).view(M, N)
    y = bufs["y"][1].view(t).view(M, N)
    rstd = bufs["rstd"][1].view(torch.float32)
    x, res, w = to_dev(h["x"], dtype), to_dev(h["residual"], dtype), to_dev(h["w"], dtype)
    rrn.add_rmsnorm_fwd(x, res, ro, w, y, rstd, wl.eps)
    torch.cuda.synchronize()
    for name, (buf, _) in bufs.items():
        host = buf.cpu().numpy()
        assert np.all(host[:G] == SENTINEL) and np.all(host[-G:] == SENTINEL), f"{name} guard band written"
    compare_fwd(h["x"], h["residual"], h["w"], dtype, wl.eps, y, ro, rstd)
    # backward
    dxb = guarded(M * N * es)
    dwb = guarded(N * 4)
    dx = dxb[1].view(t).view(M, N)
    dw = dwb[1].view(torch.float32)
    ws_bytes = rrn.rmsnorm_bwd_workspace_bytes(M, N, t)
    wsb = guarded(max(ws_bytes, 16))
    ws = wsb[1].view(torch.float32)
    dy = to_dev(h["residual"], dtype)
    rrn.rmsnorm_bwd(dy, x, w, rstd, dx, dw, ws, wl.eps)
    torch.cuda.synchronize()
    for name, (buf, _) in {"dx": dxb, "dw": dwb, "workspace": wsb}.items():
        host = buf.cpu().numpy()
        assert np.all(host[:G] == SENTINEL) and np.all(host[-G:] == SENTINEL), f"{name} guard band written"


# ------------------------------------------------------------------ extreme values
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1024, 4096, 20000, 4095])
def test_extreme_rows(dtype, N):
    rng = np.random.default_rng(51)
    base = rng.standard_normal((8, N)).astype(np.float32)
    rows = np.stack([
        base[0] * 1e37,                                   # sum of squares overflows fp32
        base[1] * 1e-30,                                  # squares underflow fp32
        np.zeros(N, np.float32),                          # all-zero row: rstd = eps^-1/2
        np.where(rng.random(N) < 0.01, 50.0, base[3]).astype(np.float32),   # outliers
        np.full(N, 3.0, np.float32),                      # constant row
        base[5] * 1e19,                                   # squares just past fp32 range
        np.where(np.arange(N) == 0, 1e30, 1e-30).astype(np.float32),        # one huge value
        base[7],
    ]).astype(np.float32)
    x_h = bits_of(rows, dtype)
    w_h = bits_of((1.0 + 0.1 * rng.standard_normal(N)).astype(np.float32), dtype)
    for eps in (1e-6, 0.0):
        keep = np.arange(8) if eps > 0 else np.array([0, 1, 3, 4, 5, 6, 7])  # eps = 0: no zero row
        xs = x_h[keep]
        for launch in (None, rrn.Launch(rrn.VARIANT_STREAM, 0, 256, 0)):
            y, _, rstd = fwd_case(xs, None, w_h, dtype, eps, launch)
            compare_fwd(xs, None, w_h, dtype, eps, y, None, rstd)


# ------------------------------------------------------------------ backward variants
def _bwd_case(h, dtype, eps, launch=None, M=None):
    x, w, dy = to_dev(h["x"], dtype), to_dev(h["w"], dtype), to_dev(h["dy"], dtype)
    _, rstd = rrn.rms_norm(x, w, eps)
    dx = torch.full_like(x, float("nan"))
    dw = torch.full((x.shape[1],), float("nan"), device="cuda")
    # An explicit launch may pick more CTAs than the automatic plan; M * N floats always suffice.
    ws = torch.empty(max(rrn.rmsnorm_bwd_workspace_bytes(x.shape[0], x.shape[1], x.dtype),
                         4 * x.numel()) // 4, device="cuda")
    if launch is None:
        rrn.rmsnorm_bwd(dy, x, w, rstd, dx, dw, ws, eps)
    else:
        rrn.rmsnorm_bwd_ex(dy, x, w, rstd, dx, dw, ws, eps, launch)
    torch.cuda.synchronize()
    return dx, dw


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1, 7, 8, 9, 256, 1000, 1024, 2048, 4095, 4096, 7168, 8192, 16384])
def test_backward_shapes(dtype, N):
    M = 203
    wl = synth.Workload("bwd", "rmsnorm_bwd", M, N, dtype, 1e-6, 61)
    h = synth.make(wl)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(h["dy"], h["x"], h["w"], wl.eps)
    cond = bwd_cond(h["x"], h["dy"], h["w"], wl.eps)
    launches = [None, rrn.Launch(rrn.VARIANT_STREAM, 0, 128, 0), rrn.Launch(rrn.VARIANT_STREAM, 0, 512, 3)]
    V = 8 if dtype == "bf16" else 4
    if N % V == 0:
        nvec = N // V
        for vpt in (1, 2, 4):
            thr = -(-(-(-nvec // vpt)) // 32) * 32
            if thr <= (256 if vpt == 4 else 512):
                # (ctas, stages, cluster): cluster > 1 adds the dw partial sums of that many
                # CTAs in distributed shared memory; 37 -> 36 CTAs in clusters of 4, 13 -> 12
                # in clusters of 2
                launches += [rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 0),
                             rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 0, 0, 8),
                             rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 13),
                             rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 37),
                             rrn.Launch(rrn.VARIANT_ROW_CTA, vpt, thr, 37, 0, 4),
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 0, 0),
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 0, 2, 8),
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 13, 1),
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 13, 1, 2),
                             rrn.Launch(rrn.VARIANT_ROW_TMA, vpt, thr, 7, 3)]
    if N % V == 0 and N // V <= 256:
        # one row per warp: the planner's grid, 64-thread CTAs, and 5 CTAs of 4 warps walking rows
        vpt = next(v for v in (1, 2, 4, 8) if 32 * v >= N // V)
        launches += [rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 128, 0), rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 64, 0),
                     rrn.Launch(rrn.VARIANT_ROW_WARP, vpt, 128, 5)]
    if N % V == 0 and N // V >= 512:
        # each row split over a cluster (CTA q owning a column slice); 3 x C CTAs: ragged rows
        for C in (2, 4, 8):
            if -(-(N // V) // C) <= 1024:
                launches += [rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 0, 0, C),
                             rrn.Launch(rrn.VARIANT_ROW_CLUSTER, 0, 0, 3 * C, 0, C)]
    for launch in launches:
        dx, dw = _bwd_case(h, dtype, wl.eps, launch)
        check_out(values(dx), dx_ref, dtype, f"dx {launch}", cond)
        check_dw(dw.cpu().numpy().astype(np.float64), dw_ref, f"dw {launch}")


# Backward of wide rows with many rows: split over a cluster (at most 512 vectors per CTA) up to
# 4096 vectors, the two-pass kernel beyond.
@pytest.mark.parametrize("dtype,N,variant,cluster", [
    ("bf16", 16384, rrn.VARIANT_ROW_CLUSTER, 4), ("bf16", 24576, rrn.VARIANT_ROW_CLUSTER, 8),
    ("bf16", 32768, rrn.VARIANT_ROW_CLUSTER, 8), ("bf16", 40000, rrn.VARIANT_STREAM, 0),
    ("f32", 16384, rrn.VARIANT_ROW_CLUSTER, 8)])
def test_wide_rows_backward_automatic_plan(dtype, N, variant, cluster):
    M = 400
    wl = synth.Workload("wide-bwd", "rmsnorm_bwd", M, N, dtype, 1e-6, 300 + N)
    h = synth.make(wl)
    x, w, dy = to_dev(h["x"], dtype), to_dev(h["w"], dtype), to_dev(h["dy"], dtype)
    plan = rrn.plan_bwd(dy, x, w, torch.empty_like(x))
    assert plan.variant == variant and plan.cluster == cluster, plan.name
    dx_ref, dw_ref = oracle.rmsnorm_bwd(h["dy"], h["x"], h["w"], wl.eps)
    cond = bwd_cond(h["x"], h["dy"], h["w"], wl.eps)
    dx, dw = _bwd_case(h, dtype, wl.eps)
    check_out(values(dx), dx_ref, dtype, "dx", cond)
    check_dw(dw.cpu().numpy().astype(np.float64), dw_ref, "dw")


def test_short_rows_backward_plan():
    """Short rows over many rows: one row per warp up to 128 vectors (64 with the gradient at
    residual_out); beyond, the ring."""
    for N, plain, fused in ((256, rrn.VARIANT_ROW_WARP, rrn.VARIANT_ROW_WARP),
                            (512, rrn.VARIANT_ROW_WARP, rrn.VARIANT_ROW_WARP),
                            (1024, rrn.VARIANT_ROW_WARP, rrn.VARIANT_ROW_TMA),
                            (2048, rrn.VARIANT_ROW_TMA, rrn.VARIANT_ROW_TMA)):
        x = torch.empty(65536, N, device="cuda", dtype=torch.bfloat16)
        w = torch.empty(N, device="cuda", dtype=torch.bfloat16)
        for g, variant in ((None, plain), (x, fused)):
            p = rrn.plan_bwd(x, x, w, x, g)
            assert p.variant == variant, (N, g is not None, p)
            if variant == rrn.VARIANT_ROW_WARP:
                assert p.vpt * 32 >= N // 8 and p.threads == 128, p
    # and the full-size workload through the automatic plan matches the oracle
    M, N = 16384, 512
    wl = synth.Workload("bwd-short", "rmsnorm_bwd", M, N, "bf16", 1e-6, 62)
    h = synth.make(wl)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(h["dy"], h["x"], h["w"], wl.eps)
    dx, dw = _bwd_case(h, "bf16", wl.eps)
    check_out(values(dx), dx_ref, "bf16", "dx", bwd_cond(h["x"], h["dy"], h["w"], wl.eps))
    check_dw(dw.cpu().numpy().astype(np.float64), dw_ref, "dw")


def test_backward_is_deterministic():
    wl = synth.get("rmsnorm_bwd_16384x4096_bf16").with_shape(4096)
    h = synth.make(wl)
    a_dx, a_dw = _bwd_case(h, "bf16", wl.eps)
    b_dx, b_dw = _bwd_case(h, "bf16", wl.eps)
    assert torch.equal(a_dx.view(torch.int16), b_dx.view(torch.int16))
    assert torch.equal(a_dw.view(torch.int32), b_dw.view(torch.int32))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N,launch", [(4096, None), (512, rrn.Launch(rrn.VARIANT_ROW_WARP, 0, 128, 0))],
                         ids=["auto", "row-per-warp"])
def test_backward_in_place(dtype, N, launch):
    M = 50
    wl = synth.Workload("bwd-alias", "rmsnorm_bwd", M, N, dtype, 1e-6, 71)
    h = synth.make(wl)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(h["dy"], h["x"], h["w"], wl.eps)
    cond = bwd_cond(h["x"], h["dy"], h["w"], wl.eps)
    x, w, dy = to_dev(h["x"], dtype), to_dev(h["w"], dtype), to_dev(h["dy"], dtype)
    _, rstd = rrn.rms_norm(x, w, wl.eps)
    dw = torch.empty(N, device="cuda")
    ws = torch.empty(max(rrn.rmsnorm_bwd_workspace_bytes(M, N, x.dtype), 4 * M * N) // 4, device="cuda")
    rrn.rmsnorm_bwd_ex(dy, x, w, rstd, dy, dw, ws, wl.eps, launch)      # dx over dy
    torch.cuda.synchronize()
    check_out(values(dy), dx_ref, dtype, "dx==dy", cond)
    rrn.rmsnorm_bwd_ex(to_dev(h["dy"], dtype), x, w, rstd, x, dw, ws, wl.eps, launch)  # dx over x
    torch.cuda.synchronize()
    check_out(values(x), dx_ref, dtype, "dx==x", cond)
    check_dw(dw.cpu().numpy().astype(np.float64), dw_ref)


def test_backward_workspace_too_small_is_rejected():
    x = torch.zeros(64, 4096, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(64, device="cuda")
    dw = torch.empty(4096, device="cuda")
    # the query covers the plain and the fused backward; this call (plain) needs one row of N
    # floats per stage-1 CTA (clusters: per cluster) and no more
    plan = rrn.plan_bwd(x, x, w, x)
    rows = plan.ctas // plan.cluster if plan.cluster > 1 else plan.ctas
    need = rows * 4096 * 4
    assert rrn.rmsnorm_bwd_workspace_bytes(64, 4096, torch.bfloat16) >= need
    ws = torch.empty(need // 4 - 1, device="cuda")
    with pytest.raises(rrn.RRNError) as e:
        rrn.rmsnorm_bwd(x, x, w, rstd, x, dw, ws, 1e-6)
    assert e.value.status == 6
    ws = torch.empty(need // 4, device="cuda")
    rrn.rmsnorm_bwd(x, x, w, rstd, x, dw, ws, 1e-6)
    torch.cuda.synchronize()


def test_bad_launch_configuration_is_rejected():
    x = torch.zeros(8, 4096, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rrn.RRNError) as e:   # 64 threads x 1 vector cannot cover 512 vectors
        rrn.add_rmsnorm_fwd_ex(x, None, None, w, x, None, 1e-6, rrn.Launch(rrn.VARIANT_ROW_CTA, 1, 64, 0))
    assert e.value.status == 8


# ------------------------------------------------------------------ streams and graphs
def test_side_stream_and_graph_capture():
    wl = synth.get("add_rmsnorm_fwd_4096x4096_bf16").with_shape(1024)
    h = synth.make(wl)
    x, res, w = to_dev(h["x"], "bf16"), to_dev(h["residual"], "bf16"), to_dev(h["w"], "bf16")
    y = torch.empty_like(x)
    ro = torch.empty_like(x)
    rstd = torch.empty(x.shape[0], device="cuda")
    dx = torch.empty_like(x)
    dw = torch.empty(x.shape[1], device="cuda")
    ws = torch.empty(rrn.rmsnorm_bwd_workspace_bytes(*x.shape, x.dtype) // 4, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rrn.add_rmsnorm_fwd(x, res, ro, w, y, rstd, wl.eps)           # current stream = s
        rrn.rmsnorm_bwd(y, ro, w, rstd, dx, dw, ws, wl.eps, stream=s)
    s.synchronize()
    ref = [t.clone() for t in (y, ro, rstd, dx, dw)]
    for t in (y, ro, rstd, dx, dw):
        t.fill_(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):   # the library neither allocates nor synchronises: capturable
        rrn.add_rmsnorm_fwd(x, res, ro, w, y, rstd, wl.eps)
        rrn.rmsnorm_bwd(y, ro, w, rstd, dx, dw, ws, wl.eps)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, (y, ro, rstd, dx, dw)):
        assert torch.equal(a, b)
    compare_fwd(h["x"], h["residual"], h["w"], "bf16", wl.eps, y, ro, rstd)


# ------------------------------------------------------------------ bounded waits
def test_bounded_wait_reports_and_context_survives():
    """No kernel above gave up on a wait; a wait made to run out on purpose sets the fault bit
    and returns, and the context keeps working."""
    assert rrn.device_faults(clear=True) == 0, "a kernel reported a timed-out wait"
    rrn.selftest_wait_timeout(50_000_000)
    torch.cuda.synchronize()
    assert rrn.device_faults(clear=True) & 1
    assert rrn.device_faults(clear=False) == 0
    wl = synth.get("rmsnorm_fwd_256x1024_bf16")
    h = synth.make(wl)
    y, _, rstd = fwd_case(h["x"], None, h["w"], "bf16", wl.eps)
    compare_fwd(h["x"], None, h["w"], "bf16", wl.eps, y, None, rstd)
