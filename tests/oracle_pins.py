"""Pins for the CPU oracle: facts fixed by the mathematics, checked without the oracle's code.

Each pin is a function ``pin_*(o)`` taking an ``oracle.Oracle`` handle and raising
``AssertionError`` when the oracle disagrees. ``test_oracle_pins.py`` runs every pin on the
real oracle, and also compiles copies of ``oracle.c`` with planted mistakes (a dropped term, a
wrong sign, a transposed or wrong index) to show that at least one pin rejects each of them.

The expected values come from: the hand-worked examples in ``golden/worked_examples.json``;
closed forms (constant row, zero row, unit-RMS row, exact power-of-two scale invariance);
the exact identity fused == RMSNorm(x + residual); central finite differences of the scalar
L = <dy, y>; the identity <dx, x> = eps * rstd^2 * <g, xhat> per row; a pure-Python brute
force of dw on tiny inputs; torch's own ``rms_norm`` and autograd in float64 (an independent
library routine); and torch's bf16 -> float cast for the bit decoding.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")


def _close(a, b, rtol, atol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    bad = ~(np.abs(a - b) <= atol + rtol * np.abs(b))
    assert not bad.any(), (f"{what}: {int(bad.sum())} mismatches, first at "
                           f"{np.argwhere(bad)[0].tolist()}: got {a[bad][0]!r}, want {b[bad][0]!r}")


def _bf16_bits(values) -> np.ndarray:
    """bf16 bit patterns of values that are exactly representable in bf16."""
    f = np.asarray(values, dtype=np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, f), "test input is not exactly representable in bf16"
    return bits


# --------------------------------------------------------------------------- decoding
def pin_decode_known_bits(o):
    """bf16 bit patterns with values known from the IEEE-754 binary32 layout."""
    bits = np.array([0x3F80, 0xC040, 0x4049, 0x0000, 0x8000, 0x7F7F, 0x0080, 0x0001, 0x3E80],
                    dtype=np.uint16)
    want = [1.0, -3.0, 3.140625, 0.0, -0.0, (2.0 - 2.0 ** -7) * 2.0 ** 127, 2.0 ** -126,
            2.0 ** -133, 0.25]
    got = o.decode(bits)
    assert got.tolist() == want, f"decode: {got.tolist()} != {want}"
    assert math.copysign(1.0, got[4]) == -1.0, "decode lost the sign of -0"


def pin_decode_matches_torch_cast(o):
    """Every finite bf16 pattern decodes to torch's own bf16 -> float64 value."""
    import torch

    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]  # drop inf/NaN
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = o.decode(bits)
    assert np.array_equal(got, want), "decode differs from torch's bf16 cast"
    f32 = np.array([1.5, -2.0 ** -149, 3.4e38, 0.1], dtype=np.float32)
    assert np.array_equal(o.decode(f32), f32.astype(np.float64)), "fp32 decode is not exact"


# --------------------------------------------------------------------------- forward
def pin_golden_worked_examples(o):
    """The hand-worked cases of ``golden/worked_examples.json``, in fp64 and as bf16 bits."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        for enc in ("f64", "bf16"):
            conv = (lambda v: np.asarray(v, dtype=np.float64)) if enc == "f64" else _bf16_bits
            x = conv(c["x"]) if "x" in c else None
            w = conv(c["w"])
            tag = f"{c['name']} ({enc})"
            if c["op"] == "rmsnorm_fwd":
                y, rstd = o.rmsnorm_fwd(x, w, c["eps"])
                _close(y, c["y"], 1e-14, 1e-15, tag + " y")
                _close(rstd, c["rstd"], 1e-14, 0.0, tag + " rstd")
            elif c["op"] == "add_rmsnorm_fwd":
                r, y, rstd = o.add_rmsnorm_fwd(x, conv(c["residual"]), w, c["eps"])
                _close(r, c["residual_out"], 0.0, 0.0, tag + " residual_out")
                _close(y, c["y"], 1e-14, 1e-15, tag + " y")
                _close(rstd, c["rstd"], 1e-14, 0.0, tag + " rstd")
            elif c["op"] == "rmsnorm_bwd":
                dx, dw = o.rmsnorm_bwd(conv(c["dy"]), x, w, c["eps"])
                _close(dx, c["dx"], 1e-13, 1e-15, tag + " dx")
                _close(dw, c["dw"], 1e-13, 1e-15, tag + " dw")
            elif c["op"] == "layernorm_fwd":
                _, y, mean, rstd = o.add_layernorm_fwd(x, None, w, conv(c["b"]), c["eps"])
                _close(y, c["y"], 1e-14, 1e-15, tag + " y")
                _close(mean, c["mean"], 1e-15, 0.0, tag + " mean")
                _close(rstd, c["rstd"], 1e-14, 0.0, tag + " rstd")
            elif c["op"] == "layernorm_bwd":
                dx, dw, db = o.add_layernorm_bwd(conv(c["dy"]), None, x, w, c["eps"])
                _close(dx, c["dx"], 1e-13, 1e-15, tag + " dx")
                _close(dw, c["dw"], 1e-13, 1e-15, tag + " dw")
                _close(db, c["db"], 1e-13, 1e-15, tag + " db")
            elif c["op"] == "add_rmsnorm_bwd":
                r = conv(c["residual_out"])
                d_r, dw = o.add_rmsnorm_bwd(conv(c["dy"]), conv(c["d_residual_out"]), r, w, c["eps"])
                _close(d_r, c["d_r"], 1e-13, 1e-15, tag + " d_r")
                _close(dw, c["dw"], 1e-13, 1e-15, tag + " dw")
            else:
                raise AssertionError(f"unknown op {c['op']}")


def pin_constant_row(o):
    """A constant row c gives rstd = 1/sqrt(c^2 + eps) and y = w * c * rstd."""
    rng = np.random.default_rng(11)
    N = 37
    for c in (-3.5, 0.125, 7.0):
        for eps in (1e-6, 0.5):
            x = np.full((2, N), c)
            w = rng.standard_normal(N)
            y, rstd = o.rmsnorm_fwd(x, w, eps)
            want_rstd = 1.0 / math.sqrt(c * c + eps)
            _close(rstd, [want_rstd] * 2, 1e-15, 0.0, "constant-row rstd")
            _close(y, np.tile(w * c * want_rstd, (2, 1)), 1e-14, 0.0, "constant-row y")


def pin_zero_row(o):
    """An all-zero row gives rstd = eps^-1/2 and y = 0."""
    N = 19
    for eps in (1e-6, 1e-5, 2.0):
        y, rstd = o.rmsnorm_fwd(np.zeros((3, N)), np.linspace(-2, 2, N), eps)
        _close(rstd, [eps ** -0.5] * 3, 1e-15, 0.0, "zero-row rstd")
        assert np.all(y == 0.0), "zero-row y is not zero"


def pin_unit_rms_row(o):
    """A row of +/-1 entries with w = 1 comes back as x / sqrt(1 + eps)."""
    rng = np.random.default_rng(12)
    N = 64
    x = np.where(rng.random((4, N)) < 0.5, -1.0, 1.0)
    for eps in (0.0, 1e-6):
        y, rstd = o.rmsnorm_fwd(x, np.ones(N), eps)
        _close(y, x / math.sqrt(1.0 + eps), 1e-15, 0.0, "unit-RMS y")
        _close(rstd, [1.0 / math.sqrt(1.0 + eps)] * 4, 1e-15, 0.0, "unit-RMS rstd")


def pin_scale_invariance(o):
    """With eps = 0, y(2^k x) == y(x) bit for bit and rstd scales by 2^-k; with a tiny eps,
    y(a x) ~= y(x) for any a > 0."""
    rng = np.random.default_rng(13)
    M, N = 5, 23
    x = rng.standard_normal((M, N))
    w = 1.0 + 0.1 * rng.standard_normal(N)
    y0, r0 = o.rmsnorm_fwd(x, w, 0.0)
    for k in (-3, 1, 5):
        yk, rk = o.rmsnorm_fwd(x * 2.0 ** k, w, 0.0)
        assert np.array_equal(yk, y0), "y(2^k x) != y(x) with eps = 0"
        assert np.array_equal(rk * 2.0 ** k, r0), "rstd(2^k x) != 2^-k rstd(x)"
    for a in (0.37, 3.7, 123.0):
        ya, _ = o.rmsnorm_fwd(x * a, w, 1e-12)
        _close(ya, y0, 1e-9, 1e-12, f"y({a} x) vs y(x)")


def pin_non_uniform_weights_follow_columns(o):
    """Column j is scaled by w_j: y / w is the same for any positive w."""
    rng = np.random.default_rng(14)
    x = rng.standard_normal((3, 11))
    w = np.arange(1, 12, dtype=np.float64)
    y1, _ = o.rmsnorm_fwd(x, np.ones(11), 1e-6)
    yw, _ = o.rmsnorm_fwd(x, w, 1e-6)
    _close(yw, y1 * w[None, :], 1e-15, 0.0, "y with weights vs unweighted y * w")


def pin_fused_is_rmsnorm_of_sum(o):
    """Fused Add + RMSNorm equals RMSNorm of x + residual; residual_out is the exact sum."""
    rng = np.random.default_rng(15)
    M, N = 6, 40
    xf = rng.standard_normal((M, N)).astype(np.float32)
    rf = (2.0 * rng.standard_normal((M, N))).astype(np.float32)
    w = (1.0 + 0.1 * rng.standard_normal(N)).astype(np.float32)
    r, y, rstd = o.add_rmsnorm_fwd(xf, rf, w, 1e-6)
    s = xf.astype(np.float64) + rf.astype(np.float64)
    assert np.array_equal(r, s), "residual_out is not x + residual"
    y2, rstd2 = o.rmsnorm_fwd(s, w, 1e-6)
    assert np.array_equal(y, y2) and np.array_equal(rstd, rstd2), "fused != rmsnorm(x + residual)"
    # and the plain op is the fused op with a zero residual
    y3, _ = o.rmsnorm_fwd(xf, w, 1e-6)
    _, y4, _ = o.add_rmsnorm_fwd(xf, np.zeros_like(xf), w, 1e-6)
    assert np.array_equal(y3, y4), "rmsnorm(x) != fused(x, 0)"


def pin_matches_torch_rms_norm(o):
    """torch.nn.functional.rms_norm in float64 on the CPU (an independent library routine)."""
    import torch

    rng = np.random.default_rng(16)
    for (M, N, eps) in ((7, 1, 1e-6), (9, 33, 1e-6), (4, 1000, 1e-5), (3, 4096, 0.1)):
        x = rng.standard_normal((M, N)) * 3.0
        w = 1.0 + 0.1 * rng.standard_normal(N)
        y, rstd = o.rmsnorm_fwd(x, w, eps)
        ty = torch.nn.functional.rms_norm(torch.from_numpy(x), (N,), torch.from_numpy(w), eps)
        _close(y, ty.numpy(), 1e-13, 1e-15, f"torch rms_norm {M}x{N}")
        tr = torch.rsqrt(torch.from_numpy(x).pow(2).mean(-1) + eps).numpy()
        _close(rstd, tr, 1e-13, 0.0, f"torch rstd {M}x{N}")


# --------------------------------------------------------------------------- backward
def _loss(o, x, w, dy, eps):
    y, _ = o.rmsnorm_fwd(x, w, eps)
    return float(np.sum(dy * y))


def pin_bwd_finite_differences(o):
    """Central differences of L = <dy, y> in fp64 match the analytic dx and dw."""
    rng = np.random.default_rng(17)
    h = 1e-6
    for (M, N, eps) in ((1, 1, 1e-6), (2, 5, 1e-6), (3, 7, 0.3)):
        x = rng.standard_normal((M, N))
        w = 1.0 + 0.3 * rng.standard_normal(N)
        dy = rng.standard_normal((M, N))
        dx, dw = o.rmsnorm_bwd(dy, x, w, eps)
        fdx = np.empty_like(x)
        for i in range(M):
            for j in range(N):
                xp, xm = x.copy(), x.copy()
                xp[i, j] += h
                xm[i, j] -= h
                fdx[i, j] = (_loss(o, xp, w, dy, eps) - _loss(o, xm, w, dy, eps)) / (2 * h)
        fdw = np.empty_like(w)
        for j in range(N):
            wp, wm = w.copy(), w.copy()
            wp[j] += h
            wm[j] -= h
            fdw[j] = (_loss(o, x, wp, dy, eps) - _loss(o, x, wm, dy, eps)) / (2 * h)
        _close(dx, fdx, 1e-6, 1e-7, f"dx vs finite differences {M}x{N}")
        _close(dw, fdw, 1e-6, 1e-7, f"dw vs finite differences {M}x{N}")


def pin_bwd_orthogonality(o):
    """Per row, <dx, x> = eps * rstd^2 * <g, xhat> (g = dy w, xhat = x rstd); 0 when eps = 0."""
    rng = np.random.default_rng(18)
    M, N = 4, 50
    x = rng.standard_normal((M, N))
    w = 1.0 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    for eps in (0.0, 0.25):
        dx, _ = o.rmsnorm_bwd(dy, x, w, eps)
        for i in range(M):
            ms = float(np.mean(x[i] ** 2))
            rstd = 1.0 / math.sqrt(ms + eps)
            g_xhat = float(np.dot(dy[i] * w, x[i] * rstd))
            lhs = float(np.dot(dx[i], x[i]))
            rhs = eps * rstd * rstd * g_xhat
            assert abs(lhs - rhs) <= 1e-12 * (1.0 + abs(g_xhat)), f"<dx,x> row {i}: {lhs} vs {rhs}"


def pin_bwd_dw_brute_force(o):
    """dw summed over rows by pure-Python loops, from the definition, on a tiny input."""
    rng = np.random.default_rng(19)
    M, N, eps = 3, 4, 1e-3
    x = rng.standard_normal((M, N))
    w = 1.0 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    want = [0.0] * N
    for i in range(M):
        ss = 0.0
        for j in range(N):
            ss += float(x[i, j]) ** 2
        rs = (ss / N + eps) ** -0.5
        for j in range(N):
            want[j] += float(dy[i, j]) * float(x[i, j]) * rs
    _, dw = o.rmsnorm_bwd(dy, x, w, eps)
    _close(dw, want, 1e-14, 1e-15, "dw brute force")


def pin_bwd_matches_torch_autograd(o):
    """torch autograd through rms_norm in float64 on the CPU gives the same dx and dw."""
    import torch

    rng = np.random.default_rng(20)
    for (M, N, eps) in ((5, 8, 1e-6), (3, 129, 1e-5), (2, 2048, 0.5)):
        x = rng.standard_normal((M, N))
        w = 1.0 + 0.1 * rng.standard_normal(N)
        dy = rng.standard_normal((M, N))
        tx = torch.from_numpy(x).requires_grad_(True)
        tw = torch.from_numpy(w).requires_grad_(True)
        ty = torch.nn.functional.rms_norm(tx, (N,), tw, eps)
        ty.backward(torch.from_numpy(dy))
        dx, dw = o.rmsnorm_bwd(dy, x, w, eps)
        _close(dx, tx.grad.numpy(), 1e-12, 1e-14, f"torch dx {M}x{N}")
        _close(dw, tw.grad.numpy(), 1e-12, 1e-13, f"torch dw {M}x{N}")


def pin_add_bwd_finite_differences(o):
    """Central differences of L = <dy, y> + <d_ro, r> (r = x + residual) with respect to x and
    to residual both give the fused backward's d_r; with respect to w, its dw."""
    rng = np.random.default_rng(21)
    h = 1e-6
    M, N, eps = 2, 6, 1e-3
    x = rng.standard_normal((M, N))
    res = rng.standard_normal((M, N))
    w = 1.0 + 0.3 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    dro = rng.standard_normal((M, N))

    def loss(xx, rr, ww):
        r, y, _ = o.add_rmsnorm_fwd(xx, rr, ww, eps)
        return float(np.sum(dy * y) + np.sum(dro * r))

    d_r, dw = o.add_rmsnorm_bwd(dy, dro, x + res, w, eps)
    for which in ("x", "residual"):
        fd = np.empty_like(x)
        for i in range(M):
            for j in range(N):
                a, b = (x.copy(), res.copy()), (x.copy(), res.copy())
                k = 0 if which == "x" else 1
                a[k][i, j] += h
                b[k][i, j] -= h
                fd[i, j] = (loss(a[0], a[1], w) - loss(b[0], b[1], w)) / (2 * h)
        _close(d_r, fd, 1e-6, 1e-7, f"d_r vs finite differences in {which}")
    fdw = np.empty_like(w)
    for j in range(N):
        wp, wm = w.copy(), w.copy()
        wp[j] += h
        wm[j] -= h
        fdw[j] = (loss(x, res, wp) - loss(x, res, wm)) / (2 * h)
    _close(dw, fdw, 1e-6, 1e-7, "fused dw vs finite differences")


def pin_add_bwd_matches_torch_autograd(o):
    """torch autograd in float64 through r = x + residual, y = rms_norm(r) * w, returning both."""
    import torch

    rng = np.random.default_rng(22)
    M, N, eps = 4, 96, 1e-5
    x = rng.standard_normal((M, N))
    res = rng.standard_normal((M, N))
    w = 1.0 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    dro = rng.standard_normal((M, N))
    tx = torch.from_numpy(x).requires_grad_(True)
    tr = torch.from_numpy(res).requires_grad_(True)
    tw = torch.from_numpy(w).requires_grad_(True)
    r = tx + tr
    y = torch.nn.functional.rms_norm(r, (N,), tw, eps)
    (torch.sum(y * torch.from_numpy(dy)) + torch.sum(r * torch.from_numpy(dro))).backward()
    d_r, dw = o.add_rmsnorm_bwd(dy, dro, x + res, w, eps)
    _close(d_r, tx.grad.numpy(), 1e-12, 1e-14, "torch d(x)")
    _close(d_r, tr.grad.numpy(), 1e-12, 1e-14, "torch d(residual)")
    _close(dw, tw.grad.numpy(), 1e-12, 1e-13, "torch fused dw")
    # with no gradient at residual_out it is the plain backward
    d0, dw0 = o.add_rmsnorm_bwd(dy, None, x + res, w, eps)
    p0, pw0 = o.rmsnorm_bwd(dy, x + res, w, eps)
    assert np.array_equal(d0, p0) and np.array_equal(dw0, pw0), "fused bwd without d_ro != plain bwd"


# --------------------------------------------------------------------------- LayerNorm
def pin_layernorm_matches_torch(o):
    """torch.nn.functional.layer_norm (forward and autograd) in float64, fused through
    r = x + residual, with weight and bias."""
    import torch

    rng = np.random.default_rng(31)
    for (M, N, eps) in ((3, 1, 1e-5), (4, 77, 1e-5), (2, 2048, 0.3)):
        x = rng.standard_normal((M, N)) * 2.0 + 0.7
        res = rng.standard_normal((M, N))
        w = 1.0 + 0.1 * rng.standard_normal(N)
        b = 0.1 * rng.standard_normal(N)
        dy = rng.standard_normal((M, N))
        dro = rng.standard_normal((M, N))
        tx = torch.from_numpy(x).requires_grad_(True)
        tr = torch.from_numpy(res).requires_grad_(True)
        tw = torch.from_numpy(w).requires_grad_(True)
        tb = torch.from_numpy(b).requires_grad_(True)
        r = tx + tr
        ty = torch.nn.functional.layer_norm(r, (N,), tw, tb, eps)
        (torch.sum(ty * torch.from_numpy(dy)) + torch.sum(r * torch.from_numpy(dro))).backward()
        ro, y, mean, rstd = o.add_layernorm_fwd(x, res, w, b, eps)
        _close(y, ty.detach().numpy(), 1e-12, 1e-14, f"torch layer_norm {M}x{N}")
        _close(mean, (x + res).mean(-1), 1e-13, 1e-14, "mean")
        dx, dw, db = o.add_layernorm_bwd(dy, dro, x + res, w, eps)
        _close(dx, tx.grad.numpy(), 1e-11, 1e-13, f"torch LN d(x) {M}x{N}")
        _close(dx, tr.grad.numpy(), 1e-11, 1e-13, f"torch LN d(residual) {M}x{N}")
        _close(dw, tw.grad.numpy(), 1e-11, 1e-12, f"torch LN dw {M}x{N}")
        _close(db, tb.grad.numpy(), 1e-11, 1e-12, f"torch LN db {M}x{N}")


def pin_layernorm_finite_differences(o):
    """Central differences of L = <dy, y> + <d_ro, r> give dx, dw and db."""
    rng = np.random.default_rng(32)
    h = 1e-6
    M, N, eps = 2, 5, 1e-2
    x = rng.standard_normal((M, N))
    w = 1.0 + 0.3 * rng.standard_normal(N)
    b = rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    dro = rng.standard_normal((M, N))

    def loss(xx, ww, bb):
        r, y, _, _ = o.add_layernorm_fwd(xx, None, ww, bb, eps)
        return float(np.sum(dy * y) + np.sum(dro * r))

    dx, dw, db = o.add_layernorm_bwd(dy, dro, x, w, eps)
    fdx = np.empty_like(x)
    for i in range(M):
        for j in range(N):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fdx[i, j] = (loss(xp, w, b) - loss(xm, w, b)) / (2 * h)
    fdw, fdb = np.empty(N), np.empty(N)
    for j in range(N):
        wp, wm, bp, bm = w.copy(), w.copy(), b.copy(), b.copy()
        wp[j] += h
        wm[j] -= h
        bp[j] += h
        bm[j] -= h
        fdw[j] = (loss(x, wp, b) - loss(x, wm, b)) / (2 * h)
        fdb[j] = (loss(x, w, bp) - loss(x, w, bm)) / (2 * h)
    _close(dx, fdx, 1e-6, 1e-7, "LN dx vs finite differences")
    _close(dw, fdw, 1e-6, 1e-7, "LN dw vs finite differences")
    _close(db, fdb, 1e-6, 1e-7, "LN db vs finite differences")


def pin_layernorm_identities(o):
    """Per row: sum_j dx_j = 0 and <dx, x - mean> = eps * rstd^2 * <g, xhat> (no d_ro);
    y(x + c) = y(x) for a constant shift c; with zero-mean rows and no bias LayerNorm equals
    RMSNorm."""
    rng = np.random.default_rng(33)
    M, N = 4, 40
    x = rng.standard_normal((M, N))
    w = 1.0 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    for eps in (0.0, 0.5):
        dx, _, _ = o.add_layernorm_bwd(dy, None, x, w, eps)
        for i in range(M):
            mu = float(np.mean(x[i]))
            s = 1.0 / math.sqrt(float(np.mean((x[i] - mu) ** 2)) + eps)
            g_xhat = float(np.dot(dy[i] * w, (x[i] - mu) * s))
            assert abs(float(np.sum(dx[i]))) <= 1e-12 * (1 + np.abs(dx[i]).sum()), "sum dx != 0"
            lhs = float(np.dot(dx[i], x[i] - mu))
            assert abs(lhs - eps * s * s * g_xhat) <= 1e-12 * (1 + abs(g_xhat)), "<dx, x - mean>"
    _, y0, _, _ = o.add_layernorm_fwd(x, None, w, None, 1e-5)
    _, y1, _, _ = o.add_layernorm_fwd(x + 3.0, None, w, None, 1e-5)
    _close(y1, y0, 1e-12, 1e-13, "shift invariance")
    xz = x - x.mean(axis=1, keepdims=True)
    _, yl, _, _ = o.add_layernorm_fwd(xz, None, w, None, 1e-5)
    yr, _ = o.rmsnorm_fwd(xz - xz.mean(axis=1, keepdims=True), w, 1e-5)
    _close(yl, yr, 1e-12, 1e-14, "zero-mean LayerNorm vs RMSNorm")


# --------------------------------------------------------------------------- fp8 e4m3
def _e4m3_values():
    import torch

    codes = np.arange(0, 0x7F, dtype=np.uint8)  # non-negative finite codes, ascending values
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_e4m3_codec_matches_torch(o):
    """Decoding of all 256 codes, and encoding (round to nearest, ties to even) of every
    representable value, every midpoint between neighbours and the fp32 values just beside each
    midpoint, agree with torch's float8_e4m3fn cast; finite values beyond 448 saturate."""
    import torch

    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([o.e4m3_decode(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(want)), "e4m3 NaN codes"
    assert np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)]), "e4m3 decode"
    vals = _e4m3_values()
    mids = (vals[:-1] + vals[1:]) / 2
    probe = np.concatenate([vals, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                            np.nextafter(mids.astype(np.float32), np.float32(1e9))]).astype(np.float32)
    probe = np.concatenate([probe, -probe])
    ref = torch.from_numpy(probe).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([o.e4m3_encode(float(v)) for v in probe], dtype=np.uint8)
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, f"e4m3 encode of {probe[bad[0]]!r}: {mine[bad[0]]:#x} vs torch {ref[bad[0]]:#x}"
    for v, c in ((448.0, 0x7E), (449.0, 0x7E), (1e30, 0x7E), (-1000.0, 0xFE), (0.0, 0x00)):
        assert o.e4m3_encode(v) == c, f"e4m3 saturation of {v}"


def pin_rmsnorm_quant_fp8(o):
    """The fused quantiser: r and rstd as the RMSNorm oracle; scale = max|y| / 448 with y from
    the RMSNorm oracle; the largest element lands exactly on +/-448; every code is the nearest
    e4m3 value to y / scale (dequantisation error at most half a code step); an all-zero row gives
    scale 0 and zero codes."""
    rng = np.random.default_rng(41)
    M, N, eps = 5, 96, 1e-6
    x = rng.standard_normal((M, N))
    res = 2.0 * rng.standard_normal((M, N))
    x[4] = -res[4]                                  # an all-zero r row
    w = 1.0 + 0.1 * rng.standard_normal(N)
    r, v, q, scale, rstd = o.rmsnorm_quant_fp8(x, res, w, eps)
    r2, y, rstd2 = o.add_rmsnorm_fwd(x, res, w, eps)
    assert np.array_equal(r, r2) and np.array_equal(rstd, rstd2), "quant: r / rstd differ"
    amax = np.max(np.abs(y), axis=1)
    _close(scale, amax / 448.0, 1e-15, 0.0, "quant scale")
    vals = _e4m3_values()
    for i in range(4):
        j = int(np.argmax(np.abs(y[i])))
        assert q[i, j] in (0x7E, 0xFE), "argmax element not at +/-448"
        deq = np.array([o.e4m3_decode(int(c)) for c in q[i]]) * scale[i]
        a = np.abs(y[i]) / scale[i]
        k = np.clip(np.searchsorted(vals, a), 1, len(vals) - 1)
        half = (vals[k] - vals[k - 1]) / 2 * scale[i]
        assert np.all(np.abs(deq - y[i]) <= half * (1 + 1e-12)), "dequantisation error above half a step"
        _close(v[i], y[i] / scale[i], 1e-15, 0.0, "quant v")
    assert scale[4] == 0.0 and np.all(q[4] == 0), "zero row"


ALL_PINS = [
    pin_decode_known_bits,
    pin_decode_matches_torch_cast,
    pin_golden_worked_examples,
    pin_constant_row,
    pin_zero_row,
    pin_unit_rms_row,
    pin_scale_invariance,
    pin_non_uniform_weights_follow_columns,
    pin_fused_is_rmsnorm_of_sum,
    pin_matches_torch_rms_norm,
    pin_bwd_finite_differences,
    pin_bwd_orthogonality,
    pin_bwd_dw_brute_force,
    pin_bwd_matches_torch_autograd,
    pin_add_bwd_finite_differences,
    pin_add_bwd_matches_torch_autograd,
    pin_layernorm_matches_torch,
    pin_layernorm_finite_differences,
    pin_layernorm_identities,
    pin_e4m3_codec_matches_torch,
    pin_rmsnorm_quant_fp8,
]
