"""The seeded input generator: determinism, shapes, encodings and distributions (CPU only)."""
import numpy as np

import synth


def test_every_workload_draws_its_tensors():
    for name, w in synth.WORKLOADS.items():
        small = w.with_shape(min(w.M, 64))
        t = synth.make(small)
        want = {"x", "w"} | ({"residual"} if w.op in ("add_rmsnorm_fwd", "add_layernorm_fwd",
                                                       "add_rmsnorm_fp8") else set()) | (
            {"dy"} if w.op in ("rmsnorm_bwd", "add_rmsnorm_bwd", "layernorm_bwd") else set()) | (
            {"d_ro"} if w.op == "add_rmsnorm_bwd" or (w.op == "layernorm_bwd" and w.residual_grad)
            else set()) | (
            {"b"} if "layernorm" in w.op else set())
        assert want <= set(t), name
        enc = np.uint16 if w.dtype == synth.BF16 else np.float32
        for k in want:
            assert t[k].dtype == enc, (name, k)
        assert t["x"].shape == (small.M, w.N) and t["w"].shape == (w.N,)


def test_deterministic_per_seed():
    w = synth.get("add_rmsnorm_fwd_4096x4096_bf16").with_shape(16)
    a, b = synth.make(w), synth.make(w)
    for k in ("x", "residual", "w"):
        assert np.array_equal(a[k], b[k])


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.0 - 2.0 ** -7 + 2.0 ** -9, 3.0],
                    dtype=np.float32)
    bits = synth.to_bf16_bits(vals)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert back.tolist() == [1.0, 1.015625, -2.0, 3.0]


def test_outlier_workload_statistics():
    w = synth.get("add_rmsnorm_fwd_16384x7168_bf16").with_shape(256)
    t = synth.make(w)
    res = (t["residual"].astype(np.uint32) << 16).view(np.float32)
    frac = float(np.mean(np.abs(res) == 50.0))
    assert 0.008 < frac < 0.012
    assert int(t["outliers"]) == int(np.sum(np.abs(res) == 50.0))
    body = res[np.abs(res) != 50.0]
    assert 1.9 < float(body.std()) < 2.1  # N(0, 4): sigma 2
    wt = (t["w"].astype(np.uint32) << 16).view(np.float32)
    assert wt.min() >= 0.5 and wt.max() <= 1.5


def test_min_bytes_matches_tensor_sizes():
    assert synth.min_bytes(synth.get("rmsnorm_fwd_256x1024_bf16")) == 1_051_648
    assert synth.min_bytes(synth.get("add_rmsnorm_fwd_4096x4096_bf16")) == 134_242_304
    assert synth.min_bytes(synth.get("add_rmsnorm_fwd_16384x4096_bf16")) == 536_944_640
    assert synth.min_bytes(synth.get("add_rmsnorm_fwd_16384x7168_bf16")) == 939_603_968
    assert synth.min_bytes(synth.get("rmsnorm_bwd_16384x4096_bf16")) == 402_743_296
    # LayerNorm backward: x, dy (, d_residual_out), dx + w + mean, rstd + dw, db
    assert synth.min_bytes(synth.get("layernorm_bwd_plain_16384x4096_bf16")) == \
        3 * 16384 * 4096 * 2 + 4096 * 2 + 8 * 16384 + 8 * 4096
    assert "d_ro" not in synth.make(synth.get("layernorm_bwd_plain_16384x4096_bf16").with_shape(4))
    assert synth.min_bytes(synth.get("rmsnorm_fwd_65536x2048_f32")) == 1_074_012_160
    # 16384 x 4096: x, residual, residual_out (bf16) + codes (1 byte) + w + scale
    assert synth.min_bytes(synth.get("add_rmsnorm_fp8_16384x4096_bf16")) == \
        3 * 16384 * 4096 * 2 + 16384 * 4096 + 4096 * 2 + 4 * 16384
