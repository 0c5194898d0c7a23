"""Helpers for the GPU parity tests: host <-> device transfer of raw encodings, and the
acceptance bounds, written once.

Bounds (each compares a GPU output, decoded exactly to fp64, with the oracle's fp64 value):
  bf16 outputs (y, residual_out, dx): |err| <= 2^-8 * |ref| + 1e-6
  fp32 outputs (y, residual_out):     |err| <= 1e-5 * |ref| + 1e-6
  fp32 gradients (dx, d_r):           |err| <= 1e-5 * (|ref| + cond) + 1e-6, where cond is the
                                      magnitude of the terms the backward formula subtracts
                                      (rstd * (|g| + |xhat| * (|c| + mean|g * xhat|)), see
                                      bwd_cond): fp32 arithmetic is exact only relative to those
                                      terms, and dx can be far smaller than they are.
  rstd (fp32):                        |err| <= 1e-5 * |ref|
  LayerNorm mean (fp32):              |err| <= 1e-5 * (|ref| + 1 / rstd_ref)   (the row's scale)
  dw, db (fp32):                      |err| <= 1e-3 * max(|ref|, 1)
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

BF16_REL = 2.0 ** -8
ABS = 1e-6
F32_REL = 1e-5
RSTD_REL = 1e-5
DW_REL = 1e-3

TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


def to_dev(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Host array in its storage encoding (uint16 bf16 bits / float32) -> CUDA tensor."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> host array in its storage encoding."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def values(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 values of a CUDA tensor's elements."""
    return oracle.decode(to_host(t))


def _worst(err, bound, got, ref, what):
    ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.inf)
    bad = ~(err <= bound)
    i = np.unravel_index(np.argmax(np.where(bad, np.inf, ratio)) if bad.any()
                         else np.argmax(ratio), err.shape)
    return (f"{what}: {int(bad.sum())} of {err.size} outside the bound; worst at {tuple(int(k) for k in i)}: "
            f"got {got[i]!r}, want {ref[i]!r}, err/bound {ratio[i]:.3g}")


def check_out(got: np.ndarray, ref: np.ndarray, dtype: str, what: str, cond=None) -> float:
    """Assert the storage-type bound elementwise; return max err/bound. ``cond`` (fp32
    gradients only) widens the fp32 bound by the size of the cancelling terms."""
    rel = BF16_REL if dtype == "bf16" else F32_REL
    err = np.abs(got - ref)
    bound = rel * np.abs(ref) + ABS
    if cond is not None and dtype != "bf16":
        bound = bound + F32_REL * cond
    ok = err <= bound
    assert ok.all(), _worst(err, bound, got, ref, what)
    return float(np.max(err / bound)) if err.size else 0.0


def check_rstd(got: np.ndarray, ref: np.ndarray, what: str = "rstd") -> float:
    err = np.abs(got - ref)
    bound = RSTD_REL * np.abs(ref)
    ok = err <= bound
    assert ok.all(), _worst(err, bound, got, ref, what)
    return float(np.max(err / np.where(bound > 0, bound, 1.0))) if err.size else 0.0


def check_mean(got: np.ndarray, ref: np.ndarray, rstd_ref: np.ndarray, what: str = "mean") -> float:
    err = np.abs(got - ref)
    bound = RSTD_REL * (np.abs(ref) + 1.0 / rstd_ref)
    ok = err <= bound
    assert ok.all(), _worst(err, bound, got, ref, what)
    return float(np.max(err / bound)) if err.size else 0.0


def check_dw(got: np.ndarray, ref: np.ndarray, what: str = "dw") -> float:
    err = np.abs(got - ref)
    bound = DW_REL * np.maximum(np.abs(ref), 1.0)
    ok = err <= bound
    assert ok.all(), _worst(err, bound, got, ref, what)
    big = np.abs(ref) >= 1.0  # the pure relative error where it is well conditioned, reported
    if big.any():
        print(f"{what}: max relative error over |ref| >= 1: {float(np.max(err[big] / np.abs(ref[big]))):.2e}")
    return float(np.max(err / bound)) if err.size else 0.0


def bwd_cond(x: np.ndarray, dy: np.ndarray, w: np.ndarray, eps: float, layernorm: bool = False):
    """Per element, the magnitude of the terms the backward formula combines, from the
    oracle's rstd (and mean): rstd * (|g| + |mean g| + |xhat| * (|mean(g xhat)| + mean|g xhat|)),
    g = dy * w, xhat = (x - mean) * rstd. Used only to size the fp32 gradient bound."""
    xv = oracle.decode(np.ascontiguousarray(x))
    g = oracle.decode(np.ascontiguousarray(dy)) * oracle.decode(np.ascontiguousarray(w))[None, :]
    if layernorm:
        _, _, mean, rstd = oracle.add_layernorm_fwd(x, None, w, None, eps)
        xhat = (xv - mean[:, None]) * rstd[:, None]
        mg = np.abs(g.mean(axis=1, keepdims=True))
    else:
        _, rstd = oracle.rmsnorm_fwd(x, w, eps)
        xhat = xv * rstd[:, None]
        mg = 0.0
    gx = g * xhat
    c = np.abs(gx.mean(axis=1, keepdims=True)) + np.abs(gx).mean(axis=1, keepdims=True)
    return rstd[:, None] * (np.abs(g) + mg + np.abs(xhat) * c)


def bits_of(values_f32: np.ndarray, dtype: str) -> np.ndarray:
    """Storage encoding of float32 values (bf16 rounded to nearest even by torch's cast)."""
    import synth

    return synth.to_bf16_bits(values_f32) if dtype == "bf16" else np.asarray(values_f32, np.float32)
