"""Tolerances and comparison helpers for CUDA-vs-oracle parity.

Tolerances (stated once, used by every parity test):
  * bf16 outputs: |o_gpu - o_ref| <= 2e-3 + ulp_bf16(|o_ref|) element-wise.
    The 2e-3 absolute bound is the stated target; one bf16 ulp of the exact
    value is added because rounding the exact result to bf16 alone already
    costs up to half an ulp, which exceeds 2e-3 once |o| >= 0.5.
  * fp32 outputs (the fp32 single-head workload): |o_gpu - o_ref| <= 1e-4.
  * LSE (fp32): |lse_gpu - lse_ref| <= 1e-4; an empty row must give -inf
    exactly on both sides.
"""
from __future__ import annotations

import numpy as np
import torch

BF16_ABS = 2e-3
F32_ABS = 1e-4
LSE_ABS = 1e-4


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 7)


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.float()
        return t.numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def check_out(out, ref, dtype, what="o"):
    o = to_np(out)
    r = np.asarray(ref, dtype=np.float64)
    assert o.shape == r.shape, (o.shape, r.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - r)
    if dtype == torch.bfloat16:
        tol = BF16_ABS + ulp_bf16(r)
    else:
        tol = np.full_like(r, F32_ABS)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} elements out of tolerance; worst at {i}: "
            f"gpu={o[i]!r} ref={r[i]!r} err={err[i]:.3e} tol={tol[i]:.3e}")
    return float(err.max()) if err.size else 0.0


def check_lse(out, ref, what="lse"):
    o = to_np(out)
    r = np.asarray(ref, dtype=np.float64)
    assert o.shape == r.shape
    empty = np.isneginf(r)
    assert np.array_equal(np.isneginf(o), empty), f"{what}: -inf pattern differs"
    if (~empty).any():
        err = np.abs(o[~empty] - r[~empty])
        assert np.all(np.isfinite(o[~empty])), f"{what}: non-finite"
        assert err.max() <= LSE_ABS, f"{what}: max err {err.max():.3e} > {LSE_ABS}"
        return float(err.max())
    return 0.0
