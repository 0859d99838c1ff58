"""Interval checker: bf16 outputs against float64 oracle values (TEST INFRASTRUCTURE).

The comparison follows TensorFold pull request #1123, section "What this
changes", bullet "core/attention_range.zig": both ends of the allowed range
are rounded to bf16 and the output is compared in value order, -0 below +0;
NaN matches only NaN and infinities match by their bits.

Reading of the tolerance: the allowed range around the float64 value o is
[o - tol, o + tol] with tol = 3e-3 for fp32 probabilities (decode) and the
two-half P (P32), 8e-3 for a single bf16 P.  A bf16 output passes when it
lies between RN_bf16(o - tol) and RN_bf16(o + tol) in value order.  A literal
max |gpu - o| <= 3e-3 cannot hold for |o| >= 1, whose bf16 half-step is
already 2^-8 (about 3.9e-3).
"""
from __future__ import annotations

import numpy as np

from . import bf16_to_f64, f64_to_bf16

TOL_FP32_P = 3e-3
TOL_P32 = 3e-3
TOL_BF16_P = 8e-3
# P in three bf16 parts: the fp32-accurate mode, held to the scalar kernel's bound 1e-5
# (TensorFold pull request #1622, review thread: "holds the tile to 1e-5 against fp64")
TOL_P3 = 1e-5


def order_key(bits) -> np.ndarray:
    """Total order of bf16 bit patterns by value, with -0 just below +0."""
    b = np.asarray(bits).astype(np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag - 1, mag)


def is_nan_bits(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint16).astype(np.int64)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def compare(gpu_bits, ref, tol: float) -> dict:
    """Compare bf16 bits against float64 values elementwise.

    Returns counts and the worst deviations; ``ok`` is True when every element
    passes.  Elements where ``ref`` is NaN because they were not sampled must
    be removed by the caller beforehand."""
    g = np.asarray(gpu_bits).astype(np.uint16).ravel()
    o = np.asarray(ref, dtype=np.float64).ravel()
    assert g.shape == o.shape, (g.shape, o.shape)
    g_nan = is_nan_bits(g)
    o_nan = np.isnan(o)
    o_inf = np.isinf(o)
    fin = ~o_nan & ~o_inf
    bad = np.zeros(g.shape, dtype=bool)
    bad |= o_nan & ~g_nan
    bad |= o_inf & (g != f64_to_bf16(o))
    with np.errstate(invalid="ignore", over="ignore"):
        lo = f64_to_bf16(np.where(fin, o - tol, 0.0))
        hi = f64_to_bf16(np.where(fin, o + tol, 0.0))
    kg = order_key(g)
    inside = (order_key(lo) <= kg) & (kg <= order_key(hi)) & ~g_nan
    bad |= fin & ~inside
    gv = bf16_to_f64(g)
    with np.errstate(invalid="ignore"):
        err = np.where(fin & ~g_nan, np.abs(gv - o), 0.0)
        rn = f64_to_bf16(np.where(fin, o, 0.0))
        ulps = np.where(fin & ~g_nan, np.abs(order_key(g) - order_key(rn)), 0)
    return {
        "ok": not bad.any(),
        "n": int(g.size),
        "n_bad": int(bad.sum()),
        "first_bad": int(np.argmax(bad)) if bad.any() else -1,
        "max_abs_err": float(err.max()) if err.size else 0.0,
        "max_ulps": int(ulps.max()) if ulps.size else 0,
        "n_bit_equal": int((fin & (g == rn)).sum()),
        "n_nonfinite_ref": int((~fin).sum()),
    }
