"""Float64 oracle for the q/k preparation and KV append (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  It shares no code with the CUDA library.

The step before attention: a token's projection row holds hq query heads, then
hkv key heads, then hkv value heads, each of d bf16 values.  The step prepares
q and k and writes k and v into ring slot pos mod ring.  Two preparations:

* ``rmsnorm`` (page "Exact Numerical Contract", section "Preparation"): per
  head, y = x / sqrt(mean(x^2) + 1e-5), normalised in fp32 and rounded once to
  bf16.  The oracle returns the float64 value of that expression; the fp32
  evaluation on the GPU is within 2^-16 of it relative (the bound of a
  sequential fp32 sum of d <= 256 squares, one square root, one divide and one
  product), which :func:`check_prep` allows before the final rounding.

* ``l2_rope`` (TensorFold pull request #1257, section "What the kernel
  computes"): rotate-half RoPE on the bf16 projection in fp32 with the angle
  fl32(pos * inv_j) and fp32 cos/sin, rounded once to bf16; then the L2 norm
  x * (1 / sqrt(sum(x^2) + 1e-6)) of the rounded head, rounded to bf16; for q
  a further product with an fp32 per-dimension scale qs, rounded to bf16.
  Rounding points: the rotated head, the normalised head, q after the scale.
  The angle is the one quantity the pages fix in fp32 (fl32 of the product),
  so the oracle forms it as an fp32 product too and takes float64 cos/sin of
  that fp32 angle.  Every other step is float64, with bf16 rounding (this
  package's own round-to-nearest-even) at the three points.

  Allowance (the pages compare "with float64's range at its rounding points
  (cosf's ulps on the fp32 angle)").  An fp32 rotation with cosf/sinf within
  2 ulps, two rounded products and a rounded difference is within
  2^-21 (|x_a cos| + |x_b sin|) of the float64 rotation.  Where the two terms
  cancel, that is many bf16 steps of the rotated value, and it reaches the
  output scaled by the normalisation (and q_scale).  So each output j is
  allowed |o_j| 2^-6 (one bf16 step at each earlier rounding point) plus
  s_j (e_j + ulp_bf16(|r_j| + e_j)) / N, with e_j the rotation bound, r_j the
  rotated value, N the head's norm and s_j the q scale (1 for k).

v is copied as is.  Reading of "rotate-half": dimension j < d/2 pairs with
j + d/2; x'_j = x_j cos - x_{j+d/2} sin and x'_{j+d/2} = x_{j+d/2} cos +
x_j sin, with the angle of frequency j.

Pins: tests/test_oracle_prep_pins.py.
"""
from __future__ import annotations

import numpy as np

from . import bf16_to_f64, f64_to_bf16

RMS_EPS = 1e-5
L2_EPS = 1e-6

__all__ = ["rmsnorm_head", "rope_angle32", "rope_rotate_half", "l2_head", "prepare", "check_prep",
           "REL_RMSNORM", "REL_L2ROPE"]

# fp32 evaluation error allowed around the float64 value before the final bf16 rounding
REL_RMSNORM = 2.0 ** -16
# l2_rope: a value near a bf16 boundary at one of the two earlier rounding points may round
# the other way in fp32, moving the output by up to one bf16 step (2^-7 relative) per point
REL_L2ROPE = 2.0 ** -6


def rmsnorm_head(x: np.ndarray) -> np.ndarray:
    """x / sqrt(mean(x^2) + 1e-5) along the last axis, float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):   # IEEE classes pass through as the formula says
        ms = np.mean(x * x, axis=-1, keepdims=True)
        return x / np.sqrt(ms + RMS_EPS)


def rope_angle32(pos: int, inv_freq32: np.ndarray) -> np.ndarray:
    """fl32(pos * inv_j): the fp32 product of the position (exact in fp32 below 2^24) and the
    fp32 inverse frequency, as float64."""
    p = np.float32(pos)
    inv = np.asarray(inv_freq32, dtype=np.float32)
    return (p * inv).astype(np.float32).astype(np.float64)


def rope_rotate_half(x: np.ndarray, ang: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE in float64: x [..., d], ang [d/2] (float64 values of the fp32 angles)."""
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def l2_head(x: np.ndarray) -> np.ndarray:
    """x * (1 / sqrt(sum(x^2) + 1e-6)) along the last axis, float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        return x * (1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS))


def _rn(x):
    """bf16 round-to-nearest-even of float64 values, back to float64 (a rounding point)."""
    return bf16_to_f64(f64_to_bf16(x))


def _ulp_bf16(a):
    """Spacing of bf16 values at magnitude a (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(a), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def _rotation_bound(x, ang):
    """Bound on |fp32 rotation - float64 rotation| per output dimension (see the module text)."""
    h = x.shape[-1] // 2
    c, s = np.abs(np.cos(ang)), np.abs(np.sin(ang))
    lo, hi = np.abs(x[..., :h]), np.abs(x[..., h:])
    e = 2.0 ** -21 * (lo * c + hi * s)
    e2 = 2.0 ** -21 * (hi * c + lo * s)
    return np.concatenate([e, e2], axis=-1)


def prepare(src_bits, pos, hq: int, hkv: int, d: int, mode: str, q_scale=None, inv_freq=None,
            with_allowance: bool = False):
    """Prepared q and k of every token (float64, before the final bf16 rounding) and v's bits.

    src_bits [n, (hq + 2 hkv) * d] bf16 bits, pos [n].  Returns (q [n, hq, d], k [n, hkv, d],
    v_bits [n, hkv, d]), and with ``with_allowance`` also the absolute allowances (q_tol, k_tol)
    of the l2_rope preparation (None for rmsnorm, whose allowance is relative).  Tokens with a
    negative position are not written by the step; the oracle still returns their values."""
    src = np.asarray(src_bits).astype(np.uint16)
    n = src.shape[0]
    x = bf16_to_f64(src[:, :(hq + 2 * hkv) * d]).reshape(n, hq + 2 * hkv, d)
    xq, xk = x[:, :hq], x[:, hq:hq + hkv]
    v_bits = src[:, (hq + hkv) * d:(hq + 2 * hkv) * d].reshape(n, hkv, d)
    if mode == "rmsnorm":
        out = (rmsnorm_head(xq), rmsnorm_head(xk), v_bits)
        return out + (None, None) if with_allowance else out
    if mode != "l2_rope":
        raise ValueError(mode)
    qs = np.ones(d) if q_scale is None else np.asarray(q_scale, dtype=np.float32).astype(np.float64)
    q_out = np.empty((n, hq, d))
    k_out = np.empty((n, hkv, d))
    q_tol = np.empty((n, hq, d))
    k_tol = np.empty((n, hkv, d))
    for t in range(n):
        ang = rope_angle32(int(pos[t]), inv_freq)
        rq64 = rope_rotate_half(xq[t], ang)
        rk64 = rope_rotate_half(xk[t], ang)
        rq = _rn(rq64)                                    # rounding point: rotated head
        rk = _rn(rk64)
        qn = _rn(l2_head(rq))                             # rounding point: normalised head
        q_out[t] = qs * qn                                # rounded by the check: q after the scale
        k_out[t] = l2_head(rk)                            # rounded by the check
        if with_allowance:
            for r64, xh, sc, o, tol in ((rq64, xq[t], qs, q_out[t], q_tol), (rk64, xk[t], 1.0, k_out[t], k_tol)):
                e = _rotation_bound(xh, ang)
                with np.errstate(invalid="ignore", over="ignore"):
                    norm = np.sqrt(np.sum(_rn(r64) ** 2, axis=-1, keepdims=True) + L2_EPS)
                    tol[t] = REL_L2ROPE * np.abs(o) + sc * (e + _ulp_bf16(np.abs(r64) + e)) / norm
    if with_allowance:
        return q_out, k_out, v_bits, q_tol, k_tol
    return q_out, k_out, v_bits


def check_prep(gpu_bits, ref, tol, min_bit_equal: float = 0.99) -> dict:
    """bf16 outputs against float64 values with an allowance before the final rounding.

    ``tol`` is a relative allowance (a float) or an array of absolute allowances.  An output
    passes when it lies in [RN(o - t), RN(o + t)] in value order.  On top, the share of outputs
    equal to RN(o) must reach ``min_bit_equal``: a missing or extra rounding point moves a large
    share of outputs by one step while staying inside the allowance."""
    from .check import compare
    o = np.asarray(ref, dtype=np.float64)
    if np.ndim(tol) == 0:
        t = float(tol) * np.abs(o).ravel()
    else:
        t = np.asarray(tol, dtype=np.float64).ravel()
    r = compare(gpu_bits, o, t)
    fin = int(np.isfinite(o).sum())
    r["bit_equal_share"] = r["n_bit_equal"] / max(1, fin)
    r["ok"] = bool(r["ok"] and r["bit_equal_share"] >= min_bit_equal)
    return r
