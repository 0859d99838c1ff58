"""Pins of the float64 preparation oracle against things other than itself (CPU).

RMSNorm (page "Exact Numerical Contract", section "Preparation") against
torch's own float64 rms_norm and a closed form; rotate-half RoPE (TensorFold
pull request #1257, "What the kernel computes") against complex
multiplication, the identity at position 0, pair norms and the relative
position property; the fp32 angle against exact rational rounding; the L2
norm against numpy's norm and its special cases; and planted mistakes at each
rounding point, which the checker must reject.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import prep


def _bf16_rows(rng, shape, scale=1.0):
    x = torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def test_rmsnorm_matches_torch_rms_norm_float64():
    rng = np.random.default_rng(1)
    for d in (128, 256):
        x = oracle.bf16_to_f64(_bf16_rows(rng, (50, d), 3.0))
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (d,), eps=1e-5).numpy()
        assert np.allclose(prep.rmsnorm_head(x), ref, rtol=1e-14, atol=0)


def test_rmsnorm_constant_vector_closed_form():
    for c in (0.5, -3.0, 1e-3):
        x = np.full(128, c)
        y = prep.rmsnorm_head(x)
        assert np.all(y == c / math.sqrt(c * c + 1e-5))


def test_rope_is_complex_multiplication():
    rng = np.random.default_rng(2)
    d = 256
    x = rng.standard_normal(d)
    ang = rng.uniform(-50, 50, d // 2)
    z = (x[:d // 2] + 1j * x[d // 2:]) * np.exp(1j * ang)
    r = prep.rope_rotate_half(x, ang)
    assert np.allclose(r[:d // 2], z.real, rtol=0, atol=1e-14)
    assert np.allclose(r[d // 2:], z.imag, rtol=0, atol=1e-14)


def test_rope_position_zero_is_identity_and_pairs_keep_their_norm():
    rng = np.random.default_rng(3)
    d = 128
    inv = (1.0 / 10000.0 ** (np.arange(0, d, 2) / d)).astype(np.float32)
    x = rng.standard_normal(d)
    assert np.array_equal(prep.rope_rotate_half(x, prep.rope_angle32(0, inv)), x)
    r = prep.rope_rotate_half(x, prep.rope_angle32(12345, inv))
    h = d // 2
    assert np.allclose(r[:h] ** 2 + r[h:] ** 2, x[:h] ** 2 + x[h:] ** 2, rtol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    # power-of-two inverse frequencies keep fl32(pos * inv) exact, so the property holds exactly
    rng = np.random.default_rng(4)
    d = 64
    inv = (2.0 ** -np.arange(d // 2, dtype=np.float64) / 4).astype(np.float32)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    def score(m, n):
        return prep.rope_rotate_half(q, prep.rope_angle32(m, inv)) @ prep.rope_rotate_half(k, prep.rope_angle32(n, inv))
    assert abs(score(10, 3) - score(1010, 1003)) < 1e-10
    assert abs(score(7, 7) - q @ k) < 1e-10


def test_angle_is_the_fp32_product_rounded_to_nearest():
    rng = np.random.default_rng(5)
    inv = rng.uniform(1e-6, 1.0, 64).astype(np.float32)
    for pos in (1, 3, 777, 199_999, 2**23 + 1):
        got = prep.rope_angle32(pos, inv)
        for j in range(0, 64, 7):
            exact = Fraction(pos) * Fraction(float(inv[j]))
            # round the exact rational to 24 significant bits, ties to even
            e = math.floor(math.log2(exact))
            q = exact / Fraction(2) ** (e - 23)
            f = math.floor(q)
            rem = q - f
            f = f + (1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1) else 0)
            assert got[j] == float(Fraction(f) * Fraction(2) ** (e - 23)), (pos, j)


def test_l2_head_against_numpy_norm_and_zero():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((10, 256)) * 4
    y = prep.l2_head(x)
    ref = x / np.sqrt(np.linalg.norm(x, axis=1, keepdims=True) ** 2 + 1e-6)
    assert np.allclose(y, ref, rtol=1e-13)
    assert np.allclose(np.linalg.norm(y, axis=1), 1.0, atol=1e-7)
    assert np.array_equal(prep.l2_head(np.zeros(128)), np.zeros(128))


def _src(rng, n, hq, hkv, d):
    return _bf16_rows(rng, (n, (hq + 2 * hkv) * d))


def test_prepare_splits_heads_and_copies_v():
    rng = np.random.default_rng(7)
    n, hq, hkv, d = 3, 4, 2, 128
    src = _src(rng, n, hq, hkv, d)
    q, k, v = prep.prepare(src, [0, 5, 9], hq, hkv, d, "rmsnorm")
    x = oracle.bf16_to_f64(src).reshape(n, hq + 2 * hkv, d)
    assert np.array_equal(q, prep.rmsnorm_head(x[:, :hq]))
    assert np.array_equal(k, prep.rmsnorm_head(x[:, hq:hq + hkv]))
    assert np.array_equal(v, src.reshape(n, hq + 2 * hkv, d)[:, hq + hkv:])


def _planted_l2_rope(src, pos, hq, hkv, d, q_scale, inv, drop):
    """The l2_rope preparation with one rounding point dropped (planted mistake)."""
    n = src.shape[0]
    x = oracle.bf16_to_f64(src).reshape(n, hq + 2 * hkv, d)
    out = np.empty((n, hq, d))
    for t in range(n):
        ang = prep.rope_angle32(int(pos[t]), inv)
        r = prep.rope_rotate_half(x[t, :hq], ang)
        if drop != "rope":
            r = prep._rn(r)
        qn = prep.l2_head(r)
        if drop != "norm":
            qn = prep._rn(qn)
        out[t] = np.asarray(q_scale, dtype=np.float64) * qn
    return out


@pytest.mark.parametrize("drop", ["rope", "norm"])
def test_checker_rejects_a_dropped_rounding_point(drop):
    rng = np.random.default_rng(8)
    n, hq, hkv, d = 16, 8, 2, 256
    src = _src(rng, n, hq, hkv, d)
    pos = rng.integers(0, 200_000, n)
    inv = (1.0 / 10000.0 ** (np.arange(0, d, 2) / d)).astype(np.float32)
    qs = rng.uniform(0.5, 2.0, d).astype(np.float32)
    q_ref, _, _, q_tol, _ = prep.prepare(src, pos, hq, hkv, d, "l2_rope", qs, inv, with_allowance=True)
    good = oracle.f64_to_bf16(_planted_l2_rope(src, pos, hq, hkv, d, qs, inv, drop=None))
    assert prep.check_prep(good, q_ref, q_tol)["ok"]
    bad = oracle.f64_to_bf16(_planted_l2_rope(src, pos, hq, hkv, d, qs, inv, drop=drop))
    r = prep.check_prep(bad, q_ref, q_tol)
    assert not r["ok"], r


def test_checker_rejects_sign_error_and_swapped_halves():
    rng = np.random.default_rng(9)
    n, hq, hkv, d = 8, 4, 2, 128
    src = _src(rng, n, hq, hkv, d)
    pos = rng.integers(1, 50_000, n)
    inv = (1.0 / 10000.0 ** (np.arange(0, d, 2) / d)).astype(np.float32)
    q_ref, k_ref, _, _, k_tol = prep.prepare(src, pos, hq, hkv, d, "l2_rope", None, inv, with_allowance=True)
    x = oracle.bf16_to_f64(src).reshape(n, hq + 2 * hkv, d)[:, hq:hq + hkv]
    for t in range(n):
        ang = prep.rope_angle32(int(pos[t]), inv)
        wrong = prep.l2_head(prep._rn(prep.rope_rotate_half(x[t], -ang)))   # rotation the wrong way
        assert not prep.check_prep(oracle.f64_to_bf16(wrong), k_ref[t], k_tol[t])["ok"]
        halves = np.concatenate([x[t][:, d // 2:], x[t][:, :d // 2]], axis=-1)   # halves swapped
        wrong = prep.l2_head(prep._rn(prep.rope_rotate_half(halves, ang)))
        assert not prep.check_prep(oracle.f64_to_bf16(wrong), k_ref[t], k_tol[t])["ok"]


def test_rotation_allowance_covers_fp32_cancellation():
    """An fp32 evaluation of the rotation (numpy float32, correctly rounded cos/sin) stays inside
    the allowance, including rows where the two terms cancel."""
    rng = np.random.default_rng(11)
    n, hq, hkv, d = 64, 4, 2, 128
    src = _src(rng, n, hq, hkv, d)
    pos = rng.integers(0, 200_000, n)
    inv = (1.0 / 10000.0 ** (np.arange(0, d, 2) / d)).astype(np.float32)
    _, k_ref, _, _, k_tol = prep.prepare(src, pos, hq, hkv, d, "l2_rope", None, inv, with_allowance=True)
    x = oracle.bf16_to_f64(src).reshape(n, hq + 2 * hkv, d)[:, hq:hq + hkv].astype(np.float32)
    out = np.empty((n, hkv, d))
    for t in range(n):
        ang = prep.rope_angle32(int(pos[t]), inv).astype(np.float32)
        c, s = np.cos(ang.astype(np.float64)).astype(np.float32), np.sin(ang.astype(np.float64)).astype(np.float32)
        lo, hi = x[t][:, :d // 2], x[t][:, d // 2:]
        r = np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1).astype(np.float64)
        r = prep._rn(r)
        ss = np.sum((r * r).astype(np.float32), axis=-1, keepdims=True, dtype=np.float32)
        out[t] = (r.astype(np.float32) * (np.float32(1) / np.sqrt(ss + np.float32(1e-6)))).astype(np.float64)
    assert prep.check_prep(oracle.f64_to_bf16(out), k_ref, k_tol)["ok"]


def test_checker_rmsnorm_allowance_is_tight_enough():
    rng = np.random.default_rng(10)
    x = oracle.bf16_to_f64(_bf16_rows(rng, (64, 256)))
    y = prep.rmsnorm_head(x)
    assert prep.check_prep(oracle.f64_to_bf16(y), y, prep.REL_RMSNORM)["ok"]
    # eps 1e-4 instead of 1e-5 on small-norm rows moves outputs by more than the allowance
    xs = x * 1e-2
    wrong = xs / np.sqrt(np.mean(xs * xs, axis=-1, keepdims=True) + 1e-4)
    assert not prep.check_prep(oracle.f64_to_bf16(wrong), prep.rmsnorm_head(xs), prep.REL_RMSNORM)["ok"]
