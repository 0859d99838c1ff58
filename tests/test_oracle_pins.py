"""Pins of the float64 oracle against things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle (a window off by
one, a dropped max subtraction, a transposed GQA map, hi ignored, a wrong
rounding) fails at least one of them; ``test_planted_*`` plant such slips in
the oracle and check that the pins see them.  Sources: TensorFold pull
request #1123 ("window_attention at head dim 256"), sections "What this
changes" (definitions) and "Receipt" (gate 1 plants, gate 4 sums).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import wa_synth
from oracle import check


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def tval(b: np.ndarray) -> torch.Tensor:
    """bf16 bits -> float64 through torch's own conversion (independent of the oracle)."""
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double()


# ---------------------------------------------------------------------------
# Brute force: dense mask from the definition + torch float64 SDPA
# ---------------------------------------------------------------------------

def brute_decode(q, k, v, pos, win, ring, scale):
    qt, kt, vt = tval(q), tval(k), tval(v)
    R, hq, d = qt.shape
    hkv = kt.shape[2]
    out = torch.zeros(R, hq, d, dtype=torch.float64)
    for r in range(R):
        P = int(pos[r])
        kabs = torch.zeros(P + 1, hkv, d, dtype=torch.float64)
        vabs = torch.zeros(P + 1, hkv, d, dtype=torch.float64)
        mask = torch.zeros(P + 1, dtype=torch.bool)
        for j in range(P + 1):
            if win == 0 or j >= P - win + 1:
                mask[j] = True
                kabs[j] = kt[r, j % ring]
                vabs[j] = vt[r, j % ring]
        for h in range(hq):
            g = h * hkv // hq
            out[r, h] = F.scaled_dot_product_attention(
                qt[r, h].view(1, 1, 1, d), kabs[:, g].view(1, 1, -1, d), vabs[:, g].view(1, 1, -1, d),
                attn_mask=mask.view(1, 1, 1, -1), scale=scale).view(d)
    return out.numpy()


def brute_prompt(q, k, v, p0, win, ring, scale, hi=None):
    qt, kt, vt = tval(q), tval(k), tval(v)
    n, hq, d = qt.shape
    hkv = kt.shape[1]
    last = p0 + n  # absolute positions 0 .. p0+n-1
    out = torch.zeros(n, hq, d, dtype=torch.float64)
    for i in range(n):
        P = p0 + i
        H = P if hi is None else int(hi[i])
        kabs = torch.zeros(last, hkv, d, dtype=torch.float64)
        vabs = torch.zeros(last, hkv, d, dtype=torch.float64)
        mask = torch.zeros(last, dtype=torch.bool)
        for j in range(last):
            if j <= H and (win == 0 or j >= P - win + 1):
                mask[j] = True
                kabs[j] = kt[j % ring]
                vabs[j] = vt[j % ring]
        for h in range(hq):
            g = h * hkv // hq
            out[i, h] = F.scaled_dot_product_attention(
                qt[i, h].view(1, 1, 1, d), kabs[:, g].view(1, 1, -1, d), vabs[:, g].view(1, 1, -1, d),
                attn_mask=mask.view(1, 1, 1, -1), scale=scale).view(d)
    return out.numpy()


DECODE_TINY = [
    # rows, hq, hkv, d, win, ring, pos, scale
    (3, 4, 2, 8, 5, 7, [3, 12, 20], 0.7),      # wrapped rings, GQA 2
    (3, 2, 2, 4, 0, 24, [0, 10, 23], 1.0),     # linear cache, MHA
    (2, 8, 2, 8, 9, 11, [30, 39], 0.35),       # GQA 4, wrap
    (2, 16, 1, 4, 6, 6, [5, 17], 1.0),         # GQA 16, window == ring
]


@pytest.mark.parametrize("case", DECODE_TINY)
def test_decode_matches_brute_force(case):
    R, hq, hkv, d, win, ring, pos, scale = case
    c = wa_synth.decode_case(R, hq, hkv, d, win, ring, pos, seed=11 + d + win)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    got = oracle.decode(q, k, v, pos, win, ring, scale)
    want = brute_decode(q, k, v, pos, win, ring, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


PROMPT_TINY = [
    # n, p0, hq, hkv, d, win, ring, hi_spans, scale
    (10, 6, 4, 2, 4, 5, 16, [(2, 5)], 1.3),
    (9, 3, 2, 1, 8, 0, 12, [], 0.9),
    (12, 20, 8, 2, 4, 4, 15, [(0, 3), (7, 11)], 1.0),   # wraps: keys 17..31 in a ring of 15
]


@pytest.mark.parametrize("case", PROMPT_TINY)
def test_prompt_matches_brute_force(case):
    n, p0, hq, hkv, d, win, ring, spans, scale = case
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=5 + n, hi_spans=spans, peak_every=3)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    hi = None if c["hi"] is None else c["hi"].numpy()
    got = oracle.prompt(q, k, v, p0, win, ring, scale, hi=hi)
    want = brute_prompt(q, k, v, p0, win, ring, scale, hi=hi)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_mpmath_50_digits():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    R, hq, hkv, d, win, ring, pos, scale = 2, 4, 2, 8, 6, 9, [4, 25], 0.8
    c = wa_synth.decode_case(R, hq, hkv, d, win, ring, pos, seed=77)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    got = oracle.decode(q, k, v, pos, win, ring, scale)
    qt, kt, vt = tval(q), tval(k), tval(v)
    for r in range(R):
        P = pos[r]
        keys = range(max(0, P - win + 1), P + 1)
        for h in range(hq):
            g = h // (hq // hkv)
            s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(qt[r, h, e])) * mpmath.mpf(float(kt[r, j % ring, g, e]))
                                                 for e in range(d)) for j in keys]
            w = [mpmath.e ** x for x in s]
            l = mpmath.fsum(w)
            for e in range(d):
                o = mpmath.fsum(wj * mpmath.mpf(float(vt[r, j % ring, g, e])) for wj, j in zip(w, keys)) / l
                assert abs(got[r, h, e] - float(o)) <= 1e-13 * max(1.0, abs(float(o)))


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def test_weights_sum_to_one():
    rng = np.random.default_rng(3)
    qg = rng.standard_normal((4, 64))
    kv = rng.standard_normal((300, 64)) * 0.3
    _, w = oracle.attend(qg, kv, kv, 1.0)
    np.testing.assert_allclose((w / w.sum(axis=1, keepdims=True)).sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_one_key_window_returns_that_value():
    c = wa_synth.decode_case(2, 4, 2, 16, 1, 8, [5, 13], seed=9)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    got = oracle.decode(q, k, v, [5, 13], 1, 8, 1.0)
    vals = oracle.bf16_to_f64(v)
    for r, P in enumerate([5, 13]):
        for h in range(4):
            assert np.array_equal(got[r, h], vals[r, P % 8, h // 2])
    # position 0 of a linear cache sees one key as well
    c = wa_synth.decode_case(1, 2, 1, 8, 0, 4, [0], seed=10)
    got = oracle.decode(bits(c["q"]), bits(c["k"]), bits(c["v"]), [0], 0, 4, 1.0)
    assert np.array_equal(got[0, 0], oracle.bf16_to_f64(bits(c["v"]))[0, 0, 0])


def test_equal_scores_give_exact_mean():
    # gate 4's idea: every weight exactly 1, small integer values, a power-of-two count
    n, d = 1024, 8
    rng = np.random.default_rng(1)
    vint = rng.integers(-8, 9, size=(n, d)).astype(np.float64)
    kv = np.repeat(rng.standard_normal((1, d)), n, axis=0)  # all keys identical
    qg = rng.standard_normal((2, d))
    o, w = oracle.attend(qg, kv, vint, 1.0)
    assert np.all(w == 1.0)
    assert np.array_equal(o, np.repeat(vint.sum(axis=0, keepdims=True) / n, 2, axis=0))
    # q = 0 gives equal scores too
    o0, _ = oracle.attend(np.zeros((1, d)), rng.standard_normal((n, d)), vint, 1.0)
    assert np.array_equal(o0[0], vint.sum(axis=0) / n)


def test_invisible_keys_have_no_effect():
    R, hq, hkv, d, win, ring, pos = 2, 4, 2, 8, 6, 10, [7, 19]
    c = wa_synth.decode_case(R, hq, hkv, d, win, ring, pos, seed=21, outside="keep")
    q, k, v = bits(c["q"]), bits(c["k"]).copy(), bits(c["v"]).copy()
    base = oracle.decode(q, k, v, pos, win, ring, 1.0)
    for fill in (0x7FC0, 0x7F80, 0xFF80, 0x4120):  # NaN, +inf, -inf, 10.0
        k2, v2 = k.copy(), v.copy()
        for r, P in enumerate(pos):
            held = {j % ring for j in range(P - win + 1, P + 1)}
            for s in range(ring):
                if s not in held:
                    k2[r, s] = fill
                    v2[r, s] = fill
        got = oracle.decode(q, k2, v2, pos, win, ring, 1.0)
        assert np.array_equal(got, base, equal_nan=False)


def _lse_merge(parts):
    M = max(m for m, _, _ in parts)
    a = [math.exp(m - M) for m, _, _ in parts]
    num = sum(ai * o for ai, (_, _, o) in zip(a, parts))
    den = sum(ai * l for ai, (_, l, _) in zip(a, parts))
    return num / den


def test_chunked_lse_merge_equals_unsplit():
    R, hq, hkv, d, win, ring, pos = 1, 2, 1, 32, 1024, 1536, [1700]
    c = wa_synth.decode_case(R, hq, hkv, d, win, ring, pos, seed=31)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    whole = oracle.decode(q, k, v, pos, win, ring, 1.0)[0]
    lo, hi = oracle.visible_decode(pos[0], win)
    qf = oracle.bf16_to_f64(q[0])
    for h in range(hq):
        parts = []
        for cidx in range(lo // 256, hi // 256 + 1):
            a, b = max(lo, 256 * cidx), min(hi, 256 * cidx + 255)
            slots = np.arange(a, b + 1) % ring
            kk = oracle.bf16_to_f64(k[0, slots, 0])
            vv = oracle.bf16_to_f64(v[0, slots, 0])
            s = qf[h] @ kk.T
            m = s.max()
            w = np.exp(s - m)
            parts.append((m, w.sum(), w @ vv))
        np.testing.assert_allclose(_lse_merge(parts), whole[h], rtol=1e-13, atol=1e-14)


def test_hi_equal_own_position_matches_null_hi():
    n, p0, win, ring = 12, 9, 6, 24
    c = wa_synth.prompt_case(n, p0, 4, 2, 8, win, ring, seed=41)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    a = oracle.prompt(q, k, v, p0, win, ring, 1.0, hi=None)
    b = oracle.prompt(q, k, v, p0, win, ring, 1.0, hi=np.arange(p0, p0 + n))
    assert np.array_equal(a, b)


def test_wide_window_matches_linear_cache():
    pos = [0, 9, 30]
    c = wa_synth.decode_case(3, 4, 2, 8, 0, 32, pos, seed=51, outside="keep")
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    a = oracle.decode(q, k, v, pos, 0, 32, 1.0)
    b = oracle.decode(q, k, v, pos, 31, 32, 1.0)   # win >= pos + 1 for every row
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# Special values (the "gate 1" plants of the receipt)
# ---------------------------------------------------------------------------

def _prompt_plain(n=8, p0=0, d=4, seed=61):
    c = wa_synth.prompt_case(n, p0, 2, 1, d, 0, n + p0, seed=seed, peaked=False)
    return bits(c["q"]).copy(), bits(c["k"]).copy(), bits(c["v"]).copy()


def test_special_nan_query_stays_in_its_row_and_head():
    q, k, v = _prompt_plain()
    q[3, 1, 2] = 0x7FC0
    out = oracle.prompt(q, k, v, 0, 0, 8, 1.0)
    assert np.isnan(out[3, 1]).all()
    assert np.isfinite(np.delete(out.reshape(-1, 4), 3 * 2 + 1, axis=0)).all()


def test_special_nan_key_reaches_only_rows_that_see_it():
    q, k, v = _prompt_plain()
    k[5, 0, 0] = 0x7FC0
    out = oracle.prompt(q, k, v, 0, 0, 8, 1.0)
    assert np.isfinite(out[:5]).all() and np.isnan(out[5:]).all()


def test_special_inf_value_seen_by_later_rows_only():
    q, k, v = _prompt_plain()
    v[6, 0, 1] = 0x7F80
    out = oracle.prompt(q, k, v, 0, 0, 8, 1.0)
    assert np.isfinite(out[:6]).all()
    assert np.all(out[6:, :, 1] == np.inf)
    assert np.isfinite(np.delete(out[6:], 1, axis=2)).all()


def test_special_plus_and_minus_inf_in_one_column_is_nan():
    q, k, v = _prompt_plain()
    v[2, 0, 3] = 0x7F80
    v[4, 0, 3] = 0xFF80
    out = oracle.prompt(q, k, v, 0, 0, 8, 1.0)
    assert np.all(out[2:4, :, 3] == np.inf)
    assert np.isnan(out[4:, :, 3]).all()


def test_special_inf_at_a_tiny_float64_weight_is_inf():
    # score gap of 200: float64 weight e^-200 > 0, fp32's would be 0
    q = oracle.f64_to_bf16(np.array([[[1.0, 0.0]]]))                 # [1,1,2]
    k = oracle.f64_to_bf16(np.array([[[200.0, 0.0]], [[0.0, 0.0]]]))  # keys 0, 1
    v = oracle.f64_to_bf16(np.array([[[1.0, 2.0]], [[np.inf, 3.0]]]))
    out = oracle.decode(q[None].reshape(1, 1, 2), k[None], v[None], [1], 0, 2, 1.0)
    assert out[0, 0, 0] == np.inf
    assert abs(out[0, 0, 1] - 2.0) < 1e-80 + 1e-15
    assert np.float32(np.exp(np.float32(-200.0))) == 0.0


# ---------------------------------------------------------------------------
# bf16 rounding (RN-even, sign kept on underflow)
# ---------------------------------------------------------------------------

def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),     # subnormals
        np.float32([0.0, -0.0, 3.3895e38, 3.3961e38, 3.4e38, -3.4e38, np.inf, -np.inf, 1e-45, -1e-45]),
        rng.integers(0, 2**32, 50000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x = x[np.isfinite(x) | np.isinf(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_roundtrip_and_ties_to_even():
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f64(allb)
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.f64_to_bf16(vals[ok]), allb[ok])
    pos = allb[(allb < 0x7F7F) & (allb > 0)]
    a, b = oracle.bf16_to_f64(pos), oracle.bf16_to_f64(pos + 1)
    mid = (a + b) / 2  # exact in float64
    even = np.where(pos % 2 == 0, pos, pos + 1)
    assert np.array_equal(oracle.f64_to_bf16(mid), even.astype(np.uint16))
    assert oracle.f64_to_bf16(np.array([-1e-300]))[0] == 0x8000


def test_p32_split_within_2_to_minus_16():
    # "Window.p32": P enters as bf16(P) + bf16(P - bf16(P)), fp32's P to 2^-16
    rng = np.random.default_rng(5)
    exps = np.arange(-30, 1)
    for e in exps:
        mant = np.concatenate([np.arange(0, 1 << 23, 97, dtype=np.uint32), rng.integers(0, 1 << 23, 4000).astype(np.uint32)])
        p = ((np.uint32(e + 127) << np.uint32(23)) | mant).view(np.float32).astype(np.float64)
        p = p[p <= 1.0]
        hi = oracle.bf16_to_f64(oracle.f64_to_bf16(p))
        lo = oracle.bf16_to_f64(oracle.f64_to_bf16(np.float32(p - hi).astype(np.float64)))
        assert np.all(np.abs(p - (hi + lo)) <= 2.0 ** -16 * p)


def test_three_part_split_is_exact_to_fp32():
    # TensorFold #1622, review thread: P carried as hi + mid + lo 16-bit parts whose fp32 sum
    # is the value.  Each residual is exact in fp32, and the three parts hold P to 2^-24.
    rng = np.random.default_rng(6)
    for e in np.arange(-30, 1):
        mant = np.concatenate([np.arange(0, 1 << 23, 89, dtype=np.uint32), rng.integers(0, 1 << 23, 4000).astype(np.uint32)])
        p = ((np.uint32(e + 127) << np.uint32(23)) | mant).view(np.float32).astype(np.float64)
        p = p[p <= 1.0]
        parts, r = [], p.copy()
        for _ in range(3):
            b16 = oracle.bf16_to_f64(oracle.f64_to_bf16(r))
            parts.append(b16)
            nr = r - b16
            assert np.array_equal(np.float32(nr).astype(np.float64), nr)   # exact in fp32
            r = nr
        assert np.all(np.abs(p - (parts[0] + parts[1] + parts[2])) <= 2.0 ** -24 * p)


# ---------------------------------------------------------------------------
# The checker
# ---------------------------------------------------------------------------

def test_checker_interval_and_classes():
    o = np.array([1.0, 1.0 + 2 ** -8, -0.5, np.nan, np.inf, -np.inf, 0.0])
    g = oracle.f64_to_bf16(np.array([1.0, 1.0 + 2 ** -7, -0.5, np.nan, np.inf, -np.inf, -0.0]))
    r = check.compare(g, o, 3e-3)
    assert r["ok"], r
    g2 = g.copy(); g2[1] = oracle.f64_to_bf16(np.array([1.0 + 2 ** -6]))[0]
    assert not check.compare(g2, o, 3e-3)["ok"]
    g3 = g.copy(); g3[3] = 0x7F80
    assert not check.compare(g3, o, 3e-3)["ok"]
    g4 = g.copy(); g4[4] = 0x7FC0
    assert not check.compare(g4, o, 3e-3)["ok"]


# ---------------------------------------------------------------------------
# Planted mistakes: each must make a pin fail
# ---------------------------------------------------------------------------

def test_planted_window_one_key_early_is_caught(monkeypatch):
    def early(p, win):
        lo = max(0, p - win) if win > 0 else 0
        return lo, p
    monkeypatch.setattr(oracle, "visible_decode", early)
    R, hq, hkv, d, win, ring, pos, scale = DECODE_TINY[0]
    c = wa_synth.decode_case(R, hq, hkv, d, win, ring, pos, seed=11 + d + win, outside="keep")
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    got = oracle.decode(q, k, v, pos, win, ring, scale)
    want = brute_decode(q, k, v, pos, win, ring, scale)
    assert not np.allclose(got, want, rtol=1e-6)


def test_planted_hi_ignored_is_caught(monkeypatch):
    real = oracle.visible_prompt
    monkeypatch.setattr(oracle, "visible_prompt", lambda p0, i, win, hi_i=None: real(p0, i, win, None))
    n, p0, hq, hkv, d, win, ring, spans, scale = PROMPT_TINY[0]
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=5 + n, hi_spans=spans, peak_every=3)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    hi = c["hi"].numpy()
    got = oracle.prompt(q, k, v, p0, win, ring, scale, hi=hi)
    want = brute_prompt(q, k, v, p0, win, ring, scale, hi=hi)
    assert not np.allclose(got, want, rtol=1e-6)


def test_planted_gqa_map_transposed_is_caught():
    R, hq, hkv, d, win, ring, pos, scale = DECODE_TINY[2]
    c = wa_synth.decode_case(R, hq, hkv, d, win, ring, pos, seed=11 + d + win)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    want = brute_decode(q, k, v, pos, win, ring, scale)
    # query head h read with key head h % hkv instead of h // G
    perm = [h % hkv * (hq // hkv) + h // hkv for h in range(hq)]
    got = oracle.decode(q[:, perm], k, v, pos, win, ring, scale)[:, np.argsort(perm)]
    assert not np.allclose(got, want, rtol=1e-6)


def test_planted_merge_without_rescale_is_caught():
    R, hq, hkv, d, win, ring, pos = 1, 1, 1, 32, 1024, 1536, [1700]
    c = wa_synth.decode_case(R, hq, hkv, d, win, ring, pos, seed=31)
    q, k, v = bits(c["q"]), bits(c["k"]), bits(c["v"])
    whole = oracle.decode(q, k, v, pos, win, ring, 1.0)[0, 0]
    lo, hi = oracle.visible_decode(pos[0], win)
    qf = oracle.bf16_to_f64(q[0, 0])
    num, den = 0.0, 0.0
    for cidx in range(lo // 256, hi // 256 + 1):
        a, b = max(lo, 256 * cidx), min(hi, 256 * cidx + 255)
        slots = np.arange(a, b + 1) % ring
        s = qf @ oracle.bf16_to_f64(k[0, slots, 0]).T
        w = np.exp(s - s.max())
        num = num + w @ oracle.bf16_to_f64(v[0, slots, 0])   # no exp(m_c - M)
        den = den + w.sum()
    r = check.compare(oracle.f64_to_bf16(num / den), whole, check.TOL_FP32_P)
    assert not r["ok"]


def test_planted_rounding_toward_zero_is_caught():
    vals = np.array([1.0 + 3 * 2 ** -9, -(1.0 + 3 * 2 ** -9)])
    trunc = (np.float32(vals).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert not np.array_equal(trunc, oracle.f64_to_bf16(vals))
