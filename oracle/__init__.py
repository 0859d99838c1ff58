"""Float64 oracle for sliding-window grouped-query attention (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library and
imports nothing from it.

What it computes, per row and query head h (key head g = h // G, G = hq/hkv),
as defined by TensorFold pull request #1123 ("window_attention at head dim
256"), section "What this changes":

* visible keys (bullets "Decode", "promptRows(..., hi)" and "Scale is a
  parameter"): a decode row at position p sees keys [lo, p]; prompt row i of
  a chunk at p0 sees keys [lo_i, hi[i]] with hi[i] defaulting to p0 + i; the
  window start is lo = max(0, p - win + 1), or 0 for win = 0 (a linear cache
  whose ring is its length);
* the slot of key j in a ring of length ``ring`` is j mod ring (bullet
  "Decode": chunks at absolute key positions over a ring cache);
* s_j = scale * sum_d q_d k_{j,d} from the exact bf16 values, m = max_j s_j,
  w_j = exp(s_j - m), o = sum_j w_j v_j / sum_j w_j, all in float64 (bullet
  "core/attention_range.zig": a head in float64, rounded only at the output).

Non-finite values follow IEEE float64 through that formula exactly as written
(bullet "A NaN or infinite output re-runs its head in float64"): a NaN score
makes m NaN, a +inf score makes s - m NaN, an infinite value with a nonzero
weight gives an infinite output, and 0 * inf gives NaN.

Every function returns float64 outputs; rounding to bf16 (round to nearest
even, an underflow keeping its sign, bullet "Includes core/bf16_round.zig")
happens only in :mod:`oracle.check`.

Pins (tests/test_oracle_pins.py): brute force over an explicitly built dense
mask through torch's float64 scaled_dot_product_attention, mpmath at 50
digits, softmax weights summing to 1, a one-key window returning its value
exactly, equal scores returning the exact mean, invisible keys having no
effect, 256-key chunking with a float64 log-sum-exp merge, and hi[i] = p0 + i
matching the null hi.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_to_f64",
    "f64_to_bf16",
    "visible_decode",
    "visible_prompt",
    "attend",
    "decode",
    "prompt",
    "prompt_sparse",
    "SPARSE_BLOCK",
]


# ---------------------------------------------------------------------------
# bf16 <-> float64 (TensorFold #1123, "What this changes", bf16_round bullet)
# ---------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16 / int16 array) as float64."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 bits, nearest-even, directly from float64.

    One rounding only (no detour through float32).  NaN becomes a quiet NaN
    with the input's sign; overflow past the largest finite bf16 goes to inf;
    an underflow to zero keeps its sign.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = (np.signbit(x).astype(np.uint32) << np.uint32(15))
    ax = np.abs(x)
    out = np.zeros(x.shape, dtype=np.uint32)
    with np.errstate(invalid="ignore", over="ignore"):
        finite = np.isfinite(ax)
        normal = finite & (ax >= 2.0 ** -126)
        sub = finite & ~normal
        # subnormal range: quantum 2^-133; 128 quanta is the least normal (bits 0x0080)
        qs = np.rint(np.where(sub, ax, 0.0) * 2.0 ** 133)
        out = np.where(sub, qs.astype(np.uint32), out)
        # normal range: 8 significant bits
        m, e = np.frexp(np.where(normal, ax, 1.0))  # ax = m * 2^e, m in [0.5, 1)
        sig = np.rint(np.ldexp(m, 8))  # in [128, 256]
        carry = sig >= 256.0
        sig = np.where(carry, 128.0, sig)
        ex = np.where(carry, e, e - 1).astype(np.int64) + 127
        nb = (np.clip(ex, 0, 255).astype(np.uint32) << np.uint32(7)) | (sig.astype(np.uint32) - np.uint32(128))
        nb = np.where(ex >= 255, np.uint32(0x7F80), nb)
        out = np.where(normal, nb, out)
        out = np.where(np.isinf(ax), np.uint32(0x7F80), out)
        out = np.where(np.isnan(x), np.uint32(0x7FC0), out)
    return (out | sign).astype(np.uint16)


# ---------------------------------------------------------------------------
# Visible key ranges (TensorFold #1123, "What this changes")
# ---------------------------------------------------------------------------

def visible_decode(p: int, win: int):
    """Inclusive key range [lo, p] of a decode row at position p."""
    lo = max(0, p - win + 1) if win > 0 else 0
    return lo, p


def visible_prompt(p0: int, i: int, win: int, hi_i=None):
    """Inclusive key range [lo_i, hi_i] of prompt row i (hi_i None: own position)."""
    p = p0 + i
    lo = max(0, p - win + 1) if win > 0 else 0
    return lo, (p if hi_i is None else int(hi_i))


# ---------------------------------------------------------------------------
# The softmax-attention definition, float64
# ---------------------------------------------------------------------------

def _dot_rows(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """a [G, d] times b [n, d]^T.  A library matmul when every input is finite;
    with a NaN or infinity present, explicit products and sums so that IEEE
    special values propagate exactly as the formula says."""
    if np.isfinite(a).all() and np.isfinite(b).all():
        return a @ b.T
    with np.errstate(invalid="ignore", over="ignore"):
        return (a[:, None, :] * b[None, :, :]).sum(axis=2)


def _weighted_sum(w: np.ndarray, v: np.ndarray) -> np.ndarray:
    """w [G, n] times v [n, d], same special-value policy as _dot_rows."""
    if np.isfinite(w).all() and np.isfinite(v).all():
        return w @ v
    with np.errstate(invalid="ignore", over="ignore"):
        return (w[:, :, None] * v[None, :, :]).sum(axis=1)


def attend(qg: np.ndarray, k_vis: np.ndarray, v_vis: np.ndarray, scale: float):
    """o = softmax(scale * q K^T) V over the visible keys, float64.

    qg [G, d], k_vis / v_vis [n, d] (float64, n >= 1).  Returns (o [G, d],
    w [G, n]) with w the unnormalised weights exp(s - m)."""
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        s = float(scale) * _dot_rows(qg, k_vis)          # s_j
        m = s.max(axis=1, keepdims=True)                 # NaN-propagating max
        w = np.exp(s - m)                                # w_j = exp(s_j - m)
        l = w.sum(axis=1, keepdims=True)                 # sum_j w_j
        o = _weighted_sum(w, v_vis) / l                  # sum_j w_j v_j / sum_j w_j
    return o, w


def _gather(ring_arr: np.ndarray, lo: int, hi: int, ring: int, g: int) -> np.ndarray:
    slots = np.arange(lo, hi + 1, dtype=np.int64) % ring
    return bf16_to_f64(ring_arr[slots, g, :])


def decode(q, k, v, pos, win: int, ring: int, scale: float, rows=None, heads=None) -> np.ndarray:
    """Decode form.  q [R,hq,d], k/v [R,ring,hkv,d] bf16 bits; pos [R].

    Row r uses its own ring k[r], v[r] (one cache per row).  Returns float64
    [len(rows), hq, d]; heads outside ``heads`` are left NaN."""
    q = np.asarray(q); k = np.asarray(k); v = np.asarray(v); pos = np.asarray(pos)
    R, hq, d = q.shape
    hkv = k.shape[2]
    G = hq // hkv
    rows = list(range(R)) if rows is None else [int(r) for r in rows]
    heads = list(range(hq)) if heads is None else [int(h) for h in heads]
    out = np.full((len(rows), hq, d), np.nan)
    for ri, r in enumerate(rows):
        lo, hi = visible_decode(int(pos[r]), win)
        for g in sorted({h // G for h in heads}):
            hs = [h for h in heads if h // G == g]
            kv_k = _gather(k[r], lo, hi, ring, g)
            kv_v = _gather(v[r], lo, hi, ring, g)
            o, _ = attend(bf16_to_f64(q[r, hs, :]), kv_k, kv_v, scale)
            out[ri, hs, :] = o
    return out


def prompt(q, k, v, p0: int, win: int, ring: int, scale: float, hi=None, rows=None, heads=None) -> np.ndarray:
    """Prompt form.  q [n,hq,d] bf16 bits (any strides), k/v [ring,hkv,d]; hi [n] or None.

    Row i sits at position p0 + i.  Rows with the same visible range share one
    gather of their keys.  Returns float64 [len(rows), hq, d]."""
    q = np.asarray(q); k = np.asarray(k); v = np.asarray(v)
    n, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    rows = list(range(n)) if rows is None else [int(r) for r in rows]
    heads = list(range(hq)) if heads is None else [int(h) for h in heads]
    out = np.full((len(rows), hq, d), np.nan)
    groups: dict = {}
    for ri, i in enumerate(rows):
        rng = visible_prompt(p0, i, win, None if hi is None else hi[i])
        groups.setdefault(rng, []).append((ri, i))
    for (lo, hi_i), members in groups.items():
        ris = [a for a, _ in members]
        idx = [b for _, b in members]
        for g in sorted({h // G for h in heads}):
            hs = [h for h in heads if h // G == g]
            kv_k = _gather(k, lo, hi_i, ring, g)
            kv_v = _gather(v, lo, hi_i, ring, g)
            qq = bf16_to_f64(q[np.ix_(idx, hs)]).reshape(len(idx) * len(hs), d)
            o, _ = attend(qq, kv_k, kv_v, scale)
            out[np.ix_(ris, hs)] = o.reshape(len(idx), len(hs), d)
    return out


# ---------------------------------------------------------------------------
# Block-sparse prompt (TensorFold pull request #1622, "What this changes")
# ---------------------------------------------------------------------------

SPARSE_BLOCK = 64   # keys per selectable block: positions [64 b, 64 b + 63]


def sparse_keys(lo: int, hi: int, sel_row) -> np.ndarray:
    """Visible keys of a row under a block selection: j in [lo, hi] whose block j // 64 is
    listed (entries < 0 are unused; repeats and order do not matter), ascending."""
    blocks = sorted({int(b) for b in np.asarray(sel_row).ravel() if int(b) >= 0})
    keys = []
    for b in blocks:
        a = max(lo, b * SPARSE_BLOCK)
        e = min(hi, b * SPARSE_BLOCK + SPARSE_BLOCK - 1)
        if a <= e:
            keys.extend(range(a, e + 1))
    return np.asarray(keys, dtype=np.int64)


def prompt_sparse(q, k, v, p0: int, win: int, ring: int, scale: float, sel, hi=None, rows=None,
                  heads=None) -> np.ndarray:
    """Block-sparse prompt: row i, query head h (key head g = h // G) attends to the keys of
    [lo_i, hi_i] that lie in the blocks sel[i, g, :] lists ("per-row block masks and causal
    ends").  q [n,hq,d], k/v [ring,hkv,d] bf16 bits, sel [n, hkv, nsel] int.

    A row with no visible key gets 0 / 0 = NaN (the empty sums of the formula).  Returns float64
    [len(rows), hq, d]."""
    q = np.asarray(q); k = np.asarray(k); v = np.asarray(v); sel = np.asarray(sel)
    n, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    rows = list(range(n)) if rows is None else [int(r) for r in rows]
    heads = list(range(hq)) if heads is None else [int(h) for h in heads]
    out = np.full((len(rows), hq, d), np.nan)
    for ri, i in enumerate(rows):
        lo, hi_i = visible_prompt(p0, i, win, None if hi is None else hi[i])
        for g in sorted({h // G for h in heads}):
            hs = [h for h in heads if h // G == g]
            keys = sparse_keys(lo, hi_i, sel[i, g])
            if keys.size == 0:
                continue   # stays NaN
            slots = keys % ring
            kv_k = bf16_to_f64(k[slots, g, :])
            kv_v = bf16_to_f64(v[slots, g, :])
            o, _ = attend(bf16_to_f64(q[i, hs, :]), kv_k, kv_v, scale)
            out[ri, hs, :] = o
    return out
