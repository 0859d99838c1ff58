"""Pins of the block-sparse prompt oracle (CPU): brute force through an explicit dense mask
and torch's float64 SDPA, the dense oracle when every block is selected, set semantics of
the selection, unselected blocks having no effect, the empty case, and a planted off-by-one
block map that the brute force catches.  TensorFold pull request #1622, "What this changes"
(per-row block masks and causal ends)."""
from __future__ import annotations

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import wa_synth
from test_oracle_pins import bits, tval

B = oracle.SPARSE_BLOCK


def brute_sparse(q, k, v, p0, win, ring, scale, sel, hi=None, block_of=lambda j: j // B):
    qt, kt, vt = tval(q), tval(k), tval(v)
    n, hq, d = qt.shape
    hkv = kt.shape[1]
    last = p0 + n
    out = torch.full((n, hq, d), float("nan"), dtype=torch.float64)
    for i in range(n):
        P = p0 + i
        H = P if hi is None else int(hi[i])
        for g in range(hkv):
            chosen = {int(b) for b in sel[i, g] if b >= 0}
            mask = torch.zeros(last, dtype=torch.bool)
            kabs = torch.zeros(last, d, dtype=torch.float64)
            vabs = torch.zeros(last, d, dtype=torch.float64)
            for j in range(last):
                if j <= H and (win == 0 or j >= P - win + 1) and block_of(j) in chosen:
                    mask[j] = True
                    kabs[j] = kt[j % ring, g]
                    vabs[j] = vt[j % ring, g]
            if not mask.any():
                continue
            for h in range(g * (hq // hkv), (g + 1) * (hq // hkv)):
                out[i, h] = F.scaled_dot_product_attention(
                    qt[i, h].view(1, 1, 1, d), kabs.view(1, 1, -1, d), vabs.view(1, 1, -1, d),
                    attn_mask=mask.view(1, 1, 1, -1), scale=scale).view(d)
    return out.numpy()


def _case(n, p0, hq, hkv, d, win, ring, seed):
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=seed, peak_every=3)
    return bits(c["q"]), bits(c["k"]), bits(c["v"])


def _random_sel(rng, n, hkv, nsel, p0, win):
    sel = np.full((n, hkv, nsel), -1, dtype=np.int64)
    for i in range(n):
        p = p0 + i
        lo_b = (max(0, p - win + 1) if win else 0) // B
        for g in range(hkv):
            m = rng.integers(1, nsel + 1)
            sel[i, g, :m] = rng.integers(max(0, lo_b - 1), p // B + 2, m)   # some outside the range
    return sel


@pytest.mark.parametrize("case", [
    # n, p0, hq, hkv, d, win, ring, nsel
    (6, 250, 4, 2, 4, 0, 256, 3),
    (5, 300, 2, 1, 8, 150, 200, 2),     # window, ring wrap
    (4, 640, 8, 2, 4, 0, 700, 5),
])
def test_sparse_matches_brute_force(case):
    n, p0, hq, hkv, d, win, ring, nsel = case
    q, k, v = _case(n, p0, hq, hkv, d, win, ring, seed=3 + n)
    sel = _random_sel(np.random.default_rng(n), n, hkv, nsel, p0, win)
    got = oracle.prompt_sparse(q, k, v, p0, win, ring, 0.8, sel)
    want = brute_sparse(q, k, v, p0, win, ring, 0.8, sel)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    np.testing.assert_allclose(got[~np.isnan(got)], want[~np.isnan(want)], rtol=1e-12, atol=1e-13)


def test_all_blocks_selected_is_the_dense_prompt():
    n, p0, hq, hkv, d, win, ring = 8, 200, 4, 2, 8, 100, 300
    q, k, v = _case(n, p0, hq, hkv, d, win, ring, seed=9)
    nb = (p0 + n) // B + 1
    sel = np.tile(np.arange(nb), (n, hkv, 1))
    np.testing.assert_allclose(oracle.prompt_sparse(q, k, v, p0, win, ring, 1.0, sel),
                               oracle.prompt(q, k, v, p0, win, ring, 1.0), rtol=1e-13, atol=1e-14)


def test_selection_is_a_set():
    n, p0, hq, hkv, d, ring = 5, 300, 2, 1, 4, 320
    q, k, v = _case(n, p0, hq, hkv, d, 0, ring, seed=10)
    sel = np.array([[[0, 4, 2, -1]]] * n)
    base = oracle.prompt_sparse(q, k, v, p0, 0, ring, 1.0, sel)
    shuffled = np.array([[[2, -1, 4, 0, 4, 2, -1]]] * n)
    assert np.array_equal(oracle.prompt_sparse(q, k, v, p0, 0, ring, 1.0, shuffled), base)


def test_unselected_blocks_have_no_effect_and_empty_is_nan():
    n, p0, hq, hkv, d, ring = 4, 260, 2, 1, 8, 270
    q, k, v = _case(n, p0, hq, hkv, d, 0, ring, seed=11)
    sel = np.array([[[1, 4]]] * n)
    base = oracle.prompt_sparse(q, k, v, p0, 0, ring, 1.0, sel)
    k2, v2 = k.copy(), v.copy()
    for b in (0, 2, 3):                       # blocks nobody selected
        k2[b * B:(b + 1) * B] = 0x7FC0         # NaN
        v2[b * B:(b + 1) * B] = 0x7F80         # +inf
    assert np.array_equal(oracle.prompt_sparse(q, k2, v2, p0, 0, ring, 1.0, sel), base)
    empty = oracle.prompt_sparse(q, k, v, p0, 0, ring, 1.0, np.array([[[7, -1]]] * n))   # block 7 lies past every row
    assert np.isnan(empty).all()


def test_planted_block_map_off_by_one_is_caught():
    n, p0, hq, hkv, d, ring = 5, 250, 2, 1, 4, 256
    q, k, v = _case(n, p0, hq, hkv, d, 0, ring, seed=12)
    sel = np.array([[[1, 3]]] * n)
    want = brute_sparse(q, k, v, p0, 0, ring, 1.0, sel)
    planted = brute_sparse(q, k, v, p0, 0, ring, 1.0, sel, block_of=lambda j: (j + 1) // B)
    assert not np.allclose(planted, want)
    np.testing.assert_allclose(oracle.prompt_sparse(q, k, v, p0, 0, ring, 1.0, sel), want, rtol=1e-12)


def test_synthetic_selection_shape_and_ranges():
    sel = wa_synth.sparse_selection(300, 3000, 2, 32, seed=1).numpy()
    assert sel.shape == (300, 2, 32)
    for i in range(300):
        p = 3000 + i
        for g in range(2):
            s = sel[i, g][sel[i, g] >= 0]
            assert len(set(s.tolist())) == len(s) == 32
            assert s.max() <= p // B and s.min() >= 0
            assert p // B in s and p // B - 1 in s and 0 in s
    early = wa_synth.sparse_selection(10, 0, 1, 32, seed=1).numpy()
    assert (early[:, 0, 0] == 0).all()
