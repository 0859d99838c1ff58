"""Block-sparse prompt on the GPU against the float64 oracle (TensorFold pull request #1622,
"What this changes": per-row selected key blocks with block masks and causal ends; the
review thread's shapes: 24/2 heads at d 256 and 6/1 heads with a 17-row tail).

Tolerances follow the P mode as in the dense prompt (oracle/check.py).  Also: a row's bits do
not depend on what the other rows select or on where a chunk is cut, and with every block
selected the sparse form gives the dense form's bits where both use 64-key tiles.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import wa_synth
from _util import assert_parity, bits, ensure_built
from oracle import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def tol(p32):
    return {0: check.TOL_BF16_P, 1: check.TOL_P32, 2: check.TOL_P3}[int(p32)]


def _case(n, p0, hq, hkv, d, win, ring, seed, spans=()):
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=seed, hi_spans=spans, peak_every=5)
    for key in ("q", "k", "v"):
        c[key] = c[key].cuda()
    if c["hi"] is not None:
        c["hi"] = c["hi"].cuda()
    return c


def _random_sel(n, hkv, nsel, p0, win, seed, spill=2):
    """Random selections with repeats, unused entries and blocks outside the row's range."""
    rng = np.random.default_rng(seed)
    sel = np.full((n, hkv, nsel), -1, dtype=np.int32)
    for i in range(n):
        p = p0 + i
        lo_b = (max(0, p - win + 1) if win else 0) // 64
        for g in range(hkv):
            m = int(rng.integers(1, nsel + 1))
            sel[i, g, :m] = rng.integers(max(0, lo_b - spill), p // 64 + 1 + spill, m)
    return torch.from_numpy(sel).cuda()


def _ref(c, sel, scale=1.0, rows=None):
    hi = None if c["hi"] is None else c["hi"].cpu().numpy()
    return oracle.prompt_sparse(bits(c["q"]), bits(c["k"]), bits(c["v"]), c["p0"], c["win"], c["ring"], scale,
                                sel.cpu().numpy(), hi=hi, rows=rows)


CASES = [
    # name, n, p0, hq, hkv, d, win, ring, nsel, p32, selection, spans
    ("served_24_2_d256_p3", 300, 3000, 24, 2, 256, 0, 3300, 32, 2, "synthetic", []),
    ("tail17_6_1_d256_p3", 17, 2000, 6, 1, 256, 0, 2017, 32, 2, "synthetic", []),
    ("mha_d128_window_wrap_bf16", 260, 900, 8, 8, 128, 700, 1200, 8, 0, "random", []),
    ("mha_d128_window_wrap_p32", 260, 900, 8, 8, 128, 700, 1200, 8, 1, "random", []),
    ("gqa16_d128_nsel64_p32", 140, 5000, 16, 1, 128, 0, 5140, 64, 1, "random", []),
    ("gqa4_d256_image_span_p32", 200, 1000, 8, 2, 256, 1024, 1536, 12, 1, "random", [(20, 90)]),
    ("gqa3_d256_bf16", 129, 400, 6, 2, 256, 0, 529, 5, 0, "random", []),
    ("gqa12_d256_p3_window", 96, 7000, 12, 1, 256, 1024, 1536, 20, 2, "random", []),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_sparse_parity(wa, case):
    name, n, p0, hq, hkv, d, win, ring, nsel, p32, kind, spans = case
    c = _case(n, p0, hq, hkv, d, win, ring, seed=len(name) * 7 + n, spans=spans)
    if kind == "synthetic":
        sel = wa_synth.sparse_selection(n, p0, hkv, nsel, seed=n, win=win, device="cuda")
    else:
        sel = _random_sel(n, hkv, nsel, p0, win, seed=n + d)
    ws = torch.empty(wa.prompt_ws_bytes(n, hq), dtype=torch.uint8, device="cuda")
    out = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, c["hi"], win, 1.0, p32=p32, ws=ws)
    assert wa.status(ws) == 0
    assert_parity(out, _ref(c, sel), tol(p32), name)


def test_rows_with_no_visible_block_are_nan(wa):
    n, p0, hq, hkv, d, ring = 40, 640, 4, 2, 128, 700
    c = _case(n, p0, hq, hkv, d, 0, ring, seed=3)
    sel = _random_sel(n, hkv, 4, p0, 0, seed=4)
    sel[5:9] = -1                        # nothing selected
    sel[12, 1] = 20                      # a block past every row: nothing visible for key head 1
    out = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, 0, 1.0, p32=1)
    ref = _ref(c, sel)
    assert np.isnan(ref[5:9]).all() and np.isnan(ref[12, 2:]).all()
    assert_parity(out, ref, check.TOL_P32, "empty rows")


def test_cta_with_no_visible_block_at_all(wa):
    n, p0, hq, hkv, d, ring = 20, 300, 4, 1, 256, 320
    c = _case(n, p0, hq, hkv, d, 0, ring, seed=5)
    sel = torch.full((n, hkv, 3), -1, dtype=torch.int32, device="cuda")
    out = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, 0, 1.0, p32=2)
    assert torch.isnan(out.float()).all()


def test_scale_sign_and_zero(wa):
    n, p0, hq, hkv, d, ring = 100, 700, 8, 2, 256, 800
    c = _case(n, p0, hq, hkv, d, 0, ring, seed=6)
    sel = _random_sel(n, hkv, 6, p0, 0, seed=7)
    for scale in (-0.5, 0.0, 0.11):
        out = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, 0, scale, p32=1)
        assert_parity(out, _ref(c, sel, scale=scale), check.TOL_P32, f"scale {scale}")


def test_other_rows_selections_do_not_change_a_rows_bits(wa):
    n, p0, hq, hkv, d, ring = 256, 2000, 8, 2, 256, 2256
    c = _case(n, p0, hq, hkv, d, 0, ring, seed=8)
    sel = _random_sel(n, hkv, 10, p0, 0, seed=9)
    base = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, 0, 1.0, p32=2)
    other = _random_sel(n, hkv, 10, p0, 0, seed=10)
    keep = torch.arange(n, device="cuda") % 3 == 0
    mixed = torch.where(keep[:, None, None], sel, other)
    out = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, mixed, None, 0, 1.0, p32=2)
    assert torch.equal(out[keep].view(torch.int16), base[keep].view(torch.int16))


def test_chunk_split_gives_every_rows_bits(wa):
    n, p0, hq, hkv, d, ring = 300, 3000, 24, 2, 256, 3300
    c = _case(n, p0, hq, hkv, d, 0, ring, seed=11)
    sel = wa_synth.sparse_selection(n, p0, hkv, 32, seed=12, device="cuda")
    whole = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, 0, 1.0, p32=2)
    for cut in (1, 5, 150, 299):
        a = wa.prompt_sparse(c["q"][:cut], c["k"], c["v"], p0, sel[:cut].contiguous(), None, 0, 1.0, p32=2)
        b = wa.prompt_sparse(c["q"][cut:], c["k"], c["v"], p0 + cut, sel[cut:].contiguous(), None, 0, 1.0, p32=2)
        assert torch.equal(torch.cat([a, b]).view(torch.int16), whole.view(torch.int16)), cut


@pytest.mark.parametrize("d,p32", [(256, 0), (256, 1), (256, 2), (128, 2)])
def test_every_block_selected_gives_the_dense_result(wa, d, p32):
    """With three P parts both forms run the same 64-key tiles in key order for every row, so the
    bits agree; with one or two parts the dense form at head dim 256 runs 128-key tiles (another
    fp32 summation order), so both are held to the oracle instead."""
    n, p0, hq, hkv, win, ring = 200, 1500, 8, 2, 1024, 1536
    c = _case(n, p0, hq, hkv, d, win, ring, seed=13)
    nb = (p0 + n - 1) // 64 + 1
    sel = torch.arange(nb, dtype=torch.int32, device="cuda").repeat(n, hkv, 1)[:, :, -64:].contiguous()
    lo_b = max(0, p0 - win + 1) // 64
    assert nb - lo_b <= 64
    sparse = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, win, 1.0, p32=p32)
    dense = wa.prompt(c["q"], c["k"], c["v"], p0, None, win, 1.0, p32=p32)
    if p32 == 2:
        assert torch.equal(sparse.view(torch.int16), dense.view(torch.int16))
    else:
        ref = oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), p0, win, ring, 1.0)
        tol = check.TOL_P32 if p32 else check.TOL_BF16_P
        assert_parity(sparse, ref, tol, "sparse, every block")
        assert_parity(dense, ref, tol, "dense")


def test_served_size_sampled(wa):
    """7,936 rows (the pages' 7.9K-token prompt), 24/2 heads, d 256, 2,048 selected keys a row."""
    n, hq, hkv, d = 7936, 24, 2, 256
    c = _case(n, 0, hq, hkv, d, 0, n, seed=14)
    sel = wa_synth.sparse_selection(n, 0, hkv, 32, seed=15, device="cuda")
    out = wa.prompt_sparse(c["q"], c["k"], c["v"], 0, sel, None, 0, 1.0, p32=2)
    rows = [0, 63, 64, 2047, 4000, 7935]
    assert_parity(out[rows], _ref(c, sel, rows=rows), check.TOL_P3, "served size")
    assert torch.isfinite(out.float()).all()
