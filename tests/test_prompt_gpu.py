"""Prompt form on the GPU against the float64 oracle, element by element.

Tolerances (interval rule, see oracle/check.py): 3e-3 with the two-half P
(P32), 8e-3 with a single bf16 P.  Cases follow TensorFold pull request #1123:
"Receipt" (512-row chunks at p0 0 / 1,300 with an image span of rows 40-300 /
5,000 where the ring wraps, 333 rows with bf16 P, a no-window prompt; a chunk
split in two gives every row's bits; the gate 1 plants) and the review thread
(a finite row next to a NaN row, alone, beside it and split across chunks, with
bf16 P and P32; ratios 8 and 16).  The dense d=128 case follows the "Exact
Numerical Contract" page, "Canonical Boundary".
"""
from __future__ import annotations

import zlib

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
    if p32 == 2:
        return check.TOL_P3
    return check.TOL_P32 if p32 else check.TOL_BF16_P


def _case(n, p0, hq, hkv, d, win, ring, seed, spans=(), outside="nan", peak_every=8):
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=seed, hi_spans=spans, outside=outside,
                             peak_every=peak_every)
    for key in ("q", "k", "v"):
        c[key] = c[key].cuda()
    if c["hi"] is not None:
        c["hi"] = c["hi"].cuda()
    return c


def _ref(c, scale=1.0, rows=None):
    hi = None if c["hi"] is None else c["hi"].cpu().numpy()
    return oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), c["p0"], c["win"], c["ring"], scale, hi=hi,
                         rows=rows)


CASES = [
    # name, n, p0, hq, hkv, d, win, ring, spans, p32
    ("chunk512_p1300_image_p32", 512, 1300, 16, 8, 256, 1024, 1536, [(40, 300)], True),
    ("chunk512_p1300_image_bf16", 512, 1300, 16, 8, 256, 1024, 1536, [(40, 300)], False),
    ("wrap333_p5000_bf16", 333, 5000, 32, 16, 256, 1024, 1536, [], False),
    ("chunk512_p0_p32", 512, 0, 16, 8, 256, 1024, 1536, [], True),
    ("linear_causal_700_p32", 700, 0, 16, 8, 256, 0, 700, [], True),
    ("one_row", 1, 77, 4, 2, 256, 16, 64, [], True),
    ("ring1000_wrapcopy_d256", 300, 2000, 8, 4, 256, 500, 1000, [(10, 60)], True),
    ("ring1000_wrapcopy_d128", 300, 2000, 8, 4, 128, 500, 1000, [(250, 299)], False),
    ("d128_sliding_mha", 260, 900, 4, 4, 128, 700, 1200, [], False),
    ("d128_gqa8_p32", 200, 300, 16, 2, 128, 256, 512, [(0, 199)], True),
    ("d256_gqa16_bf16", 150, 100, 16, 1, 256, 128, 256, [], False),
    ("d256_gqa3", 129, 4000, 6, 2, 256, 1024, 1536, [(120, 128)], True),
    ("window_1", 130, 40, 2, 1, 128, 1, 256, [], True),
    # head dim 128 with P32 (two query tiles a CTA): causal, ring-wrap copies, image spans, and a
    # call whose one pair of tiles has no second tile
    ("d128_linear_causal_700_p32", 700, 0, 8, 4, 128, 0, 700, [], True),
    ("d128_wrapcopy_p32", 300, 2000, 8, 4, 128, 500, 1000, [(10, 60)], True),
    ("d128_chunk512_p1300_image_p32", 512, 1300, 16, 8, 128, 1024, 1536, [(40, 300)], True),
    ("d128_one_tile_n100_p32", 100, 3000, 4, 2, 128, 1024, 1536, [], True),
    ("d128_one_tile_n100_bf16", 100, 3000, 4, 2, 128, 1024, 1536, [], False),
    ("linear_causal_700_bf16", 700, 0, 16, 8, 256, 0, 700, [], False),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prompt_parity(wa, case):
    name, n, p0, hq, hkv, d, win, ring, spans, p32 = case
    c = _case(n, p0, hq, hkv, d, win, ring, seed=zlib.crc32(name.encode()) % 100000, spans=spans)
    ws = torch.empty(wa.prompt_ws_bytes(n, hq), dtype=torch.uint8, device="cuda")
    out = wa.prompt(c["q"], c["k"], c["v"], p0, c["hi"], win, 1.0, p32=p32, ws=ws)
    assert wa.status(ws) == 0
    r = assert_parity(out, _ref(c), tol(p32), name)
    assert r["n_nonfinite_ref"] == 0


P3_CASES = [c[:-1] + (2,) for c in CASES if c[0] in (
    "chunk512_p1300_image_p32", "wrap333_p5000_bf16", "linear_causal_700_p32", "ring1000_wrapcopy_d128",
    "d128_sliding_mha", "d128_gqa8_p32", "d256_gqa3", "window_1", "one_row")]


@pytest.mark.parametrize("case", P3_CASES, ids=[c[0] + "_as_p3" for c in P3_CASES])
def test_prompt_parity_three_part_p(wa, case):
    """P as hi + mid + lo: every output within [RN(o - 1e-5), RN(o + 1e-5)]."""
    name, n, p0, hq, hkv, d, win, ring, spans, p32 = case
    c = _case(n, p0, hq, hkv, d, win, ring, seed=zlib.crc32(name.encode()) % 100000, spans=spans)
    ws = torch.empty(wa.prompt_ws_bytes(n, hq), dtype=torch.uint8, device="cuda")
    out = wa.prompt(c["q"], c["k"], c["v"], p0, c["hi"], win, 1.0, p32=2, ws=ws)
    assert wa.status(ws) == 0
    assert_parity(out, _ref(c), check.TOL_P3, name + " as p3")


@pytest.mark.parametrize("d", [128, 256])
def test_three_part_p_is_closer_to_float64_than_two_part(wa, d):
    """Outputs that differ from RN(o): fewer with three parts than with two, and under 0.5 %."""
    c = _case(700, 0, 16, 8, d, 0, 700, seed=17, outside="keep", peak_every=64)
    ref = _ref(c)
    rn = oracle.f64_to_bf16(ref)
    miss = {}
    for p32 in (1, 2):
        out = wa.prompt(c["q"], c["k"], c["v"], 0, None, 0, 1.0, p32=p32)
        miss[p32] = int((bits(out) != rn.reshape(bits(out).shape)).sum())
    assert miss[2] < miss[1], miss
    assert miss[2] < 0.005 * rn.size, miss


def test_three_part_p_long_rows_sampled(wa):
    """Causal 8,192 rows at d 256 and dense 4,096 rows at d 128: sampled rows within 1e-5."""
    c = _case(8192, 0, 16, 8, 256, 0, 8192, seed=18, outside="keep")
    out = wa.prompt(c["q"], c["k"], c["v"], 0, None, 0, 1.0, p32=2)
    rows = [0, 1, 4095, 8190, 8191]
    assert_parity(out[rows], _ref(c, rows=rows), check.TOL_P3, "causal 8192 p3")
    dc = wa_synth.dense_qkv_case(4096, 8, 128, seed=19, device="cuda")
    hi = torch.full((4096,), 4095, dtype=torch.int32, device="cuda")
    out = wa.prompt(dc["q"], dc["k"], dc["v"], 0, hi, 0, dc["scale"], p32=2)
    rows = [0, 2048, 4095]
    ref = oracle.prompt(bits(dc["q"]), bits(dc["k"]), bits(dc["v"]), 0, 0, 4096, dc["scale"],
                        hi=np.full(4096, 4095), rows=rows)
    assert_parity(out[rows], ref, check.TOL_P3, "dense 4096 p3")


def test_three_part_p_chunk_split_gives_every_rows_bits(wa):
    n, p0 = 512, 1300
    c = _case(n, p0, 16, 8, 128, 1024, 1536, seed=20, spans=[(40, 300)], outside="keep")
    whole = wa.prompt(c["q"], c["k"], c["v"], p0, c["hi"], 1024, 1.0, p32=2)
    for cut in (1, 301, 384):
        a = wa.prompt(c["q"][:cut], c["k"], c["v"], p0, c["hi"][:cut].contiguous(), 1024, 1.0, p32=2)
        b = wa.prompt(c["q"][cut:], c["k"], c["v"], p0 + cut, c["hi"][cut:].contiguous(), 1024, 1.0, p32=2)
        assert torch.equal(torch.cat([a, b]).view(torch.int16), whole.view(torch.int16)), cut


@pytest.mark.parametrize("scale", [0.37, -0.5, 0.0])
@pytest.mark.parametrize("d", [128, 256])
def test_prompt_scale_parameter(wa, scale, d):
    c = _case(200, 500, 8, 4, d, 300, 600, seed=5)
    out = wa.prompt(c["q"], c["k"], c["v"], 500, None, 300, scale, p32=True)
    assert_parity(out, _ref(c, scale=scale), check.TOL_P32, f"scale {scale}")


def test_chunk_split_gives_every_rows_bits(wa):
    for p32 in (False, True):
        n, p0 = 512, 1300
        c = _case(n, p0, 16, 8, 256, 1024, 1536, seed=11, spans=[(40, 300)], outside="keep")
        whole = wa.prompt(c["q"], c["k"], c["v"], p0, c["hi"], 1024, 1.0, p32=p32)
        for cut in (1, 37, 301, 384, 511):   # cuts outside the image span (hi < p0 + n)
            a = wa.prompt(c["q"][:cut], c["k"], c["v"], p0, c["hi"][:cut].contiguous(), 1024, 1.0, p32=p32)
            b = wa.prompt(c["q"][cut:], c["k"], c["v"], p0 + cut, c["hi"][cut:].contiguous(), 1024, 1.0, p32=p32)
            both = torch.cat([a, b])
            assert torch.equal(both.view(torch.int16), whole.view(torch.int16)), (p32, cut)


@pytest.mark.parametrize("p32", [False, True])
def test_chunk_split_gives_every_rows_bits_d128(wa, p32):
    """Head dim 128 (two 128-row query tiles a CTA): cuts on and off the 128- and 256-row tile
    edges, with a window over a wrapping ring, give every row the bits of the whole chunk."""
    n, p0, win, ring = 600, 1300, 700, 1400
    c = _case(n, p0, 16, 8, 128, win, ring, seed=31, spans=[(500, 560)], outside="keep")
    whole = wa.prompt(c["q"], c["k"], c["v"], p0, c["hi"], win, 1.0, p32=p32)
    for cut in (1, 128, 255, 256, 301, 384, 499, 599):   # outside the image span (hi < p0 + cut)
        a = wa.prompt(c["q"][:cut], c["k"], c["v"], p0, c["hi"][:cut].contiguous(), win, 1.0, p32=p32)
        b = wa.prompt(c["q"][cut:], c["k"], c["v"], p0 + cut, c["hi"][cut:].contiguous(), win, 1.0, p32=p32)
        both = torch.cat([a, b])
        assert torch.equal(both.view(torch.int16), whole.view(torch.int16)), (p32, cut)


def test_other_rows_do_not_change_a_rows_bits_d128(wa):
    """A row's bits at head dim 128 depend on its own q and the keys it sees only: changing the
    q of every other row (the tile that shares its CTA included) leaves them unchanged."""
    n, p0 = 512, 0
    c = _case(n, p0, 8, 2, 128, 0, 512, seed=32, outside="keep")
    base = wa.prompt(c["q"], c["k"], c["v"], p0, None, 0, 1.0, p32=False)
    keep = torch.arange(n, device="cuda") % 5 == 0
    q2 = torch.where(keep[:, None, None], c["q"], -2 * c["q"])
    out = wa.prompt(q2, c["k"], c["v"], p0, None, 0, 1.0, p32=False)
    assert torch.equal(out[keep].view(torch.int16), base[keep].view(torch.int16))


def test_linear_cache_declared_16x_longer_gives_same_bits(wa):
    c = _case(300, 0, 8, 4, 128, 0, 300, seed=12, outside="keep")
    a = wa.prompt(c["q"], c["k"], c["v"], 0, None, 0, 1.0, p32=True)
    k16 = torch.zeros((4800, 4, 128), dtype=torch.bfloat16, device="cuda")
    v16 = torch.zeros_like(k16)
    k16[:300] = c["k"]
    v16[:300] = c["v"]
    b = wa.prompt(c["q"], k16, v16, 0, None, 0, 1.0, p32=True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_repeats_are_byte_identical(wa):
    c = _case(333, 5000, 32, 16, 256, 1024, 1536, seed=13, outside="keep")
    first = wa.prompt(c["q"], c["k"], c["v"], 5000, None, 1024, 1.0, p32=False)
    for _ in range(4):
        again = wa.prompt(c["q"], c["k"], c["v"], 5000, None, 1024, 1.0, p32=False)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


def test_bad_hi_is_clamped_and_reported(wa):
    c = _case(64, 100, 4, 2, 128, 0, 200, seed=14, outside="keep")
    hi = torch.arange(100, 164, dtype=torch.int32, device="cuda")
    hi[3] = 50          # before its own position
    ws = torch.empty(wa.prompt_ws_bytes(64, 4), dtype=torch.uint8, device="cuda")
    wa.prompt(c["q"], c["k"], c["v"], 100, hi, 0, 1.0, ws=ws)
    assert wa.status(ws) & wa.WA_STATUS_BAD_HI
    wa.prompt(c["q"], c["k"], c["v"], 100, None, 0, 1.0, ws=ws)
    assert wa.status(ws) == 0


# --------------------------- special values ---------------------------

def _plain(n=160, p0=40, hq=4, hkv=2, d=128, win=0, ring=200):
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=21, outside="keep", peaked=False)
    return bits(c["q"]).copy(), bits(c["k"]).copy(), bits(c["v"]).copy()


def _to_dev(x):
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("p32", [False, True])
@pytest.mark.parametrize("plant", ["nan_query", "nan_key", "inf_value_later_rows", "pm_inf_column",
                                   "inf_at_tiny_weight"])
def test_nonfinite_classes_match_float64(wa, plant, p32):
    q, k, v = _plain()
    p0 = 40
    if plant == "nan_query":
        q[17, 1, 3] = 0x7FC0
    elif plant == "nan_key":
        k[p0 + 90, 0, 5] = 0x7FC0           # rows 90.. of key head 0 see it
    elif plant == "inf_value_later_rows":
        v[p0 + 120, 1, 7] = 0x7F80          # only rows >= 120 see it
    elif plant == "pm_inf_column":
        v[p0 + 10, 0, 2] = 0x7F80
        v[p0 + 30, 0, 2] = 0xFF80
    elif plant == "inf_at_tiny_weight":
        row = 100
        qv = oracle.bf16_to_f64(q[row, 0])
        k[p0 + 95, 0] = oracle.f64_to_bf16(qv * (200.0 / float(qv @ qv)))
        v[p0 + 20, 0, 9] = 0x7F80
    ref = oracle.prompt(q, k, v, p0, 0, 200, 1.0)
    out = wa.prompt(_to_dev(q), _to_dev(k), _to_dev(v), p0, None, 0, 1.0, p32=p32)
    r = assert_parity(out, ref, tol(p32), plant)
    assert r["n_nonfinite_ref"] > 0


@pytest.mark.parametrize("p32", [False, True])
def test_finite_row_next_to_a_nan_row(wa, p32):
    """The review thread's device test: a finite row alone, beside a NaN row, and split across chunks."""
    q, k, v = _plain(n=128, p0=0, ring=128)
    nan_row, row = 64, 65
    q2 = q.copy()
    q2[nan_row, :, 0] = 0x7FC0
    kd, vd = _to_dev(k), _to_dev(v)
    beside = wa.prompt(_to_dev(q2), kd, vd, 0, None, 0, 1.0, p32=p32)
    alone = wa.prompt(_to_dev(q[row:row + 1].copy()), kd, vd, row, None, 0, 1.0, p32=p32)
    split = wa.prompt(_to_dev(q2[row:].copy()), kd, vd, row, None, 0, 1.0, p32=p32)
    assert torch.isnan(beside[nan_row].float()).all()
    assert torch.isfinite(beside[row].float()).all()
    assert torch.equal(beside[row].view(torch.int16), alone[0].view(torch.int16))
    assert torch.equal(beside[row].view(torch.int16), split[0].view(torch.int16))


# --------------------------- full sizes, sampled ---------------------------

def test_causal_8192_p32_sampled(wa):
    """8,192 rows at p0 0 over a linear cache, 16/8 heads, d 256, causal, P32."""
    c = wa_synth.prompt_case(8192, 0, 16, 8, 256, 0, 8192, seed=20260005, device="cuda", outside="keep")
    out = wa.prompt(c["q"], c["k"], c["v"], 0, None, 0, 1.0, p32=True)
    torch.cuda.synchronize()
    rows = [0, 1, 127, 128, 129, 4095, 4096, 6000, 8190, 8191]
    assert_parity(out[rows], _ref(c, rows=rows), check.TOL_P32, "causal 8192")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("p32", [False, True])
def test_dense_37810_sampled(wa, p32):
    """N=37,810, 56 heads, d 128, interleaved QKV (row 21,504), RMSNormed Q/K, non-causal, 256 rows per head."""
    N, H, d = 37810, 56, 128
    c = wa_synth.dense_qkv_case(N, H, d, seed=20260006, device="cuda")
    hi = torch.full((N,), N - 1, dtype=torch.int32, device="cuda")
    out = wa.prompt(c["q"], c["k"], c["v"], 0, hi, 0, c["scale"], p32=p32)
    torch.cuda.synchronize()
    gen = np.random.default_rng(20260006)
    rows = sorted(set([0, N - 1, 37760, 37759] + gen.choice(N, 252, replace=False).tolist()))
    ref = oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), 0, 0, N, c["scale"], hi=hi.cpu().numpy(),
                        rows=rows)
    assert_parity(out[rows], ref, tol(p32), "dense 37810")
    assert torch.isfinite(out.float()).all()
