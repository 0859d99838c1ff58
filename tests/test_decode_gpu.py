"""Decode form on the GPU against the float64 oracle, element by element.

Tolerance (fp32 probabilities): a bf16 output must lie in
[RN(o - 3e-3), RN(o + 3e-3)] around the float64 value o; NaN matches NaN and
infinities match by bits.  Cases follow TensorFold pull request #1123,
sections "Receipt" (rows 1, 3, 17, 64; positions to 40,000; wrapped rings;
a no-window decode; the gate 1 plants) and the review thread (query-to-key
head ratios 8 and 16).
"""
from __future__ import annotations

import zlib

import numpy as np
import pytest
import torch

import oracle
import wa_synth
from _util import assert_parity, bits, decode_ref, ensure_built
from oracle import check

pytestmark = pytest.mark.gpu

TOL = check.TOL_FP32_P


@pytest.fixture(scope="module")
def wa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _case(rows, hq, hkv, d, win, ring, pos, seed, outside="nan", device="cuda"):
    c = wa_synth.decode_case(rows, hq, hkv, d, win, ring, pos, seed=seed, outside=outside)
    for key in ("q", "k", "v", "pos"):
        c[key] = c[key].to(device)
    return c


CASES = [
    # name, rows, hq, hkv, d, win, ring, pos
    ("tiny_16_8_d256", 3, 16, 8, 256, 1024, 1536, [900, 1700, 2047]),
    ("ragged_ring1000", 4, 8, 4, 256, 700, 1000, [0, 255, 256, 5000]),
    ("linear_d128", 3, 8, 8, 128, 0, 2000, [0, 1023, 1999]),
    ("mha_d128_ring333", 2, 4, 4, 128, 300, 333, [299, 1234]),
    ("gqa3_d256", 2, 12, 4, 256, 517, 600, [516, 9999]),
    ("gqa8_d128", 2, 16, 2, 128, 1024, 1536, [40000, 777]),
    ("gqa16_d256", 2, 16, 1, 256, 1024, 1536, [3000, 1025]),
    ("gqa16_d128", 17, 32, 2, 128, 1024, 1536, list(range(100, 40000, 2350))[:17]),
    ("one_key_window", 2, 4, 2, 256, 1, 4, [0, 17]),
    ("chunk_edges", 6, 4, 2, 256, 513, 1024, [255, 256, 511, 512, 767, 768]),
    # groups of 3 and more run on the tensor cores
    ("gqa4_ring1000_wrap", 4, 16, 4, 256, 700, 1000, [0, 255, 256, 5000]),
    ("gqa8_linear_d256", 3, 16, 2, 256, 0, 2000, [0, 1023, 1999]),
    ("gqa4_d128_chunk_edges", 6, 8, 2, 128, 513, 1024, [255, 256, 511, 512, 767, 768]),
    ("gqa16_one_key_window", 2, 16, 1, 256, 1, 4, [0, 17]),
    ("gqa8_d128_ring333", 2, 8, 1, 128, 300, 333, [299, 1234]),
    ("gqa5_d256", 3, 10, 2, 256, 1024, 1536, [1536, 77, 30000]),
    ("gqa16_d128_many_units", 40, 32, 2, 128, 1024, 1100, list(range(3, 40000, 997))[:40]),
    # linear caches of 16 chunks or more: units taken from the shared counter, longest first
    ("gqa8_linear_d128_20_chunks", 5, 16, 2, 128, 0, 5000, [0, 255, 256, 4999, 3000]),
    ("gqa4_linear_d256_17_chunks", 24, 16, 4, 256, 0, 4100, [0, 1, 255, 256, 257, 511, 512, 4095, 4096, 4099]
     + list(range(37, 4100, 293))[:14]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_parity(wa, case):
    _, rows, hq, hkv, d, win, ring, pos = case
    c = _case(rows, hq, hkv, d, win, ring, pos, seed=zlib.crc32(case[0].encode()) % 10000)
    ws = torch.empty(wa.decode_ws_bytes(rows, hq, d, win, ring), dtype=torch.uint8, device="cuda")
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0, ws=ws)
    assert wa.status(ws) == 0
    r = assert_parity(out, decode_ref(c), TOL, case[0])
    assert r["n_nonfinite_ref"] == 0


@pytest.mark.parametrize("hkv", [8, 2])
@pytest.mark.parametrize("scale", [0.0625, -0.5, 0.0])
def test_decode_scale_parameter(wa, scale, hkv):
    c = _case(3, 16, hkv, 256, 1024, 1536, [900, 1700, 2047], seed=3)
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, scale)
    assert_parity(out, decode_ref(c, scale=scale), TOL, f"scale {scale}")


@pytest.mark.parametrize("hkv", [8, 2, 1])
def test_batch_composition_and_slot_do_not_change_bits(wa, hkv):
    pos = [40000, 5, 1023, 1024, 7777]
    c = _case(5, 16, hkv, 256, 1024, 1536, pos, seed=8)
    full = wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, 1.0)
    for order in ([4, 3, 2, 1, 0], [2], [0, 4], [1, 3]):
        sel = torch.tensor(order, device="cuda")
        part = wa.decode(c["q"][sel].contiguous(), c["k"][sel].contiguous(), c["v"][sel].contiguous(),
                         c["pos"][sel].contiguous(), 1024, 1.0)
        assert torch.equal(part.view(torch.int16), full[sel].view(torch.int16)), order


@pytest.mark.parametrize("hq", [8, 32])
def test_linear_cache_declared_16x_longer_gives_same_bits(wa, hq):
    pos = [0, 700, 1999]
    c = _case(3, hq, 4, 128, 0, 2000, pos, seed=9)
    a = wa.decode(c["q"], c["k"], c["v"], c["pos"], 0, 1.0)
    k16 = torch.zeros((3, 32000, 4, 128), dtype=torch.bfloat16, device="cuda")
    v16 = torch.zeros_like(k16)
    k16[:, :2000] = c["k"]
    v16[:, :2000] = c["v"]
    b = wa.decode(c["q"], k16, v16, c["pos"], 0, 1.0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_repeats_are_byte_identical(wa):
    c = _case(4, 32, 16, 256, 1024, 1536, [1500, 20000, 2, 39999], seed=10)
    first = wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, 1.0)
    for _ in range(4):
        again = wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, 1.0)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


# --------------------------- special values (gate 1 plants) ---------------------------

def _nonfinite_case(mutate, hq=4):
    c = wa_synth.decode_case(3, hq, 2, 256, 600, 1024, [700, 1500, 599], seed=12, outside="keep")
    q, k, v = bits(c["q"]).copy(), bits(c["k"]).copy(), bits(c["v"]).copy()
    mutate(q, k, v)
    dev = {n: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for n, x in (("q", q), ("k", k), ("v", v))}
    pos = torch.tensor([700, 1500, 599], dtype=torch.int32, device="cuda")
    ref = oracle.decode(q, k, v, [700, 1500, 599], 600, 1024, 1.0)
    return dev, pos, ref


@pytest.mark.parametrize("hq", [4, 16])
@pytest.mark.parametrize("plant", ["nan_query", "nan_key", "inf_value", "pm_inf_column", "inf_at_tiny_weight"])
def test_nonfinite_classes_match_float64(wa, plant, hq):
    def mutate(q, k, v):
        if plant == "nan_query":
            q[1, 3, 7] = 0x7FC0
        elif plant == "nan_key":
            k[0, 650 % 1024, 1, 5] = 0x7FC0                  # visible to row 0 only
        elif plant == "inf_value":
            v[1, 1400 % 1024, 0, 9] = 0x7F80
        elif plant == "pm_inf_column":
            v[2, 10, 1, 3] = 0x7F80
            v[2, 400, 1, 3] = 0xFF80
        elif plant == "inf_at_tiny_weight":
            # row 0, key head 0: one key scores about 200 above every other key
            qv = oracle.bf16_to_f64(q[0, 0])
            big = oracle.f64_to_bf16(qv * (200.0 / float(qv @ qv)))
            k[0, 690 % 1024, 0] = big
            v[0, 300 % 1024, 0, 11] = 0x7F80                 # weight near e^-200 in float64, 0 in fp32
    dev, pos, ref = _nonfinite_case(mutate, hq)
    out = wa.decode(dev["q"], dev["k"], dev["v"], pos, 600, 1.0)
    r = assert_parity(out, ref, TOL, plant)
    assert r["n_nonfinite_ref"] > 0


@pytest.mark.parametrize("hkv", [8, 2])
def test_batch_composition_does_not_change_bits_linear_many_chunks(wa, hkv):
    pos = [4999, 0, 1300, 256, 4095, 2047]
    c = _case(6, 16, hkv, 128, 0, 5000, pos, seed=14)
    full = wa.decode(c["q"], c["k"], c["v"], c["pos"], 0, 1.0)
    for order in ([5, 4, 3, 2, 1, 0], [0], [1, 4], [2, 3, 5]):
        sel = torch.tensor(order, device="cuda")
        part = wa.decode(c["q"][sel].contiguous(), c["k"][sel].contiguous(), c["v"][sel].contiguous(),
                         c["pos"][sel].contiguous(), 0, 1.0)
        assert torch.equal(part.view(torch.int16), full[sel].view(torch.int16)), order


@pytest.mark.parametrize("hkv", [2, 1])
def test_bad_positions_clamped_on_a_linear_cache_of_many_chunks(wa, hkv):
    """Out-of-range positions on the tensor-core path (groups of 4 and 8, 16 chunks a row): reported,
    and the rows computed as at the clamped positions."""
    c = _case(3, 8, hkv, 128, 0, 4096, [0, 4095, 100], seed=15, outside="keep")
    ws = torch.empty(wa.decode_ws_bytes(3, 8, 128, 0, 4096), dtype=torch.uint8, device="cuda")
    bad = torch.tensor([-3, 7000, 100], dtype=torch.int32, device="cuda")
    out = wa.decode(c["q"], c["k"], c["v"], bad, 0, 1.0, ws=ws)
    assert wa.status(ws) & wa.WA_STATUS_BAD_POS
    clamped = wa.decode(c["q"], c["k"], c["v"], c["pos"], 0, 1.0, ws=ws)
    assert wa.status(ws) == 0
    assert torch.equal(out.view(torch.int16), clamped.view(torch.int16))


def test_linear_cache_past_the_sorted_schedule(wa):
    """A linear cache of 1,026 chunks a row: too many for the tensor-core decode's sorted schedule,
    so its units go out in a plain stride."""
    ring = 1025 * 256 + 44
    c = _case(2, 8, 1, 128, 0, ring, [ring - 1, 5000], seed=16)
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], 0, 1.0)
    assert_parity(out, decode_ref(c), TOL, "stride schedule")


def test_many_rows_past_the_sorted_schedule(wa):
    """2,100 rows at groups of 4: more rows than the tensor-core decode's sorted schedule holds, so
    its units go out in a plain stride; sampled rows against the oracle."""
    gen = torch.Generator().manual_seed(17)
    pos = torch.randint(0, 5000, (2100,), generator=gen).tolist()
    c = _case(2100, 4, 1, 128, 64, 64, pos, seed=17, outside="keep")
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], 64, 1.0)
    rows = [0, 1, 777, 2047, 2048, 2099]
    assert_parity(out[rows], decode_ref(c, rows=rows), TOL, "stride schedule, many rows")


def test_bad_positions_are_clamped_and_reported(wa):
    c = _case(2, 4, 2, 128, 0, 512, [10, 20], seed=13, outside="keep")
    ws = torch.empty(wa.decode_ws_bytes(2, 4, 128, 0, 512), dtype=torch.uint8, device="cuda")
    pos = torch.tensor([-3, 700], dtype=torch.int32, device="cuda")
    wa.decode(c["q"], c["k"], c["v"], pos, 0, 1.0, ws=ws)
    assert wa.status(ws) & wa.WA_STATUS_BAD_POS
    wa.decode(c["q"], c["k"], c["v"], c["pos"], 0, 1.0, ws=ws)
    assert wa.status(ws) == 0


# --------------------------- full size: three caches, three streams ---------------------------

def test_decode_at_scale_three_streams_sampled(wa):
    """64 rows, 32/16 heads, d 256, window 1024 over 1536, positions to 40,000, three caches on three streams."""
    gen = torch.Generator().manual_seed(20260003)
    cases, outs, streams = [], [], [torch.cuda.Stream() for _ in range(3)]
    for i in range(3):
        pos = torch.randint(0, 40001, (64,), generator=gen).tolist()
        pos[0] = 40000
        cases.append(wa_synth.decode_case(64, 32, 16, 256, 1024, 1536, pos, seed=20260030 + i, device="cuda",
                                          outside="keep"))
    torch.cuda.synchronize()
    for c, s in zip(cases, streams):
        with torch.cuda.stream(s):
            outs.append(wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, 1.0))
    torch.cuda.synchronize()
    for c, out in zip(cases, outs):
        rows = [0, 17, 40, 63]
        ref = decode_ref(c, rows=rows)
        assert_parity(out[rows], ref, TOL, "at scale")
        assert torch.isfinite(out.float()).all()


def test_decode_gqa8_at_scale_sampled(wa):
    """64 rows, 32 query heads over 4 key heads (tensor-core path), d 256, window 1024 over 1536."""
    gen = torch.Generator().manual_seed(20260005)
    pos = torch.randint(0, 40001, (64,), generator=gen).tolist()
    pos[0] = 40000
    c = wa_synth.decode_case(64, 32, 4, 256, 1024, 1536, pos, seed=20260050, device="cuda", outside="keep")
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, 1.0)
    torch.cuda.synchronize()
    rows = [0, 9, 33, 63]
    assert_parity(out[rows], decode_ref(c, rows=rows), TOL, "gqa8 at scale")
    assert torch.isfinite(out.float()).all()


def test_decode_gqa16_linear_32768_sampled(wa):
    """64 rows over a linear cache of 32,768 keys, 32 query heads over 2 key heads (tensor-core path)."""
    gen = torch.Generator().manual_seed(20260006)
    pos = torch.randint(0, 32768, (64,), generator=gen).tolist()
    pos[7] = 32767
    c = wa_synth.decode_case(64, 32, 2, 256, 0, 32768, pos, seed=20260060, device="cuda", outside="keep")
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], 0, 1.0)
    torch.cuda.synchronize()
    rows = [7, 40]
    assert_parity(out[rows], decode_ref(c, rows=rows), TOL, "gqa16 linear 32768")
    assert torch.isfinite(out.float()).all()


def test_decode_linear_32768_sampled(wa):
    """64 rows over a linear cache of 32,768 keys (window 0), one row at the last position."""
    gen = torch.Generator().manual_seed(20260004)
    pos = torch.randint(0, 32768, (64,), generator=gen).tolist()
    pos[5] = 32767
    c = wa_synth.decode_case(64, 32, 16, 256, 0, 32768, pos, seed=20260040, device="cuda", outside="keep",
                             peaked=True)
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], 0, 1.0)
    torch.cuda.synchronize()
    rows = [5, 31]
    assert_parity(out[rows], decode_ref(c, rows=rows), TOL, "linear 32768")
    assert torch.isfinite(out.float()).all()
