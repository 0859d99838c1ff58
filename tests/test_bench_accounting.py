"""The bench's algorithmic work, checked against independent counts (CPU).

Decode bytes count each visible key's K and V row once per key head (plus q and out); prompt
flops count 4*d per visible (row, key, head); the block-sparse prompt counts only the keys of
selected blocks inside each row's range.  Each is recounted here key by key from the oracle's
own visibility functions, so a slip in a closed form (a window off by one, a repeated block
counted twice) fails.
"""
from __future__ import annotations

import numpy as np
import torch

import bench
import oracle


def test_decode_bytes_count_each_visible_key_once():
    hq, hkv, d = 32, 16, 256
    for win, pos in ((1024, [0, 1, 1023, 1024, 40000]), (0, [0, 5, 32767])):
        keys = sum(hi - lo + 1 for lo, hi in (oracle.visible_decode(p, win) for p in pos))
        want = keys * hkv * d * 2 * 2 + 2 * len(pos) * hq * d * 2
        assert bench.decode_bytes(pos, hq, hkv, d, win) == want


def test_prompt_flops_against_a_key_by_key_count():
    p0, n, win, hq, d = 100, 50, 30, 4, 128
    rows = range(n)
    count = 0
    for i in rows:
        lo, hi = oracle.visible_prompt(p0, i, win)
        count += sum(1 for _ in range(lo, hi + 1))
    assert bench.prompt_flops_rows(rows, p0, win, lambda r: p0 + r, hq, d) == count * hq * 4 * d


def test_causal_and_dense_part_flops():
    s = bench.SPEC["prompt_causal"]
    n = s["n"]
    assert bench.part_work("prompt_causal")["flops"] == n * (n + 1) // 2 * s["hq"] * 4 * s["d"]
    s = bench.SPEC["prompt_dense"]
    assert bench.part_work("prompt_dense")["flops"] == s["N"] ** 2 * s["H"] * 4 * s["d"]


def test_sparse_visible_keys_match_the_oracle_key_sets():
    s = dict(bench.SPEC["prompt_sparse"])
    s.update(n=300, p0=3000, ring=3300)
    vis = bench.sparse_visible_keys(s)
    sel = bench.sparse_selection_of(s).numpy()
    for i in (0, 1, 63, 64, 150, 299):
        lo, hi = oracle.visible_prompt(s["p0"], i, s["win"])
        for g in range(s["hkv"]):
            assert vis[i, g] == len(oracle.sparse_keys(lo, hi, sel[i, g]))
    # repeats and unused entries count nothing extra
    s2 = dict(s, n=2, p0=200, nsel=4)
    bench._SEL_CACHE[(2, 200, s2["hkv"], 4, s2["seed"], s2["win"])] = torch.tensor(
        [[[1, 1, -1, 3]] * s2["hkv"], [[0, 3, 3, 3]] * s2["hkv"]], dtype=torch.int32)
    v2 = bench.sparse_visible_keys(s2)
    assert v2[0, 0] == 64 + (200 - 192 + 1)       # block 1 whole, block 3 up to position 200
    assert v2[1, 0] == 64 + (201 - 192 + 1)


def test_prep_bytes_and_weak_scaling():
    s = bench.SPEC["prep_dense"]
    assert bench.part_work("prep_dense")["bytes"] == 2 * s["N"] * 2 * s["H"] * s["d"] * 2
    assert bench.weak_scaling_value(2.0, 4000.0, 1) == 0.5
    assert bench.weak_scaling_value(2.0, 4000.0, 4) == 2.0


def test_roofline_seconds_adds_bytes_and_flops():
    """Bytes at the copy bandwidth, flops at the burst bf16 rate (each part is timed alone)."""
    pk = {"hbm_gbs": 1000.0, "bf16_tflops": 1000.0, "bf16_tflops_sustained": 500.0}
    t = bench.roofline_seconds(["decode_linear", "prompt_dense"], pk)
    w1, w2 = bench.part_work("decode_linear"), bench.part_work("prompt_dense")
    assert np.isclose(t, w1["bytes"] / 1e12 + w2["flops"] / 1e15)


def test_dense_workload_is_timed_in_both_p_modes():
    """The dense workload's P precision is open, so the step holds it with one and with two P parts;
    both count the same algorithmic flops (the second part's products are issued, not algorithmic)."""
    assert "prompt_dense" in bench.PARTS and "prompt_dense_p32" in bench.PARTS
    a, b = bench.part_work("prompt_dense"), bench.part_work("prompt_dense_p32")
    assert a["flops"] == b["flops"]
    assert a["issued_flops_factor"] == 1.0 and b["issued_flops_factor"] == 1.5


def test_part_report_fractions_use_the_burst_peak():
    pk = {"hbm_gbs": 1000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    w = bench.part_work("prompt_causal")
    ms = w["flops"] / 1e12 / 1000.0 * 1e3          # 1,000 TFLOP/s
    r = bench.report_part("prompt_causal", ms, pk)
    assert np.isclose(r["TFLOP/s"], 1000.0)
    assert np.isclose(r["frac_bf16"], 0.5) and np.isclose(r["frac_bf16_sustained"], 0.625)


def _flow_shop_span(order, first, second):
    """Span of jobs through two machines in series, each job's second stage after its first."""
    t1 = t2 = 0.0
    for i in order:
        t1 += first[i]
        t2 = max(t2, t1) + second[i]
    return t2


def test_e2e_part_order_is_a_shortest_two_stage_schedule():
    """The e2e leg issues the parts' copies in Johnson's order; by brute force over every order of
    small random instances, that order reaches the shortest two-machine span."""
    import itertools
    rng = np.random.default_rng(5)
    for _ in range(200):
        n = int(rng.integers(1, 7))
        first = list(rng.uniform(0.1, 10.0, n))
        second = list(rng.uniform(0.1, 10.0, n))
        best = min(_flow_shop_span(p, first, second) for p in itertools.permutations(range(n)))
        got = bench.johnson_order(first, second)
        assert sorted(got) == list(range(n))
        assert _flow_shop_span(got, first, second) <= best * (1 + 1e-12)
    # the default step's shape: dense prompts (short copies, long kernels) first, then the cache
    # parts by kernel time
    order = bench.johnson_order([7.6, 7.6, 0.7, 11.4, 161.0], [38.0, 28.0, 0.5, 0.6, 3.7])
    assert order == [0, 1, 4, 3, 2]
