"""Facts the pages print, recomputed from the definitions the code uses (CPU only)."""
import json
import math
import os

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "page_facts.json")))


def test_dense_layout_strides():
    f = FACTS["dense_layout"]
    N, H, d = f["N"], f["heads"], f["d"]
    assert 3 * H * d == f["row_width"]
    assert [0, H * d, 2 * H * d] == f["offsets"]
    assert [N * 3 * H * d, 3 * H * d, d, 1] == f["strides"]
    assert H * d == f["out_token_major_width"]


def test_dense_tail_counts():
    f, N = FACTS["dense_tails"], FACTS["dense_layout"]["N"]
    assert N - (math.ceil(N / f["q_tile"]) - 1) * f["q_tile"] == f["valid_rows_last_q_tile"]
    assert N - (math.ceil(N / f["k_tile"]) - 1) * f["k_tile"] == f["valid_rows_last_k_tile"]
    assert math.ceil(N / f["k_tile"]) - 1 == f["last_k_tile_index"]


def test_scale_shapes():
    f, N = FACTS["scale_shapes"], FACTS["dense_layout"]["N"]
    assert math.ceil(N / f["q_cta_rows"]) * (f["q_cta_rows"] // f["q_group_rows"]) == f["q_groups"]
    assert math.ceil(N / f["k_block_rows"]) == f["k_blocks"]


def test_decode_bytes_of_one_row():
    f = FACTS["decode_bytes"]
    lo, hi = oracle.visible_decode(10_000, f["win"])
    nvis = hi - lo + 1
    assert f["hkv"] * nvis * f["d"] * 2 * 2 == f["bytes"]
    assert abs(f["bytes"] / (f["us"] * 1e-6) / 1e9 - f["gbs_about"]) < 1.0


def test_chunk_plus_window_fits_ring():
    f = FACTS["gemma_sliding"]
    lo, _ = oracle.visible_prompt(5000, 0, f["win"])
    assert (5000 + f["chunk"] - 1) - lo + 1 <= f["ring"]
