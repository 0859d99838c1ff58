"""The entry points inside a captured CUDA graph (a serving loop replays one decode step).

Each call is a status clear and kernel launches on the caller's stream, with its tensor maps
encoded on the host at capture time, so a graph of it replays the same work: the replayed
outputs must carry the eager call's bits, also after the inputs change in place.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import wa_synth
from _util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _eq(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("hkv", [16, 4])   # CUDA-core and tensor-core decode
def test_decode_step_in_a_graph(wa, hkv):
    rows, hq, d, win, ring = 16, 32, 256, 1024, 1536
    pos = list(range(1500, 40000, 2400))[:rows]
    c = wa_synth.decode_case(rows, hq, hkv, d, win, ring, pos, seed=5, device="cuda", outside="keep")
    out = torch.empty_like(c["q"])
    ws = torch.empty(wa.decode_ws_bytes(rows, hq, d, win, ring), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0, out=out, ws=ws, stream=s)   # warm-up, attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0, out=out, ws=ws, stream=s)
    for step in range(3):
        c["pos"].add_(1)                                   # the next token of every row
        c["q"].copy_(torch.roll(c["q"], 1, dims=1))
        g.replay()
        torch.cuda.synchronize()
        want = wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0)
        torch.cuda.synchronize()
        assert _eq(out, want), step
        assert wa.status(ws) == 0


def test_prompt_sparse_and_preparation_in_one_graph(wa):
    n, p0, hq, hkv, d, ring = 256, 2000, 24, 2, 256, 2256
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, 0, ring, seed=6, device="cuda", outside="keep")
    sel = wa_synth.sparse_selection(n, p0, hkv, 32, seed=7, device="cuda")
    out_d = torch.empty_like(c["q"])
    out_s = torch.empty_like(c["q"])
    ws_d = torch.empty(wa.prompt_ws_bytes(n, hq), dtype=torch.uint8, device="cuda")
    ws_s = torch.empty_like(ws_d)
    gen = torch.Generator(device="cuda").manual_seed(8)
    src = torch.randn((8, (hq + 2 * hkv) * d), generator=gen, device="cuda").to(torch.bfloat16)
    q_out = torch.empty((8, hq, d), dtype=torch.bfloat16, device="cuda")
    k_ring = torch.zeros((8, 512, hkv, d), dtype=torch.bfloat16, device="cuda")
    pos = torch.arange(100, 108, dtype=torch.int32, device="cuda")
    inv = torch.from_numpy((1.0 / 10000.0 ** (np.arange(0, d, 2) / d)).astype(np.float32)).cuda()
    ws_p = torch.empty(256, dtype=torch.uint8, device="cuda")

    def step(st):
        wa.prompt(c["q"], c["k"], c["v"], p0, None, 0, 1.0, p32=True, out=out_d, ws=ws_d, stream=st)
        wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, 0, 1.0, p32=2, out=out_s, ws=ws_s, stream=st)
        wa.prep_append(src, pos, q_out, k_ring, None, mode="l2_rope", inv_freq=inv, ws=ws_p, stream=st)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    c["q"].mul_(-1)          # change the inputs in place; the graph reads them afresh
    src.mul_(0.5)
    g.replay()
    torch.cuda.synchronize()
    want_d = wa.prompt(c["q"], c["k"], c["v"], p0, None, 0, 1.0, p32=True)
    want_s = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, 0, 1.0, p32=2)
    want_q = torch.empty_like(q_out)
    want_k = torch.zeros_like(k_ring)
    wa.prep_append(src, pos, want_q, want_k, None, mode="l2_rope", inv_freq=inv)
    torch.cuda.synchronize()
    assert _eq(out_d, want_d) and _eq(out_s, want_s)
    assert _eq(q_out, want_q) and _eq(k_ring, want_k)
