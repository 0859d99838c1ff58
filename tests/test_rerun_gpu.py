"""The float64 re-run with thousands of flagged (row, head) pairs.

TensorFold pull request #1123, "What this changes", bullet "A NaN or infinite output re-runs its
head in float64", limited to the affected row and head (review thread).  One non-finite key or
value that every row can see flags every row of its key head's group, so the re-run must scale
with the flag count: a 4,096-row prompt at head dim 128 with a NaN key token (every key head) that
every row sees flags all 32,768 (row, head) pairs; an infinite value flags 8,192.  Sampled rows
are checked against the float64 oracle, and each whole call (prompt kernel and re-run) must take
under a second: the re-run used to walk its list with 64 CTAs and serial float64 dot products, a
time of minutes at this size.
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

N, HQ, HKV, D = 4096, 8, 4, 128
ROWS = [0, 1, 777, 2048, 2999, 3000, 3001, 4095]


@pytest.fixture(scope="module")
def wa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _timed(fn):
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    out = fn()
    b.record()
    torch.cuda.synchronize()
    return out, a.elapsed_time(b)


def test_nan_key_token_seen_by_every_row(wa):
    """Non-causal (hi = N - 1): key 3,000 is NaN in every key head, so every output is NaN."""
    c = wa_synth.prompt_case(N, 0, HQ, HKV, D, 0, N, seed=601, device="cuda", outside="keep")
    c["k"][3000, :, 7] = float("nan")
    hi = torch.full((N,), N - 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(wa.prompt_ws_bytes(N, HQ), dtype=torch.uint8, device="cuda")
    wa.prompt(c["q"], c["k"], c["v"], 0, hi, 0, 1.0, p32=True, ws=ws)          # warm-up
    out, ms = _timed(lambda: wa.prompt(c["q"], c["k"], c["v"], 0, hi, 0, 1.0, p32=True, ws=ws))
    assert wa.status(ws) == 0
    nflag = int(ws[4:8].view(torch.int32).item())
    assert nflag == N * HQ, nflag
    assert torch.isnan(out.float()).all()
    ref = oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), 0, 0, N, 1.0, hi=hi.cpu().numpy(), rows=ROWS)
    assert_parity(out[ROWS], ref, check.TOL_P32, "nan key token")
    print(f"\n{nflag} flagged heads, prompt + re-run {ms:.2f} ms")
    assert ms < 1000.0, ms


def test_inf_value_seen_by_every_row(wa):
    """Causal: value 10 of key head 1 holds +inf in one dim, so rows 10 .. N-1 of query heads 2 and 3
    are flagged; rows 0 .. 9, which cannot see it, share its key tile, where P = 0 meets the
    infinity as 0 * inf = NaN in the tensor-core product, so they are flagged and repaired as
    well (8,192 pairs in all).  The other dims come out of the float64 passes."""
    c = wa_synth.prompt_case(N, 0, HQ, HKV, D, 0, N, seed=602, device="cuda", outside="keep")
    c["v"][10, 1, 5] = float("inf")
    ws = torch.empty(wa.prompt_ws_bytes(N, HQ), dtype=torch.uint8, device="cuda")
    wa.prompt(c["q"], c["k"], c["v"], 0, None, 0, 1.0, p32=True, ws=ws)
    out, ms = _timed(lambda: wa.prompt(c["q"], c["k"], c["v"], 0, None, 0, 1.0, p32=True, ws=ws))
    assert wa.status(ws) == 0
    nflag = int(ws[4:8].view(torch.int32).item())
    assert (N - 10) * 2 <= nflag <= N * 2, nflag
    ref = oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), 0, 0, N, 1.0, rows=ROWS)
    assert_parity(out[ROWS], ref, check.TOL_P32, "inf value")
    # the re-run heads are float64 results rounded once: within the three-part bound as well
    assert_parity(out[ROWS][:, 2:4], ref[:, 2:4], check.TOL_P3, "inf value, re-run heads")
    assert np.isinf(ref[2:, 2:4, 5]).all() and np.isfinite(ref[:2]).all()
    print(f"\n{nflag} flagged heads, prompt + re-run {ms:.2f} ms")
    assert ms < 1000.0, ms
