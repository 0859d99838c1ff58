"""wa_decode_static, the allocation-free decode entry point, through the C ABI.

It serves callers that cannot allocate device memory (a plug-in inside a host
framework that owns all device memory, or a serving loop that forbids
cudaMalloc after start-up).  Its output must match the workspace-taking
wa_decode within the parity tolerance, on two calls in a row over the shared
library-owned scratch, and sizes beyond the fixed scratch must be refused.
This file is collected last on purpose.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import wa_synth
from _util import bits, ensure_built
from oracle import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m = ensure_built()
    L = m.lib()
    P, I = ctypes.c_void_p, ctypes.c_int32
    L.wa_decode_static.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_float, P, P]
    L.wa_decode_static.restype = ctypes.c_int
    return m


def _static(wa, c, win, out, stream):
    rows, hq, d = c["q"].shape
    _, ring, hkv, _ = c["k"].shape
    return wa.lib().wa_decode_static(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["pos"].data_ptr(),
                                     rows, hq, hkv, d, win, ring, 1.0, out.data_ptr(), stream.cuda_stream)


def _dev(c):
    for key in ("q", "k", "v", "pos"):
        c[key] = c[key].cuda()
    return c


def test_static_matches_workspace_entry_two_calls_in_a_row(wa):
    stream = torch.cuda.current_stream()
    a = _dev(wa_synth.decode_case(3, 16, 8, 256, 1024, 1536, [900, 1700, 2047], seed=71, outside="nan"))
    b = _dev(wa_synth.decode_case(16, 32, 16, 256, 1024, 1536, list(range(1000, 40000, 2437))[:16], seed=72))
    # the second call plants a NaN query, so it also exercises the re-run list in the shared scratch
    b["q"][5, 3, 17] = float("nan")
    for c in (a, b):
        want = wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, 1.0)
        got = torch.empty_like(want)
        rc = _static(wa, c, 1024, got, stream)
        assert rc == wa.WA_OK, rc
        torch.cuda.synchronize()
        r = check.compare(bits(got), wa_synth_value(want), check.TOL_FP32_P)
        assert r["ok"], r
        assert torch.equal(torch.isnan(got.float()), torch.isnan(want.float()))


def test_static_tensor_core_decode_gives_the_workspace_bits(wa):
    """Groups of 8 query heads per key head take the tensor-core partial kernel; over the
    library-owned scratch it must give the workspace entry's bits."""
    stream = torch.cuda.current_stream()
    c = _dev(wa_synth.decode_case(4, 32, 4, 256, 1024, 1536, [1535, 700, 40000, 2049], seed=74))
    want = wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, 1.0)
    got = torch.empty_like(want)
    assert _static(wa, c, 1024, got, stream) == wa.WA_OK
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def wa_synth_value(t):
    return t.float().cpu().numpy().astype(np.float64)


def test_static_refuses_sizes_beyond_its_scratch(wa):
    c = _dev(wa_synth.decode_case(2, 4, 2, 128, 0, 64, [10, 20], seed=73))
    out = torch.empty_like(c["q"])
    L = wa.lib()
    # 64 rows x 32 heads over a linear cache of 32,768 keys needs ~272 MB of partials
    need = L.wa_decode_ws_bytes(64, 32, 256, 0, 32768)
    assert need > 16 * 1024 * 1024
    rc = L.wa_decode_static(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["pos"].data_ptr(),
                            64, 32, 16, 256, 0, 32768, 1.0, out.data_ptr(), None)
    assert rc == -5, rc
    assert b"16 MiB" in L.wa_strerror(rc)
