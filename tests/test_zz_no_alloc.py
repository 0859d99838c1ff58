"""wa_decode_static, the allocation-free decode entry point, through the C ABI.

It serves callers that cannot allocate device memory: a plug-in inside a host
framework that owns all device memory and hands out no allocator, or a serving
loop that forbids cudaMalloc after start-up because the call can synchronize the
device.  Its scratch is one library-owned array per device, shared by every call.

Checked here: two calls enqueued back to back on one stream (one synchronize
after both) each give the float64 oracle's values within the decode tolerance
and the workspace entry point's exact bits, on the CUDA-core decode (groups of
2 query heads per key head) and the tensor-core decode (groups of 8), also at a
size close to the scratch's limit; a bad position is reported through
wa_status(NULL, stream); sizes beyond the scratch are refused.  This file is
collected last on purpose.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import wa_synth
from _util import assert_parity, decode_ref, ensure_built
from oracle import check

pytestmark = pytest.mark.gpu

CAP = 16 * 1024 * 1024


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


@pytest.mark.parametrize("hkv", [8, 2], ids=["cuda_core_g2", "tensor_core_g8"])
def test_two_calls_in_a_row_match_the_oracle_and_the_workspace_bits(wa, hkv):
    stream = torch.cuda.current_stream()
    a = _dev(wa_synth.decode_case(3, 16, hkv, 256, 1024, 1536, [900, 1700, 2047], seed=71, outside="nan"))
    b = _dev(wa_synth.decode_case(16, 32, 2 * hkv, 256, 1024, 1536, list(range(1000, 40000, 2437))[:16], seed=72))
    # the second call plants a NaN query, so it also uses the re-run list in the shared scratch
    b["q"][5, 3, 17] = float("nan")
    outs = [torch.empty_like(a["q"]), torch.empty_like(b["q"])]
    # both calls enqueued before one synchronize: the second clears and refills the scratch the
    # first used, so its stream order is what keeps the first call's result intact
    for c, o in zip((a, b), outs):
        assert _static(wa, c, 1024, o, stream) == wa.WA_OK
    torch.cuda.synchronize()
    assert wa.status(None) == 0
    for c, o in zip((a, b), outs):
        want = wa.decode(c["q"], c["k"], c["v"], c["pos"], 1024, 1.0)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), want.view(torch.int16))
        assert_parity(o, decode_ref(c), check.TOL_FP32_P, "static decode")
    assert torch.isnan(outs[1][5, 3].float()).all()


@pytest.mark.parametrize("hkv", [16, 4], ids=["cuda_core_g2", "tensor_core_g8"])
def test_near_the_scratch_limit(wa, hkv):
    """100 rows, 32 query heads, window 1024 (five 256-key chunks a row): 99 % of the scratch."""
    rows, hq, d, win, ring = 100, 32, 256, 1024, 1536
    need = wa.lib().wa_decode_ws_bytes(rows, hq, d, win, ring)
    assert 0.98 * CAP < need <= CAP
    gen = torch.Generator().manual_seed(75)
    pos = torch.randint(0, 40001, (rows,), generator=gen).tolist()
    pos[:4] = [0, 1023, 1024, 40000]
    c = _dev(wa_synth.decode_case(rows, hq, hkv, d, win, ring, pos, seed=76, outside="nan"))
    out = torch.empty_like(c["q"])
    assert _static(wa, c, win, out, torch.cuda.current_stream()) == wa.WA_OK
    want = wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0)
    torch.cuda.synchronize()
    assert wa.status(None) == 0
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    assert_parity(out, decode_ref(c), check.TOL_FP32_P, "static decode near the limit")


def test_bad_position_is_reported_through_the_null_status(wa):
    c = _dev(wa_synth.decode_case(2, 4, 2, 128, 0, 512, [10, 20], seed=77, outside="keep"))
    out = torch.empty_like(c["q"])
    bad = torch.tensor([-3, 700], dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    good = c["pos"]
    c["pos"] = bad
    assert _static(wa, c, 0, out, stream) == wa.WA_OK
    assert wa.lib().wa_status(None, stream.cuda_stream) & wa.WA_STATUS_BAD_POS
    c["pos"] = good
    assert _static(wa, c, 0, out, stream) == wa.WA_OK
    assert wa.lib().wa_status(None, stream.cuda_stream) == 0
    assert_parity(out, decode_ref(c), check.TOL_FP32_P, "static decode after a bad call")


def test_static_refuses_sizes_beyond_its_scratch(wa):
    c = _dev(wa_synth.decode_case(2, 4, 2, 128, 0, 64, [10, 20], seed=73))
    out = torch.empty_like(c["q"])
    L = wa.lib()
    # 64 rows x 32 heads over a linear cache of 32,768 keys needs ~272 MB of partials
    need = L.wa_decode_ws_bytes(64, 32, 256, 0, 32768)
    assert need > CAP
    rc = L.wa_decode_static(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["pos"].data_ptr(),
                            64, 32, 16, 256, 0, 32768, 1.0, out.data_ptr(), None)
    assert rc == -5, rc
    assert b"16 MiB" in L.wa_strerror(rc)
