"""Controls: the GPU parity checks must go red on the six faults the receipt plants, and stay
green on the same inputs without them (TensorFold pull request #1123, "Receipt", kernel-contract
bullet: decode window one key early, merge without exp(m_c - M), merge rounding toward zero, P32
window one key early, P32 ignoring hi, P rounded to bf16 under the P32 range).

No kernel is broken on purpose.  Each fault's effect is produced from correct calls, or planted on
the host in data the kernels produced:

* a window one key early is the kernel called with win + 1 (it then sees exactly one more key, at
  the window's low end) and compared with the oracle at win.  A key equal to a query head sits
  just outside the window, so that one extra key carries most of the weight;
* ignoring hi is the kernel called with hi = None and compared with the oracle under the image
  span's hi;
* the two merge faults are planted in a host merge (float64, chunk order) of the decode kernel's
  own chunk partials, read from the workspace; the same merge without the fault is green;
* P rounded to bf16 under the P32 range is the prompt's one-part mode (p32 = 0) judged with the
  P32 tolerance on a crafted case: two keys a row (win = 2), values of RMS 4, so a bf16 P's error
  (2^-9 relative) moves outputs by more than 3e-3, while P32 keeps them inside.

Also here: every P mode's fp32 sums are exact when every weight is 1 (gate 4, "sums": all keys
alike, integer values, a power-of-two key count, so the exact mean is known), and two P parts
round to the float64 value more often than one.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import wa_synth
from _util import bits, decode_ref, ensure_built
from oracle import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _ok(got_bits, ref, tol):
    return check.compare(got_bits, ref, tol)


def _peak_key(q_head: torch.Tensor, rms: float = 0.1) -> torch.Tensor:
    """A key equal to a query head rescaled to RMS ``rms`` (score about |q| sqrt(d) rms, ~25 at d 256)."""
    qf = q_head.float()
    return (qf * (rms / torch.sqrt((qf * qf).mean()))).to(torch.bfloat16)


# --------------------------------------------------------------------------- decode window

@pytest.mark.parametrize("hkv", [8, 2], ids=["cuda_core_g2", "tensor_core_g8"])
def test_decode_window_one_key_early_goes_red(wa, hkv):
    rows, hq, d, win, ring = 3, 16, 256, 1024, 1536
    pos = [1100, 1700, 40000]
    c = wa_synth.decode_case(rows, hq, hkv, d, win, ring, pos, seed=501, outside="keep", peaked=False)
    G = hq // hkv
    for r, p in enumerate(pos):   # the key one before the window start: query head g*G of row r
        for g in range(hkv):
            c["k"][r, (p - win) % ring, g] = _peak_key(c["q"][r, g * G])
    for key in ("q", "k", "v", "pos"):
        c[key] = c[key].cuda()
    ref = decode_ref(c)
    good = _ok(bits(wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0)), ref, check.TOL_FP32_P)
    early = _ok(bits(wa.decode(c["q"], c["k"], c["v"], c["pos"], win + 1, 1.0)), ref, check.TOL_FP32_P)
    assert good["ok"], good
    assert not early["ok"] and early["n_bad"] > 100, early


# --------------------------------------------------------------------------- merge faults

def _chunk_partials(wa, ws: torch.Tensor, rows: int, hq: int, d: int, win: int, ring: int) -> np.ndarray:
    """The decode workspace's fp32 chunk records [rows, hq, cmax, d + 4] = (m, l, -, -, o[d]): after the
    256-byte header and the int32 re-run list (rounded up to 256 bytes)."""
    cmax = (win - 1 + 255) // 256 + 1 if win > 0 else (ring + 255) // 256
    flags = (rows * hq * 4 + 255) // 256 * 256
    raw = ws.cpu().numpy()
    n = rows * hq * cmax * (d + 4)
    assert wa.decode_ws_bytes(rows, hq, d, win, ring) == 256 + flags + 4 * n
    return raw[256 + flags:256 + flags + 4 * n].view(np.float32).reshape(rows, hq, cmax, d + 4)


def _host_merge(part: np.ndarray, pos, win: int, rescale=True, toward_zero=False) -> np.ndarray:
    """Merge of the chunk records in chunk order: o = sum_c a_c o_c / sum_c a_c l_c, a_c = exp(m_c - M)
    (TensorFold #1123, "What this changes", bullet "Decode"), in float64 from the fp32 records, then to
    bf16 by nearest-even, or toward zero (the fp32 value's top 16 bits) for that fault."""
    rows, hq, _, dd = part.shape
    d = dd - 4
    out = np.zeros((rows, hq, d), dtype=np.uint16)
    for r in range(rows):
        lo = max(0, pos[r] - win + 1) if win > 0 else 0
        nc = pos[r] // 256 - lo // 256 + 1
        for h in range(hq):
            rec = part[r, h, :nc].astype(np.float64)
            m, l, o = rec[:, 0], rec[:, 1], rec[:, 4:]
            a = np.exp(m - m.max()) if rescale else np.ones_like(m)
            val = (a[:, None] * o).sum(axis=0) / (a * l).sum()
            if toward_zero:
                out[r, h] = (val.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            else:
                out[r, h] = oracle.f64_to_bf16(val)
    return out


@pytest.mark.parametrize("hkv", [8, 2], ids=["cuda_core_g2", "tensor_core_g8"])
def test_merge_faults_go_red_on_the_kernels_own_partials(wa, hkv):
    rows, hq, d, win, ring = 3, 16, 256, 1024, 1536
    pos = [900, 1700, 2047]
    c = wa_synth.decode_case(rows, hq, hkv, d, win, ring, pos, seed=502, device="cuda", outside="nan")
    ws = torch.empty(wa.decode_ws_bytes(rows, hq, d, win, ring), dtype=torch.uint8, device="cuda")
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0, ws=ws)
    torch.cuda.synchronize()
    assert wa.status(ws) == 0
    ref = decode_ref(c)
    assert _ok(bits(out), ref, check.TOL_FP32_P)["ok"]
    part = _chunk_partials(wa, ws, rows, hq, d, win, ring)
    good = _ok(_host_merge(part, pos, win), ref, check.TOL_FP32_P)
    no_rescale = _ok(_host_merge(part, pos, win, rescale=False), ref, check.TOL_FP32_P)
    toward_zero = _ok(_host_merge(part, pos, win, toward_zero=True), ref, check.TOL_FP32_P)
    assert good["ok"], good
    assert not no_rescale["ok"] and no_rescale["n_bad"] > 1000, no_rescale
    assert not toward_zero["ok"], toward_zero


# --------------------------------------------------------------------------- prompt P32 faults

@pytest.mark.parametrize("d", [256, 128])
def test_p32_window_one_key_early_goes_red(wa, d):
    n, p0, hq, hkv, win, ring = 300, 1300, 16, 8, 700, 1536
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=503, outside="keep", peaked=False)
    G = hq // hkv
    for i in range(0, n, 37):   # the key one before row i's window: a query head of row i
        for g in range(hkv):
            c["k"][(p0 + i - win) % ring, g] = _peak_key(c["q"][i, g * G], rms=0.1)
    for key in ("q", "k", "v"):
        c[key] = c[key].cuda()
    ref = oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), p0, win, ring, 1.0)
    good = _ok(bits(wa.prompt(c["q"], c["k"], c["v"], p0, None, win, 1.0, p32=True)), ref, check.TOL_P32)
    early = _ok(bits(wa.prompt(c["q"], c["k"], c["v"], p0, None, win + 1, 1.0, p32=True)), ref, check.TOL_P32)
    assert good["ok"], good
    assert not early["ok"] and early["n_bad"] > 100, early


@pytest.mark.parametrize("d", [256, 128])
def test_p32_ignoring_hi_goes_red(wa, d):
    n, p0, hq, hkv, win, ring = 512, 1300, 16, 8, 1024, 1536
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=504, hi_spans=[(40, 300)], outside="keep")
    G = hq // hkv
    for g in range(hkv):   # the image span's last key matches a query head of its first row
        c["k"][(p0 + 300) % ring, g] = _peak_key(c["q"][40, g * G])
    for key in ("q", "k", "v", "hi"):
        c[key] = c[key].cuda()
    ref = oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), p0, win, ring, 1.0, hi=c["hi"].cpu().numpy())
    good = _ok(bits(wa.prompt(c["q"], c["k"], c["v"], p0, c["hi"], win, 1.0, p32=True)), ref, check.TOL_P32)
    no_hi = _ok(bits(wa.prompt(c["q"], c["k"], c["v"], p0, None, win, 1.0, p32=True)), ref, check.TOL_P32)
    assert good["ok"], good
    assert not no_hi["ok"] and no_hi["n_bad"] > 100, no_hi


def _two_key_case(n, p0, hq, hkv, d, seed, v_rms=4.0):
    """Two visible keys a row (win = 2) with scores a few units apart, so P = exp(s_other - s_max) is
    spread over (0, 1], and values of RMS ``v_rms``: a bf16 P's relative error 2^-9 then moves the
    output by up to about 2^-9 * 4 * |v| / 2, above 3e-3, where P32's 2^-17 stays far below it."""
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, 2, 2 * n + 8, seed=seed, outside="keep", peaked=False)
    c["v"] = (c["v"].float() * v_rms).to(torch.bfloat16)
    return c


@pytest.mark.parametrize("d", [256, 128])
def test_bf16_p_under_the_p32_range_goes_red(wa, d):
    n, p0 = 512, 600
    c = _two_key_case(n, p0, 16, 8, d, seed=505)
    for key in ("q", "k", "v"):
        c[key] = c[key].cuda()
    ref = oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), p0, 2, c["ring"], 1.0)
    r = {p32: _ok(bits(wa.prompt(c["q"], c["k"], c["v"], p0, None, 2, 1.0, p32=p32)), ref, check.TOL_P32)
         for p32 in (0, 1, 2)}
    assert not r[0]["ok"] and r[0]["n_bad"] > 50, r[0]
    assert r[1]["ok"], r[1]
    assert r[2]["ok"], r[2]
    # and the bf16 P stays within its own 8e-3 reading only where |v| is unit: here it need not


def _bf16_p_decode(q, k, v, pos, win, ring):
    """The decode formula with each weight exp(s_j - m) rounded to bf16 before it meets v (the sum
    keeps the unrounded weights): the "P rounded to bf16" fault planted in a float64 evaluation."""
    q = oracle.bf16_to_f64(q)
    rows, hq, d = q.shape
    hkv = k.shape[2]
    G = hq // hkv
    out = np.zeros((rows, hq, d))
    for r in range(rows):
        lo = max(0, pos[r] - win + 1) if win > 0 else 0
        slots = np.arange(lo, pos[r] + 1) % ring
        for h in range(hq):
            kk = oracle.bf16_to_f64(k[r, slots, h // G])
            vv = oracle.bf16_to_f64(v[r, slots, h // G])
            s = kk @ q[r, h]
            w = np.exp(s - s.max())
            wq = oracle.bf16_to_f64(oracle.f64_to_bf16(w))
            out[r, h] = (wq @ vv) / w.sum()
    return out


@pytest.mark.parametrize("hkv", [8, 2], ids=["cuda_core_g2", "tensor_core_g8"])
def test_decode_probabilities_hold_the_p32_range_where_bf16_p_cannot(wa, hkv):
    """Decode keeps P to fp32 (the CUDA-core kernel) or to two bf16 parts (the tensor-core kernel):
    on two keys a row with values of RMS 4 it stays within 3e-3, while the same arithmetic with P
    rounded to bf16, planted in a float64 evaluation, does not."""
    rows, hq, d, win, ring = 64, 16, 256, 2, 8
    gen = torch.Generator().manual_seed(506)
    pos = torch.randint(1, 40000, (rows,), generator=gen).tolist()
    c = wa_synth.decode_case(rows, hq, hkv, d, win, ring, pos, seed=506, outside="nan", peaked=False)
    c["v"] = (c["v"].float() * 4.0).to(torch.bfloat16)
    ref = decode_ref(c)
    planted = _bf16_p_decode(bits(c["q"]), bits(c["k"]), bits(c["v"]), pos, win, ring)
    fault = _ok(oracle.f64_to_bf16(planted), ref, check.TOL_FP32_P)
    assert not fault["ok"] and fault["n_bad"] > 50, fault
    for key in ("q", "k", "v", "pos"):
        c[key] = c[key].cuda()
    got = _ok(bits(wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0)), ref, check.TOL_FP32_P)
    assert got["ok"], got


@pytest.mark.parametrize("d", [256, 128])
def test_two_p_parts_round_to_float64_more_often_than_one(wa, d):
    """On the receipt's distributions (unit-RMS values), outputs equal to RN(o): more with P32 than
    with a bf16 P, and more again with three parts."""
    c = wa_synth.prompt_case(700, 0, 16, 8, d, 0, 700, seed=507, device="cuda", outside="keep", peak_every=64)
    ref = oracle.prompt(bits(c["q"]), bits(c["k"]), bits(c["v"]), 0, 0, 700, 1.0)
    rn = oracle.f64_to_bf16(ref).ravel()
    hits = {}
    for p32 in (0, 1, 2):
        out = bits(wa.prompt(c["q"], c["k"], c["v"], 0, None, 0, 1.0, p32=p32)).ravel()
        hits[p32] = int((out == rn).sum())
    assert hits[0] < hits[1] < hits[2], hits


# --------------------------------------------------------------------------- gate 4: sums

def _integer_values(shape, seed, device):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(-8, 9, shape, generator=g).to(torch.bfloat16).to(device)


@pytest.mark.parametrize("hkv", [8, 2], ids=["cuda_core_g2", "tensor_core_g8"])
@pytest.mark.parametrize("d", [256, 128])
def test_decode_equal_weights_give_the_exact_mean(wa, hkv, d):
    """Every visible key is the zero vector, so every score is 0 and every weight exactly 1; values
    are integers in [-8, 8] and each row sees 1,024 keys, so o is the exact mean, and its bf16
    rounding is the only rounding: every output bit-equal to RN(mean)."""
    rows, hq, win, ring = 4, 16, 1024, 1536
    pos = [1023, 1500, 2047, 40000]
    c = wa_synth.decode_case(rows, hq, hkv, d, win, ring, pos, seed=508, device="cuda", outside="nan", peaked=False)
    for r, p in enumerate(pos):
        slots = torch.arange(p - win + 1, p + 1, device="cuda") % ring
        c["k"][r, slots] = 0
        c["v"][r, slots] = _integer_values((win, hkv, d), 509 + r, "cuda")
    out = wa.decode(c["q"], c["k"], c["v"], c["pos"], win, 1.0)
    torch.cuda.synchronize()
    G = hq // hkv
    v = bits(c["v"])
    for r, p in enumerate(pos):
        slots = np.arange(p - win + 1, p + 1) % ring
        mean = oracle.bf16_to_f64(v[r, slots]).sum(axis=0) / win          # [hkv, d], exact
        want = oracle.f64_to_bf16(np.repeat(mean, G, axis=0))
        assert np.array_equal(bits(out[r]), want), r


@pytest.mark.parametrize("p32", [0, 1, 2])
@pytest.mark.parametrize("d", [256, 128])
def test_prompt_equal_weights_give_the_exact_mean(wa, d, p32):
    """As above for every P mode of the prompt: 300 rows at p0 1000, window 256 (every row sees
    256 keys), keys all zero, integer values."""
    n, p0, hq, hkv, win, ring = 300, 1000, 8, 4, 256, 1536
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, win, ring, seed=510, device="cuda", outside="nan", peaked=False)
    lo, hi = p0 - win + 1, p0 + n - 1
    slots = torch.arange(lo, hi + 1, device="cuda") % ring
    c["k"][slots] = 0
    c["v"][slots] = _integer_values((hi - lo + 1, hkv, d), 511, "cuda")
    out = wa.prompt(c["q"], c["k"], c["v"], p0, None, win, 1.0, p32=p32)
    torch.cuda.synchronize()
    v = oracle.bf16_to_f64(bits(c["v"]))
    csum = np.concatenate([np.zeros((1, hkv, d)), np.cumsum(v[(np.arange(lo, hi + 1)) % ring], axis=0)])
    G = hq // hkv
    for i in (0, 1, 127, 128, 255, 256, 299):
        mean = (csum[i + win] - csum[i]) / win                               # keys p0+i-255 .. p0+i
        want = oracle.f64_to_bf16(np.repeat(mean, G, axis=0))
        assert np.array_equal(bits(out[i]), want), i
    got = bits(out)
    idx = np.arange(n)
    means = (csum[idx + win] - csum[idx]) / win
    assert np.array_equal(got, oracle.f64_to_bf16(np.repeat(means, G, axis=1)))


@pytest.mark.parametrize("p32", [0, 2])
def test_block_sparse_equal_weights_give_the_exact_mean(wa, p32):
    """Block-sparse prompt: each row selects the four whole 64-key blocks before its own block
    (256 keys, all visible), keys zero, integer values."""
    n, p0, hq, hkv, d = 200, 640, 12, 2, 256
    ring = p0 + n
    c = wa_synth.prompt_case(n, p0, hq, hkv, d, 0, ring, seed=512, device="cuda", outside="keep", peaked=False)
    c["k"].zero_()
    c["v"].copy_(_integer_values((ring, hkv, d), 513, "cuda"))
    bp = (p0 + np.arange(n)) // 64
    sel_np = np.stack([bp - 4, bp - 3, bp - 2, bp - 1], axis=1)[:, None, :].repeat(hkv, axis=1).astype(np.int32)
    sel = torch.from_numpy(sel_np).cuda()
    out = wa.prompt_sparse(c["q"], c["k"], c["v"], p0, sel, None, 0, 1.0, p32=p32)
    torch.cuda.synchronize()
    v = oracle.bf16_to_f64(bits(c["v"]))
    G = hq // hkv
    want = np.zeros((n, hq, d), dtype=np.uint16)
    for i in range(n):
        keys = np.arange((bp[i] - 4) * 64, bp[i] * 64)
        want[i] = oracle.f64_to_bf16(np.repeat(v[keys].sum(axis=0) / 256.0, G, axis=0))
    assert np.array_equal(bits(out), want)
