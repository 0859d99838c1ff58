"""q/k preparation and KV append on the GPU against the float64 preparation oracle.

RMSNorm (page "Exact Numerical Contract", section "Preparation") and the L2 +
rotate-half RoPE preparation (TensorFold pull request #1257, "What the kernel
computes"), written into ring slot pos mod ring.  Prepared values are checked
with oracle.prep.check_prep (the fp32 allowance before the final bf16
rounding, and at least 99 % of outputs equal to the oracle's rounding); v and
every slot the step must not touch are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from _util import bits, ensure_built
from oracle import prep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _inv_freq(d, theta=10000.0):
    # the fp32 inverse frequencies a host forms as 1 / theta^(2j/d) (float64 rounded to fp32)
    return (1.0 / theta ** (np.arange(0, d, 2, dtype=np.float64) / d)).astype(np.float32)


def _src(n, hq, hkv, d, seed, scale=1.0, row=None):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = (hq + 2 * hkv) * d
    row = w if row is None else row
    x = (torch.randn((n, row), generator=g, device="cuda") * scale).to(torch.bfloat16)
    return x


def _sentinel(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)


def _mode_args(mode, d, seed):
    if mode == "rmsnorm":
        return None, None
    rng = np.random.default_rng(seed)
    qs = rng.uniform(0.5, 2.0, d).astype(np.float32)
    return qs, _inv_freq(d)


def _reference(src, pos, hq, hkv, d, mode, qs, inv):
    """Oracle values and allowances: relative for RMSNorm, per element for L2 + RoPE."""
    q, k, v, tq, tk = prep.prepare(bits(src), pos, hq, hkv, d, mode, qs, inv, with_allowance=True)
    if mode == "rmsnorm":
        tq = tk = prep.REL_RMSNORM
    return q, k, v, tq, tk


def _run_decode_layout(wa, n, hq, hkv, d, ring, pos, mode, seed, with_qs=True):
    src = _src(n, hq, hkv, d, seed)
    q_out = torch.zeros((n, hq, d), dtype=torch.bfloat16, device="cuda")
    k_ring = _sentinel((n, ring, hkv, d), seed + 1)
    v_ring = _sentinel((n, ring, hkv, d), seed + 2)
    k0, v0 = k_ring.clone(), v_ring.clone()
    qs, inv = _mode_args(mode, d, seed)
    if not with_qs:
        qs = None
    pos_t = torch.tensor(pos, dtype=torch.int32, device="cuda")
    ws = wa.prep_append(src, pos_t, q_out, k_ring, v_ring, mode=mode,
                        q_scale=None if qs is None else torch.from_numpy(qs).cuda(),
                        inv_freq=None if inv is None else torch.from_numpy(inv).cuda())
    assert wa.status(ws) == 0
    q_ref, k_ref, v_bits, tq, tk = _reference(src, pos, hq, hkv, d, mode, qs, inv)
    rq = prep.check_prep(bits(q_out), q_ref, tq)
    assert rq["ok"], rq
    slots = [p % ring for p in pos]
    ksel = torch.stack([k_ring[t, s] for t, s in enumerate(slots)])
    vsel = torch.stack([v_ring[t, s] for t, s in enumerate(slots)])
    rk = prep.check_prep(bits(ksel), k_ref, tk)
    assert rk["ok"], rk
    assert np.array_equal(bits(vsel), v_bits)
    # every other slot keeps its bits
    mask = torch.ones((n, ring), dtype=torch.bool, device="cuda")
    mask[torch.arange(n, device="cuda"), torch.tensor(slots, device="cuda")] = False
    assert torch.equal(k_ring[mask].view(torch.int16), k0[mask].view(torch.int16))
    assert torch.equal(v_ring[mask].view(torch.int16), v0[mask].view(torch.int16))
    return q_out, k_ring, v_ring


@pytest.mark.parametrize("mode", ["rmsnorm", "l2_rope"])
@pytest.mark.parametrize("hq,hkv,d", [(16, 4, 256), (32, 16, 256), (8, 8, 128), (32, 2, 128)])
def test_decode_layout_parity(wa, mode, hq, hkv, d):
    rng = np.random.default_rng(hq * 1000 + d)
    n, ring = 24, 1536
    pos = rng.integers(0, 200_000, n).tolist()
    pos[:3] = [0, 1535, 199_999]
    _run_decode_layout(wa, n, hq, hkv, d, ring, pos, mode, seed=hq + d)


def test_l2_rope_without_q_scale(wa):
    _run_decode_layout(wa, 8, 16, 4, 256, 512, [5, 600, 70_000, 3, 511, 512, 1, 99_999], "l2_rope", seed=3,
                       with_qs=False)


@pytest.mark.parametrize("mode", ["rmsnorm", "l2_rope"])
def test_prompt_chunk_into_shared_ring_with_wrap(wa, mode):
    """333 tokens at p0 = 5000 into one ring of 1536 slots (slots 392..724 after the wrap)."""
    n, hq, hkv, d, ring, p0 = 333, 32, 16, 256, 1536, 5000
    src = _src(n, hq, hkv, d, 41)
    q_out = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    k_ring = _sentinel((ring, hkv, d), 42)
    v_ring = _sentinel((ring, hkv, d), 43)
    k0, v0 = k_ring.clone(), v_ring.clone()
    qs, inv = _mode_args(mode, d, 44)
    pos = list(range(p0, p0 + n))
    ws = wa.prep_append(src, torch.tensor(pos, dtype=torch.int32, device="cuda"), q_out, k_ring, v_ring, mode=mode,
                        q_scale=None if qs is None else torch.from_numpy(qs).cuda(),
                        inv_freq=None if inv is None else torch.from_numpy(inv).cuda())
    assert wa.status(ws) == 0
    q_ref, k_ref, v_bits, tq, tk = _reference(src, pos, hq, hkv, d, mode, qs, inv)
    rq = prep.check_prep(bits(q_out), q_ref, tq)
    assert rq["ok"], rq
    slots = torch.tensor([p % ring for p in pos], device="cuda")
    rk = prep.check_prep(bits(k_ring[slots]), k_ref, tk)
    assert rk["ok"], rk
    assert np.array_equal(bits(v_ring[slots]), v_bits)
    keep = torch.ones(ring, dtype=torch.bool, device="cuda")
    keep[slots] = False
    assert torch.equal(k_ring[keep].view(torch.int16), k0[keep].view(torch.int16))
    assert torch.equal(v_ring[keep].view(torch.int16), v0[keep].view(torch.int16))


def _inplace_dense(N, H, d, seed):
    """The dense workload's interleaved QKV buffer and in-place views (row 3*H*d)."""
    W = 3 * H * d
    qkv = _src(N, H, H, d, seed)
    q = qkv.as_strided((N, H, d), (W, d, 1), 0)
    k = qkv.as_strided((N, H, d), (W, d, 1), H * d)
    return qkv, q, k


def test_dense_rmsnorm_in_place(wa):
    N, H, d = 2048, 56, 128
    qkv, q, k = _inplace_dense(N, H, d, 51)
    before = bits(qkv).copy()
    ws = wa.prep_append(qkv, torch.arange(N, dtype=torch.int32, device="cuda"), q, k, None, mode="rmsnorm")
    assert wa.status(ws) == 0
    q_ref, k_ref, _ = prep.prepare(before, np.arange(N), H, H, d, "rmsnorm")
    after = bits(qkv).reshape(N, 3, H, d)
    assert prep.check_prep(after[:, 0], q_ref, prep.REL_RMSNORM)["ok"]
    assert prep.check_prep(after[:, 1], k_ref, prep.REL_RMSNORM)["ok"]
    assert np.array_equal(after[:, 2], before.reshape(N, 3, H, d)[:, 2])


def test_dense_rmsnorm_in_place_full_size_sampled(wa):
    """N = 37,810, 56 heads, d 128, row 21,504: the full dense preparation, 256 sampled tokens checked."""
    N, H, d = 37810, 56, 128
    qkv, q, k = _inplace_dense(N, H, d, 52)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(7).integers(0, N, 254)]))
    before = bits(qkv[torch.from_numpy(rows).cuda()]).copy()
    ws = wa.prep_append(qkv, torch.arange(N, dtype=torch.int32, device="cuda"), q, k, None, mode="rmsnorm")
    assert wa.status(ws) == 0
    q_ref, k_ref, _ = prep.prepare(before, rows, H, H, d, "rmsnorm")
    after = bits(qkv[torch.from_numpy(rows).cuda()]).reshape(len(rows), 3, H, d)
    assert prep.check_prep(after[:, 0], q_ref, prep.REL_RMSNORM)["ok"]
    assert prep.check_prep(after[:, 1], k_ref, prep.REL_RMSNORM)["ok"]
    assert np.array_equal(after[:, 2], before.reshape(len(rows), 3, H, d)[:, 2])


def test_negative_position_is_reported_and_skipped(wa):
    n, hq, hkv, d, ring = 4, 8, 2, 128, 64
    src = _src(n, hq, hkv, d, 61)
    q_out = torch.zeros((n, hq, d), dtype=torch.bfloat16, device="cuda")
    k_ring = _sentinel((n, ring, hkv, d), 62)
    k0 = k_ring.clone()
    pos = torch.tensor([3, -1, 70, -5], dtype=torch.int32, device="cuda")
    ws = wa.prep_append(src, pos, q_out, k_ring, None, mode="rmsnorm")
    assert wa.status(ws) & wa.WA_STATUS_BAD_POS
    assert torch.equal(k_ring[1].view(torch.int16), k0[1].view(torch.int16))
    assert torch.equal(k_ring[3].view(torch.int16), k0[3].view(torch.int16))
    assert not q_out[1].any() and not q_out[3].any()
    ws = wa.prep_append(src, torch.tensor([3, 1, 70, 5], dtype=torch.int32, device="cuda"), q_out, k_ring, None,
                        mode="rmsnorm", ws=ws)
    assert wa.status(ws) == 0


def test_bits_do_not_depend_on_the_batch(wa):
    n, hq, hkv, d, ring = 12, 16, 4, 256, 256
    pos = [7, 900, 123_456, 2, 255, 256, 77_777, 31, 199_000, 5, 64, 128]
    src = _src(n, hq, hkv, d, 71)
    inv = torch.from_numpy(_inv_freq(d)).cuda()
    qs = torch.from_numpy(np.random.default_rng(1).uniform(0.5, 2, d).astype(np.float32)).cuda()

    def run(sel):
        q_out = torch.empty((len(sel), hq, d), dtype=torch.bfloat16, device="cuda")
        k_ring = torch.zeros((len(sel), ring, hkv, d), dtype=torch.bfloat16, device="cuda")
        p = torch.tensor([pos[i] for i in sel], dtype=torch.int32, device="cuda")
        wa.prep_append(src[sel].contiguous(), p, q_out, k_ring, None, mode="l2_rope", q_scale=qs, inv_freq=inv)
        return q_out, k_ring

    qa, ka = run(list(range(n)))
    for sel in ([11, 3, 7], [0], [5, 6, 7, 8]):
        qb, kb = run(sel)
        assert torch.equal(qb.view(torch.int16), qa[sel].view(torch.int16))
        assert torch.equal(kb.view(torch.int16), ka[sel].view(torch.int16))


def test_positions_past_2_to_24(wa):
    """fl32(pos) itself rounds above 2^24; the angle is fl32(fl32(pos) * inv) on both sides."""
    pos = [2**24 - 1, 2**24 + 1, 2**25 + 3, 123_456_789, 2**31 - 1]
    _run_decode_layout(wa, len(pos), 16, 4, 256, 4096, pos, "l2_rope", seed=81)


@pytest.mark.parametrize("mode", ["rmsnorm", "l2_rope"])
def test_nonfinite_projections_follow_float64(wa, mode):
    n, hq, hkv, d, ring = 6, 8, 2, 128, 64
    src = _src(n, hq, hkv, d, 91)
    src[1, 5] = float("nan")                      # query head 0 of token 1
    src[2, hq * d + 7] = float("inf")             # key head 0 of token 2
    src[3, 3 * d + 1] = float("-inf")             # query head 3 of token 3
    src[4, (hq + hkv) * d + 2] = float("nan")     # a value: copied as is
    q_out = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    k_ring = torch.zeros((n, ring, hkv, d), dtype=torch.bfloat16, device="cuda")
    v_ring = torch.zeros_like(k_ring)
    qs, inv = _mode_args(mode, d, 92)
    pos = [1, 2, 3, 4, 5, 6]
    ws = wa.prep_append(src, torch.tensor(pos, dtype=torch.int32, device="cuda"), q_out, k_ring, v_ring, mode=mode,
                        q_scale=None if qs is None else torch.from_numpy(qs).cuda(),
                        inv_freq=None if inv is None else torch.from_numpy(inv).cuda())
    assert wa.status(ws) == 0
    q_ref, k_ref, v_bits, tq, tk = _reference(src, pos, hq, hkv, d, mode, qs, inv)
    assert np.isnan(q_ref[1, 0]).any() and not np.isfinite(k_ref[2, 0]).all()
    with np.errstate(invalid="ignore"):
        tq = np.nan_to_num(tq, nan=0.0) if not np.isscalar(tq) else tq
        tk = np.nan_to_num(tk, nan=0.0) if not np.isscalar(tk) else tk
    rq = prep.check_prep(bits(q_out), q_ref, tq)
    assert rq["ok"], rq
    sl = torch.arange(n, device="cuda")
    slots = torch.tensor(pos, device="cuda") % ring
    rk = prep.check_prep(bits(k_ring[sl, slots]), k_ref, tk)
    assert rk["ok"], rk
    assert np.array_equal(bits(v_ring[sl, slots]), v_bits)
