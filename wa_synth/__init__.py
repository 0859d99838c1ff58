"""Seeded synthetic inputs for sliding-window grouped-query attention.

This module is the one piece shared by the float64 oracle side (tests, the CPU
baseline) and the CUDA side (tests, bench, smoke).  It holds none of the
attention arithmetic: only random draws, the RMS scaling of those draws, bf16
rounding through torch's own conversion, and the placement of keys into ring
slots.

Value distributions follow the receipt of TensorFold pull request #1123
("window_attention at head dim 256"), section "Receipt", environment bullet:
query rows at RMS 0.95..1.05, keys at RMS 0.06..0.13, values at unit RMS, and
every few rows one key equal to a query head rescaled to the key RMS, so that
its score is near 30 and the softmax is peaked as well as flat.

The dense non-causal case follows the "Canonical Boundary" and "Preparation"
sections of the page "Exact Numerical Contract": interleaved QKV rows of
3*H*d bf16 elements, Q at offset 0, K at H*d, V at 2*H*d, and a per-head
RMSNorm of Q and K (eps 1e-5) computed in fp32 and rounded to bf16.

Every tensor is drawn from its own torch.Generator keyed by (seed, tag), so a
case is reproducible on a given device.  Tests that compare against the oracle
copy the exact device bits back to the host; nothing here assumes that CPU and
CUDA generators agree.
"""
from __future__ import annotations

import math

import torch

__all__ = [
    "decode_case",
    "prompt_case",
    "dense_qkv_case",
    "sparse_selection",
    "window_lo",
]

_TAGS = {"q": 1, "k": 2, "v": 3, "qr": 4, "kr": 5, "peak": 6, "pos": 7, "misc": 8}


def _gen(seed: int, tag: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + _TAGS[tag] * 7919) % (2**63 - 1))
    return g


def window_lo(p: int, win: int) -> int:
    """First key position a row at position p can see (0 for a linear cache)."""
    return max(0, p - win + 1) if win > 0 else 0


def _unit_rms(x: torch.Tensor) -> torch.Tensor:
    return x / torch.sqrt((x * x).mean(dim=-1, keepdim=True)).clamp_min(1e-30)


def _draw_rows(shape, rms_lo, rms_hi, gen_v, gen_r, device):
    """Gaussian vectors along the last dim, each rescaled to an RMS drawn from U(rms_lo, rms_hi)."""
    x = torch.randn(shape, generator=gen_v, device=device, dtype=torch.float32)
    r = torch.empty(shape[:-1] + (1,), device=device, dtype=torch.float32)
    r.uniform_(rms_lo, rms_hi, generator=gen_r)
    return _unit_rms(x) * r, r


def decode_case(rows, hq, hkv, d, win, ring, pos, seed, device="cpu",
                outside="nan", peaked=True):
    """Decode inputs: q [rows,hq,d], k/v rings [rows,ring,hkv,d] (bf16), pos int32 [rows].

    Each row owns its ring.  Ring slots that hold no key of the row's window
    are filled with NaN when ``outside == "nan"`` (correctness runs), else keep
    their finite random values (timed runs).  With ``peaked`` one visible key
    per (row, key head) is replaced by a query head of that group rescaled to
    the key's RMS.
    """
    device = torch.device(device)
    pos = [int(p) for p in pos]
    assert len(pos) == rows
    G = hq // hkv
    q, _ = _draw_rows((rows, hq, d), 0.95, 1.05, _gen(seed, "q", device), _gen(seed, "qr", device), device)
    q16 = q.to(torch.bfloat16)
    k16 = torch.empty((rows, ring, hkv, d), dtype=torch.bfloat16, device=device)
    v16 = torch.empty((rows, ring, hkv, d), dtype=torch.bfloat16, device=device)
    gk, gkr, gv = _gen(seed, "k", device), _gen(seed, "kr", device), _gen(seed, "v", device)
    kr = torch.empty((rows, ring, hkv, 1), dtype=torch.float32, device=device)
    for r in range(rows):  # one row at a time keeps the fp32 temporaries bounded
        kk, rr = _draw_rows((ring, hkv, d), 0.06, 0.13, gk, gkr, device)
        k16[r] = kk.to(torch.bfloat16)
        kr[r] = rr
        v16[r] = torch.randn((ring, hkv, d), generator=gv, device=device).to(torch.bfloat16)
    if peaked:
        gp = _gen(seed, "peak", "cpu")
        qf = q16.float()
        for r in range(rows):
            lo = window_lo(pos[r], win)
            for g in range(hkv):
                j = lo + int(torch.randint(pos[r] - lo + 1, (1,), generator=gp))
                h = g * G + int(torch.randint(G, (1,), generator=gp))
                s = j % ring
                qh = qf[r, h]
                k16[r, s, g] = (qh * (kr[r, s, g] / torch.sqrt((qh * qh).mean()))).to(torch.bfloat16)
    if outside == "nan":
        for r in range(rows):
            lo = window_lo(pos[r], win)
            if pos[r] - lo + 1 >= ring:
                continue
            held = torch.zeros(ring, dtype=torch.bool)
            held[torch.arange(lo, pos[r] + 1) % ring] = True
            mask = (~held).to(device)
            k16[r][mask] = float("nan")
            v16[r][mask] = float("nan")
    pos_t = torch.tensor(pos, dtype=torch.int32, device=device)
    return {"q": q16, "k": k16, "v": v16, "pos": pos_t,
            "rows": rows, "hq": hq, "hkv": hkv, "d": d, "win": win, "ring": ring}


def prompt_case(n, p0, hq, hkv, d, win, ring, seed, hi_spans=(), device="cpu",
                outside="nan", peaked=True, peak_every=8):
    """Prompt inputs: q [n,hq,d], k/v [ring,hkv,d] (bf16), hi int32 [n] or None.

    ``hi_spans`` lists (a, b) row ranges, inclusive, whose rows all get last key
    p0+b, so they see each other (an image span).  Rows outside every span get
    their own position; with no span, hi is None (the null form).
    Keys the chunk can see, [window_lo(p0), p0+n-1], are random; other slots
    hold NaN for ``outside == "nan"``.  With ``peaked`` every ``peak_every``-th
    row gets, per key head, one visible key equal to a query head of the group
    rescaled to that key's RMS (a later row wins a shared slot).
    """
    device = torch.device(device)
    G = hq // hkv
    span_lo = window_lo(p0, win)
    span_hi = p0 + n - 1
    assert span_hi - span_lo + 1 <= ring, "chunk plus window must fit the ring"
    q, _ = _draw_rows((n, hq, d), 0.95, 1.05, _gen(seed, "q", device), _gen(seed, "qr", device), device)
    q16 = q.to(torch.bfloat16)
    kk, kr = _draw_rows((ring, hkv, d), 0.06, 0.13, _gen(seed, "k", device), _gen(seed, "kr", device), device)
    k16 = kk.to(torch.bfloat16)
    v16 = torch.randn((ring, hkv, d), generator=_gen(seed, "v", device), device=device).to(torch.bfloat16)
    hi = None
    hi_list = [p0 + i for i in range(n)]
    if hi_spans:
        for a, b in hi_spans:
            for i in range(a, b + 1):
                hi_list[i] = p0 + b
        hi = torch.tensor(hi_list, dtype=torch.int32, device=device)
    if peaked:
        gp = _gen(seed, "peak", "cpu")
        qf = q16.float()
        for i in range(0, n, peak_every):
            lo = window_lo(p0 + i, win)
            for g in range(hkv):
                j = lo + int(torch.randint(hi_list[i] - lo + 1, (1,), generator=gp))
                h = g * G + int(torch.randint(G, (1,), generator=gp))
                s = j % ring
                qh = qf[i, h]
                k16[s, g] = (qh * (kr[s, g] / torch.sqrt((qh * qh).mean()))).to(torch.bfloat16)
    if outside == "nan" and span_hi - span_lo + 1 < ring:
        held = torch.zeros(ring, dtype=torch.bool)
        held[torch.arange(span_lo, span_hi + 1) % ring] = True
        mask = (~held).to(device)
        k16[mask] = float("nan")
        v16[mask] = float("nan")
    return {"q": q16, "k": k16, "v": v16, "hi": hi, "p0": p0, "n": n,
            "hq": hq, "hkv": hkv, "d": d, "win": win, "ring": ring}


def dense_qkv_case(N, H, d, seed, device="cpu", eps=1e-5):
    """Interleaved QKV [N, 3*H*d] bf16 with per-(token, head) RMSNormed Q and K.

    Returns the buffer and strided views q, k, v of logical shape [N, H, d]
    (token stride 3*H*d elements, head stride d).  The RMSNorm takes the bf16
    draw to fp32, scales it by 1/sqrt(mean(x^2) + eps) with unit weight, and
    rounds to bf16; values are N(0, 1) rounded to bf16.
    """
    device = torch.device(device)
    W = 3 * H * d
    qkv = torch.empty((N, W), dtype=torch.bfloat16, device=device)
    g = _gen(seed, "q", device)
    step = max(1, (1 << 24) // W)
    for a in range(0, N, step):
        b = min(N, a + step)
        x = torch.randn((b - a, W), generator=g, device=device).to(torch.bfloat16)
        for part in (0, 1):  # Q, then K: RMSNorm per head in fp32
            sl = x[:, part * H * d:(part + 1) * H * d].float().view(b - a, H, d)
            ms = (sl * sl).mean(dim=-1, keepdim=True)
            y = sl * (1.0 / torch.sqrt(ms + eps))
            x[:, part * H * d:(part + 1) * H * d] = y.view(b - a, H * d).to(torch.bfloat16)
        qkv[a:b] = x
    q = qkv.as_strided((N, H, d), (W, d, 1), 0)
    k = qkv.as_strided((N, H, d), (W, d, 1), H * d)
    v = qkv.as_strided((N, H, d), (W, d, 1), 2 * H * d)
    return {"qkv": qkv, "q": q, "k": k, "v": v, "N": N, "H": H, "d": d,
            "scale": 1.0 / math.sqrt(d)}


def sparse_selection(n, p0, hkv, nsel, seed, win=0, slice_rows=64, block=64, device="cpu"):
    """Per-row selected key blocks [n, hkv, nsel] int32 (-1 = unused), shaped like the pages'
    sparse prompt (TensorFold pull request #1622: 2,048 selected keys a row as 64-key blocks,
    rows grouped in 64-row slices).

    Row i at position p (block bp = p // block) and key head g select bp and bp - 1 (the
    causal end), block 0, and a set of random earlier blocks shared by the row's 64-row slice
    and key head (an indexer's choices are alike for neighbouring rows), up to nsel blocks.
    Rows whose window holds at most nsel blocks select all of them.  Blocks are drawn from the
    row's window [window_lo(p), p]."""
    gen = torch.Generator().manual_seed(int(seed) * 7919 + 17)
    sel = torch.full((n, hkv, nsel), -1, dtype=torch.int32)
    shared = {}
    for i in range(n):
        p = p0 + i
        lo_b = window_lo(p, win) // block
        bp = p // block
        s = i // slice_rows
        for g in range(hkv):
            if bp - lo_b + 1 <= nsel:
                blocks = list(range(lo_b, bp + 1))
            else:
                key = (s, g)
                if key not in shared:
                    # candidates: the slice's first row's window minus its own two end blocks
                    p_first = p0 + s * slice_rows
                    c_lo = max(window_lo(p_first, win) // block, lo_b, 1)
                    c_hi = max(c_lo, p_first // block - 2)
                    perm = torch.randperm(c_hi - c_lo + 1, generator=gen)[:nsel] + c_lo
                    shared[key] = perm.tolist()
                blocks = [bp, bp - 1] + ([0] if lo_b == 0 else [])
                for b in shared[key]:
                    if len(blocks) >= nsel:
                        break
                    if lo_b <= b <= bp and b not in blocks:
                        blocks.append(b)
            sel[i, g, :len(blocks)] = torch.tensor(blocks[:nsel], dtype=torch.int32)
    return sel.to(device)
