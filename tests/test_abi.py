"""The C ABI without a GPU: the library loads, exports what include/wa.h declares,
sizes workspaces, and rejects bad arguments before touching CUDA."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from _util import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    hdr_dir = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(hdr_dir)):
        if fn.endswith(".h"):
            src = open(os.path.join(hdr_dir, fn)).read()
            names += re.findall(r"^\s*(?:int|size_t|const char\s*\*)\s*(wa_\w+)\s*\(", src, re.M)
    return names


def test_every_declared_symbol_is_exported():
    wa = ensure_built()
    names = _declared()
    assert {"wa_decode", "wa_prompt", "wa_decode_ws_bytes", "wa_prompt_ws_bytes", "wa_status",
            "wa_strerror", "wa_version"} <= set(names)
    raw = ctypes.CDLL(wa.lib_path())
    for n in names:
        assert hasattr(raw, n), n


def test_workspace_sizes():
    wa = ensure_built()
    L = wa.lib()
    # header 256 + flags (3*16 int32 -> 256) + 3*16 partial sets * 5 chunks * (256+4) fp32
    assert L.wa_decode_ws_bytes(3, 16, 256, 1024, 1536) == 256 + 256 + 3 * 16 * 5 * 260 * 4
    # linear cache of 32768 keys: 128 chunks
    assert L.wa_decode_ws_bytes(64, 32, 256, 0, 32768) == 256 + 8192 + 64 * 32 * 128 * 260 * 4
    assert L.wa_decode_ws_bytes(1, 1, 128, 1, 1) == 256 + 256 + 132 * 4
    assert L.wa_decode_ws_bytes(0, 16, 256, 1024, 1536) == 0
    assert L.wa_decode_ws_bytes(3, 16, 64, 1024, 1536) == 0
    assert L.wa_decode_ws_bytes(3, 16, 256, 2000, 1536) == 0
    assert L.wa_prompt_ws_bytes(512, 16) == 256 + 512 * 16 * 4
    assert L.wa_prompt_ws_bytes(0, 16) == 0


def test_argument_errors_before_any_cuda_call():
    wa = ensure_built()
    L = wa.lib()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first
    E = wa.WA_EINVAL
    args = dict(q=fake, k=fake, v=fake, pos=fake, rows=3, hq=16, hkv=8, d=256, win=1024, ring=1536, scale=1.0,
                out=fake, ws=fake, ws_bytes=1 << 30, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return L.wa_decode(a["q"], a["k"], a["v"], a["pos"], a["rows"], a["hq"], a["hkv"], a["d"], a["win"],
                           a["ring"], a["scale"], a["out"], a["ws"], a["ws_bytes"], a["stream"])

    assert call(q=None) == E
    assert call(hq=12, hkv=8) == E            # not a multiple
    assert call(hq=34, hkv=2) == E            # group of 17 > 16
    assert call(d=192) == E
    assert call(win=-1) == E
    assert call(win=2000) == E                # window longer than the ring
    assert call(scale=float("nan")) == E
    assert call(q=ctypes.c_void_p((1 << 20) + 2)) == E   # misaligned
    assert call(ws=None) == wa.WA_EWORKSPACE
    assert call(ws_bytes=100) == wa.WA_EWORKSPACE

    def pcall(**kw):
        a = dict(q=fake, k=fake, v=fake, p0=1300, n=512, hi=None, hq=16, hkv=8, d=256, win=1024, ring=1536,
                 scale=1.0, p32=1, st=None, out=fake, ws=fake, ws_bytes=1 << 30, stream=None)
        a.update(kw)
        return L.wa_prompt(a["q"], a["k"], a["v"], a["p0"], a["n"], a["hi"], a["hq"], a["hkv"], a["d"], a["win"],
                           a["ring"], a["scale"], a["p32"], a["st"], a["out"], a["ws"], a["ws_bytes"], a["stream"])

    assert pcall(n=0) == E
    assert pcall(p0=-1) == E
    assert pcall(n=514) == E                  # 514 + 1023 keys do not fit a ring of 1536
    assert pcall(win=0, ring=1000) == E       # linear cache shorter than p0 + n
    assert pcall(p32=3) == E
    assert pcall(p32=-1) == E
    assert pcall(hq=48, hkv=2) == E


def test_prep_append_argument_errors_before_any_cuda_call():
    wa = ensure_built()
    L = wa.lib()
    fake = ctypes.c_void_p(1 << 20)
    E = wa.WA_EINVAL
    d, hq, hkv = 256, 16, 4

    def call(lay=None, **kw):
        a = dict(src=fake, pos=fake, n=8, hq=hq, hkv=hkv, d=d, mode=2, qs=None, inv=fake, ring=1536, q=fake, k=fake,
                 v=fake, ws=fake, ws_bytes=256, stream=None)
        a.update(kw)
        lay = lay or wa._PrepLayout((hq + 2 * hkv) * d, hq * d, 1536 * hkv * d, hkv * d)
        return L.wa_prep_append(a["src"], a["pos"], a["n"], a["hq"], a["hkv"], a["d"], a["mode"], a["qs"], a["inv"],
                                a["ring"], ctypes.byref(lay), a["q"], a["k"], a["v"], a["ws"], a["ws_bytes"],
                                a["stream"])

    assert call(src=None) == E
    assert call(mode=3) == E
    assert call(inv=None) == E                      # the RoPE needs its frequencies
    assert call(d=192) == E
    assert call(hq=12, hkv=8) == E
    assert call(ring=0) == E
    assert call(k=ctypes.c_void_p((1 << 20) + 8)) == E
    assert call(lay=wa._PrepLayout(100, hq * d, 0, hkv * d)) == E             # row shorter than the heads
    assert call(lay=wa._PrepLayout((hq + 2 * hkv) * d + 4, hq * d, 0, hkv * d)) == E   # not a multiple of 8
    assert call(ws=None) == wa.WA_EWORKSPACE
    assert call(ws_bytes=128) == wa.WA_EWORKSPACE


def test_prompt_sparse_argument_errors():
    wa = ensure_built()
    L = wa.lib()
    fake = ctypes.c_void_p(1 << 20)
    E = wa.WA_EINVAL

    def call(**kw):
        a = dict(p0=1300, n=512, hq=16, hkv=8, d=256, win=1024, ring=1536, p32=1, sel=fake, nsel=32, ws_bytes=1 << 30)
        a.update(kw)
        return L.wa_prompt_sparse(fake, fake, fake, a["p0"], a["n"], None, a["hq"], a["hkv"], a["d"], a["win"],
                                  a["ring"], 1.0, a["p32"], a["sel"], a["nsel"], None, fake, fake, a["ws_bytes"], None)

    assert call(sel=None) == E
    assert call(nsel=0) == E
    assert call(nsel=65) == E
    assert call(p32=3) == E
    assert call(win=0, ring=5_000_000, p0=0, n=4_500_000) == E   # key span over 65,536 blocks
    assert call(ws_bytes=8) == wa.WA_EWORKSPACE


def test_strerror_and_version():
    wa = ensure_built()
    L = wa.lib()
    assert L.wa_strerror(0) == b"ok"
    assert b"invalid" in L.wa_strerror(wa.WA_EINVAL)
    assert L.wa_version() >= 100


@pytest.mark.parametrize("name", ["decode", "prompt"])
def test_binding_raises_without_cuda_tensors(name):
    import torch
    wa = ensure_built()
    x = torch.zeros(2, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        if name == "decode":
            wa.decode(x, x, x, torch.zeros(2, dtype=torch.int32), 0)
        else:
            wa.prompt(x, x, x, 0)
