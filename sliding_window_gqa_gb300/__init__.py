"""Sliding-window grouped-query attention for one GB300 (sm_103a).

A thin ctypes binding of ``libwa.so`` (the C ABI declared in ``include/wa.h``):
it checks dtypes and devices, turns tensors into pointers and strides, and
calls the library on the current CUDA stream.  Every step of the attention
runs in the library's CUDA kernels; there is no Python or CPU fallback, and
calling an entry point without the built library raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

__all__ = [
    "WAError", "lib", "lib_path", "decode", "decode_static", "prompt", "prompt_sparse", "prep_append", "status",
    "decode_ws_bytes", "prompt_ws_bytes",
    "WA_OK", "WA_EINVAL", "WA_EWORKSPACE", "WA_ECUDA", "WA_EDEVICE",
    "WA_STATUS_BAD_POS", "WA_STATUS_BAD_HI", "WA_STATUS_TIMEOUT",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libwa.so")
_HEADER = os.path.join(os.path.dirname(_HERE), "include", "wa.h")


def _header_constants() -> dict:
    consts = {}
    with open(_HEADER) as f:
        for line in f:
            m = re.match(r"#define\s+(WA_\w+)\s+\(?(-?\d+)\)?", line)
            if m:
                consts[m.group(1)] = int(m.group(2))
    return consts


_C = _header_constants()
WA_OK = _C["WA_OK"]
WA_EINVAL = _C["WA_EINVAL"]
WA_EWORKSPACE = _C["WA_EWORKSPACE"]
WA_ECUDA = _C["WA_ECUDA"]
WA_EDEVICE = _C["WA_EDEVICE"]
WA_STATUS_BAD_POS = _C["WA_STATUS_BAD_POS"]
WA_STATUS_BAD_HI = _C["WA_STATUS_BAD_HI"]
WA_STATUS_TIMEOUT = _C["WA_STATUS_TIMEOUT"]


class WAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {lib().wa_strerror(code).decode()} ({code})")


class _Strides(ctypes.Structure):
    _fields_ = [("q", ctypes.c_int64), ("k", ctypes.c_int64), ("v", ctypes.c_int64), ("out", ctypes.c_int64)]


class _PrepLayout(ctypes.Structure):
    _fields_ = [("src_tok", ctypes.c_int64), ("q_tok", ctypes.c_int64), ("ring_row", ctypes.c_int64),
                ("slot", ctypes.c_int64)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int32


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(_LIB_PATH)
        L.wa_decode_ws_bytes.argtypes = [_I, _I, _I, _I, _I]
        L.wa_decode_ws_bytes.restype = ctypes.c_size_t
        L.wa_decode.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, ctypes.c_size_t, _P]
        L.wa_decode.restype = ctypes.c_int
        L.wa_decode_static.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P]
        L.wa_decode_static.restype = ctypes.c_int
        L.wa_prompt_ws_bytes.argtypes = [_I, _I]
        L.wa_prompt_ws_bytes.restype = ctypes.c_size_t
        L.wa_prompt.argtypes = [_P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _I, ctypes.c_float, _I,
                                ctypes.POINTER(_Strides), _P, _P, ctypes.c_size_t, _P]
        L.wa_prompt.restype = ctypes.c_int
        L.wa_prompt_sparse.argtypes = [_P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P, _I,
                                       ctypes.POINTER(_Strides), _P, _P, ctypes.c_size_t, _P]
        L.wa_prompt_sparse.restype = ctypes.c_int
        L.wa_prep_append.argtypes = [_P, _P, _I, _I, _I, _I, _I, _P, _P, _I, ctypes.POINTER(_PrepLayout),
                                     _P, _P, _P, _P, ctypes.c_size_t, _P]
        L.wa_prep_append.restype = ctypes.c_int
        L.wa_status.argtypes = [_P, _P]
        L.wa_status.restype = ctypes.c_int
        L.wa_strerror.argtypes = [ctypes.c_int]
        L.wa_strerror.restype = ctypes.c_char_p
        L.wa_version.argtypes = []
        L.wa_version.restype = ctypes.c_int
        _lib = L
    return _lib


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check_bf16(name: str, t: torch.Tensor) -> None:
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a bf16 CUDA tensor")


def decode_ws_bytes(rows: int, hq: int, d: int, win: int, ring: int) -> int:
    return int(lib().wa_decode_ws_bytes(rows, hq, d, win, ring))


def prompt_ws_bytes(n: int, hq: int) -> int:
    return int(lib().wa_prompt_ws_bytes(n, hq))


def _workspace(nbytes: int, device, ws):
    if ws is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or ws.device != device or not ws.is_contiguous():
        raise TypeError("ws must be a contiguous CUDA tensor on the inputs' device")
    return ws


def _ws_bytes(ws) -> int:
    return int(ws.numel() * ws.element_size())


def _same_device(device, **ts) -> None:
    for name, t in ts.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, the other inputs on {device}")


# Shape agreement between the tensors of one call.  The C ABI receives bare pointers and
# trusts these extents, so a mismatch here would become an out-of-bounds access there.

def _decode_shapes(q, k_ring, v_ring, pos, out):
    """(rows, hq, hkv, d, ring) of a decode call; ValueError if the tensors disagree."""
    if q.dim() != 3 or k_ring.dim() != 4:
        raise ValueError("q must be [rows, hq, d] and k_ring [rows, ring, hkv, d]")
    rows, hq, d = q.shape
    if k_ring.shape[0] != rows or k_ring.shape[3] != d:
        raise ValueError(f"k_ring {tuple(k_ring.shape)} does not match q {tuple(q.shape)}")
    if tuple(v_ring.shape) != tuple(k_ring.shape):
        raise ValueError(f"v_ring {tuple(v_ring.shape)} must have k_ring's shape {tuple(k_ring.shape)}")
    if pos.dim() != 1 or pos.numel() != rows or not pos.is_contiguous():
        raise ValueError(f"pos must be a contiguous vector of {rows} positions")
    if out is not None and (out.dtype != torch.bfloat16 or tuple(out.shape) != tuple(q.shape)
                            or not out.is_contiguous()):
        raise ValueError(f"out must be a contiguous bf16 tensor of q's shape {tuple(q.shape)}")
    return rows, hq, k_ring.shape[2], d, k_ring.shape[1]


def _prompt_shapes(q, k, v, hi, out):
    """(n, hq, hkv, d, ring) of a prompt call; ValueError if the tensors disagree."""
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q must be [n, hq, d] and k, v [ring, hkv, d]")
    n, hq, d = q.shape
    ring, hkv, dk = k.shape
    if dk != d:
        raise ValueError(f"k's head dim {dk} differs from q's {d}")
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"v {tuple(v.shape)} must have k's shape {tuple(k.shape)}")
    if hi is not None and (hi.dtype != torch.int32 or hi.dim() != 1 or hi.numel() != n or not hi.is_contiguous()):
        raise TypeError("hi must be None or a contiguous int32 tensor of n elements")
    if out is not None and (out.dtype != torch.bfloat16 or tuple(out.shape) != (n, hq, d)):
        raise ValueError(f"out must be a bf16 tensor of shape {(n, hq, d)}")
    return n, hq, hkv, d, ring


def _prep_shapes(src, pos, q_out, k_ring, v_ring):
    """(n, hq, hkv, d) of a preparation call; ValueError if the tensors disagree."""
    if src.dim() != 2 or q_out.dim() != 3 or k_ring.dim() not in (3, 4):
        raise ValueError("src must be [n, row], q_out [n, hq, d], k_ring [ring, hkv, d] or [n, ring, hkv, d]")
    n = src.shape[0]
    d = k_ring.shape[-1]
    hq, hkv = q_out.shape[1], k_ring.shape[-2]
    if q_out.shape[0] != n or q_out.shape[2] != d:
        raise ValueError(f"q_out {tuple(q_out.shape)} does not match {n} tokens of head dim {d}")
    if src.shape[1] < (hq + 2 * hkv) * d:
        raise ValueError(f"src rows hold {src.shape[1]} values, fewer than (hq + 2 hkv) d = {(hq + 2 * hkv) * d}")
    if k_ring.dim() == 4 and k_ring.shape[0] != n:
        raise ValueError(f"per-token rings: k_ring has {k_ring.shape[0]} rings for {n} tokens")
    if v_ring is not None and tuple(v_ring.shape) != tuple(k_ring.shape):
        raise ValueError(f"v_ring {tuple(v_ring.shape)} must have k_ring's shape {tuple(k_ring.shape)}")
    if pos.dim() != 1 or pos.numel() != n or not pos.is_contiguous():
        raise ValueError(f"pos must be a contiguous vector of {n} positions")
    return n, hq, hkv, d


def decode(q, k_ring, v_ring, pos, win: int, scale: float = 1.0, out=None, ws=None, stream=None):
    """Decode attention: q [rows,hq,d], k_ring/v_ring [rows,ring,hkv,d] (bf16, dense), pos int32 [rows].

    Returns out [rows,hq,d] bf16.  ``ws`` may be a reused uint8 CUDA buffer of
    at least decode_ws_bytes(...) bytes; the call is asynchronous on ``stream``."""
    for n_, t in (("q", q), ("k_ring", k_ring), ("v_ring", v_ring)):
        _check_bf16(n_, t)
        if not t.is_contiguous():
            raise ValueError(f"{n_} must be contiguous")
    if pos.dtype != torch.int32 or not pos.is_cuda:
        raise TypeError("pos must be an int32 CUDA tensor")
    rows, hq, hkv, d, ring = _decode_shapes(q, k_ring, v_ring, pos, out)
    _same_device(q.device, k_ring=k_ring, v_ring=v_ring, pos=pos, out=out)
    if out is None:
        out = torch.empty_like(q)
    nbytes = decode_ws_bytes(rows, hq, d, win, ring)
    ws = _workspace(nbytes, q.device, ws)
    rc = lib().wa_decode(q.data_ptr(), k_ring.data_ptr(), v_ring.data_ptr(), pos.data_ptr(), rows, hq, hkv, d,
                         win, ring, float(scale), out.data_ptr(), ws.data_ptr(), _ws_bytes(ws),
                         _stream_handle(stream))
    if rc != WA_OK:
        raise WAError(rc, "wa_decode")
    return out


def decode_static(q, k_ring, v_ring, pos, win: int, scale: float = 1.0, out=None, stream=None):
    """decode() without a workspace: the library's fixed device scratch (WA_STATIC_WS_BYTES a
    device) holds the partials, for callers that cannot allocate device memory.  Calls that
    may overlap on the GPU share that scratch and must be ordered by the caller; the status
    bits of the last call are status(None)."""
    for n_, t in (("q", q), ("k_ring", k_ring), ("v_ring", v_ring)):
        _check_bf16(n_, t)
        if not t.is_contiguous():
            raise ValueError(f"{n_} must be contiguous")
    if pos.dtype != torch.int32 or not pos.is_cuda:
        raise TypeError("pos must be an int32 CUDA tensor")
    rows, hq, hkv, d, ring = _decode_shapes(q, k_ring, v_ring, pos, out)
    _same_device(q.device, k_ring=k_ring, v_ring=v_ring, pos=pos, out=out)
    if out is None:
        out = torch.empty_like(q)
    rc = lib().wa_decode_static(q.data_ptr(), k_ring.data_ptr(), v_ring.data_ptr(), pos.data_ptr(), rows, hq, hkv,
                                d, win, ring, float(scale), out.data_ptr(), _stream_handle(stream))
    if rc != WA_OK:
        raise WAError(rc, "wa_decode_static")
    return out


def _token_stride(name: str, t: torch.Tensor, d: int) -> int:
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != d:
        raise ValueError(f"{name} must be [tokens, heads, d] with head stride d and unit dim stride")
    return int(t.stride(0))


def prompt(q, k, v, p0: int, hi=None, win: int = 0, scale: float = 1.0, p32=False,
           out=None, ws=None, stream=None):
    """Prompt attention for rows p0 .. p0+n-1: q [n,hq,d], k/v [ring,hkv,d] (bf16, token-strided).

    ``hi`` is None (each row's last key is its own position) or an int32 CUDA
    tensor [n].  ``p32``: False / 0 (one bf16 P), True / 1 (two parts) or 2 (three
    parts).  Returns out [n,hq,d] bf16."""
    for n_, t in (("q", q), ("k", k), ("v", v)):
        _check_bf16(n_, t)
    n, hq, hkv, d, ring = _prompt_shapes(q, k, v, hi, out)
    _same_device(q.device, k=k, v=v, hi=hi, out=out)
    if out is None:
        out = torch.empty((n, hq, d), dtype=torch.bfloat16, device=q.device)
    st = _Strides(_token_stride("q", q, d), _token_stride("k", k, d), _token_stride("v", v, d),
                  _token_stride("out", out, d))
    ws = _workspace(prompt_ws_bytes(n, hq), q.device, ws)
    rc = lib().wa_prompt(q.data_ptr(), k.data_ptr(), v.data_ptr(), int(p0), n,
                         None if hi is None else hi.data_ptr(), hq, hkv, d, int(win), ring, float(scale),
                         int(p32), ctypes.byref(st), out.data_ptr(), ws.data_ptr(), _ws_bytes(ws),
                         _stream_handle(stream))
    if rc != WA_OK:
        raise WAError(rc, "wa_prompt")
    return out


def prompt_sparse(q, k, v, p0: int, sel, hi=None, win: int = 0, scale: float = 1.0, p32=False,
                  out=None, ws=None, stream=None):
    """Block-sparse prompt: as prompt(), with sel an int32 CUDA tensor [n, hkv, nsel] of selected
    64-key blocks (-1 = unused).  Returns out [n,hq,d] bf16."""
    for n_, t in (("q", q), ("k", k), ("v", v)):
        _check_bf16(n_, t)
    n, hq, hkv, d, ring = _prompt_shapes(q, k, v, hi, out)
    if sel.dtype != torch.int32 or not sel.is_cuda or not sel.is_contiguous() or sel.dim() != 3 or \
            sel.shape[0] != n or sel.shape[1] != hkv:
        raise TypeError("sel must be a contiguous int32 CUDA tensor [n, hkv, nsel]")
    _same_device(q.device, k=k, v=v, hi=hi, sel=sel, out=out)
    if out is None:
        out = torch.empty((n, hq, d), dtype=torch.bfloat16, device=q.device)
    st = _Strides(_token_stride("q", q, d), _token_stride("k", k, d), _token_stride("v", v, d),
                  _token_stride("out", out, d))
    ws = _workspace(prompt_ws_bytes(n, hq), q.device, ws)
    rc = lib().wa_prompt_sparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), int(p0), n,
                                None if hi is None else hi.data_ptr(), hq, hkv, d, int(win), ring, float(scale),
                                int(p32), sel.data_ptr(), sel.shape[2], ctypes.byref(st), out.data_ptr(),
                                ws.data_ptr(), _ws_bytes(ws), _stream_handle(stream))
    if rc != WA_OK:
        raise WAError(rc, "wa_prompt_sparse")
    return out


_PREP_MODES = {"rmsnorm": _C["WA_PREP_RMSNORM"], "l2_rope": _C["WA_PREP_L2_ROPE"]}


def _ring_layout(name: str, t: torch.Tensor, d: int):
    """(ring, ring_row, slot) of a [ring, hkv, d] shared ring or [tokens, ring, hkv, d] per-token rings."""
    if t.stride(-1) != 1 or t.stride(-2) != d:
        raise ValueError(f"{name} must have head stride d and unit dim stride")
    if t.dim() == 3:
        return t.shape[0], 0, int(t.stride(0))
    if t.dim() == 4:
        return t.shape[1], int(t.stride(0)), int(t.stride(1))
    raise ValueError(f"{name} must be [ring, hkv, d] or [tokens, ring, hkv, d]")


def prep_append(src, pos, q_out, k_ring, v_ring=None, mode: str = "rmsnorm", q_scale=None, inv_freq=None,
                ws=None, stream=None):
    """q/k preparation and KV append.

    src [n, >= (hq + 2 hkv) d] bf16 projection rows (unit inner stride), pos int32 [n],
    q_out [n, hq, d] (token-strided), k_ring / v_ring [ring, hkv, d] (one shared ring) or
    [n, ring, hkv, d] (one ring per token).  v_ring None leaves v where it is.  mode "rmsnorm"
    or "l2_rope" (then inv_freq fp32 [d/2], q_scale fp32 [d] or None).  Returns the workspace,
    whose status wa_status / status() reads."""
    _check_bf16("src", src)
    _check_bf16("q_out", q_out)
    _check_bf16("k_ring", k_ring)
    if v_ring is not None:
        _check_bf16("v_ring", v_ring)
    if pos.dtype != torch.int32 or not pos.is_cuda:
        raise TypeError("pos must be an int32 CUDA tensor")
    if src.dim() != 2 or src.stride(1) != 1:
        raise ValueError("src must be [n, row] with unit inner stride")
    n, hq, hkv, d = _prep_shapes(src, pos, q_out, k_ring, v_ring)
    _same_device(src.device, pos=pos, q_out=q_out, k_ring=k_ring, v_ring=v_ring, q_scale=q_scale, inv_freq=inv_freq)
    ring, ring_row, slot = _ring_layout("k_ring", k_ring, d)
    if v_ring is not None and _ring_layout("v_ring", v_ring, d) != (ring, ring_row, slot):
        raise ValueError("v_ring must have k_ring's layout")
    for n_, t, cnt in (("q_scale", q_scale, d), ("inv_freq", inv_freq, d // 2)):
        if t is not None and (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.numel() != cnt):
            raise TypeError(f"{n_} must be a contiguous fp32 CUDA tensor of {cnt} elements")
    lay = _PrepLayout(int(src.stride(0)), _token_stride("q_out", q_out, d), ring_row, slot)
    ws = _workspace(256, src.device, ws)
    rc = lib().wa_prep_append(src.data_ptr(), pos.data_ptr(), n, hq, hkv, d, _PREP_MODES[mode],
                              None if q_scale is None else q_scale.data_ptr(),
                              None if inv_freq is None else inv_freq.data_ptr(), ring, ctypes.byref(lay),
                              q_out.data_ptr(), k_ring.data_ptr(), None if v_ring is None else v_ring.data_ptr(),
                              ws.data_ptr(), _ws_bytes(ws), _stream_handle(stream))
    if rc != WA_OK:
        raise WAError(rc, "wa_prep_append")
    return ws


def status(ws, stream=None) -> int:
    """WA_STATUS_* bits of the last call on ``ws`` (waits for the stream); ``ws`` None reads those
    of the last decode_static call on the current device."""
    rc = lib().wa_status(None if ws is None else ws.data_ptr(), _stream_handle(stream))
    if rc < 0:
        raise WAError(rc, "wa_status")
    return rc
