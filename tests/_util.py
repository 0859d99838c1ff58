"""Helpers shared by the tests: the built library, bit views, oracle comparison."""
from __future__ import annotations

import os
import threading

import numpy as np
import torch

import oracle
from oracle import check

_lock = threading.Lock()


def ensure_built():
    """Import the binding, building libwa.so first if it is missing."""
    import sliding_window_gqa_gb300 as wa
    with _lock:
        if not os.path.exists(wa.lib_path()):
            from sliding_window_gqa_gb300 import build
            build.build()
    wa.lib()
    return wa


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_parity(got: torch.Tensor, ref: np.ndarray, tol: float, what: str = "") -> dict:
    r = check.compare(bits(got), ref, tol)
    assert r["ok"], f"{what}: {r}"
    return r


def decode_ref(c, rows=None, heads=None, scale=1.0):
    pos = c["pos"].cpu().numpy()
    if rows is None:
        return oracle.decode(bits(c["q"]), bits(c["k"]), bits(c["v"]), pos, c["win"], c["ring"], scale, heads=heads)
    q = bits(c["q"][rows])
    k = bits(c["k"][rows])
    v = bits(c["v"][rows])
    return oracle.decode(q, k, v, pos[rows], c["win"], c["ring"], scale, heads=heads)
