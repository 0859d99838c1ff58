#!/usr/bin/env python3
"""Throughput of the sliding-window GQA hot path on GB300, as a fraction of the roofline.

One step runs the whole path once over a fixed synthetic workload, shaped like
the pages' workloads (TensorFold pull request #1123, "Receipt"; the "Exact
Numerical Contract" page, "Canonical Boundary"):

  decode_sliding  3 independent caches x 64 rows, 32/16 heads, d 256, window 1024
                  over a ring of 1536, positions uniform to 40,000, three streams
  decode_linear   64 rows, 32/16 heads, d 256, linear cache of 32,768 keys
  prompt_causal   8,192 rows at p0 0, 16/8 heads, d 256, linear cache, causal, P32
  prompt_dense    37,810 rows, 56 heads (MHA), d 128, interleaved QKV (row 21,504),
                  RMSNormed Q/K, scale 1/sqrt(128), non-causal (hi = N-1), bf16 P
  prompt_dense_p32  the same workload with P as two bf16 parts (the page leaves the
                  dense workload's P precision open, so it is timed both ways)

The "next" parts run after the step, each timed the same way but outside the
step and its value (they are not the headline workloads): decode_gqa8
(decode_sliding with 32 query heads over 4 key heads) and decode_gqa16_linear
(decode_linear with 32 over 2), the groups the tensor-core decode serves;
prep_dense, the dense workload's q/k preparation (per-head RMSNorm of Q and K in
place in the interleaved QKV buffer, 37,810 tokens, 56 heads, d 128), HBM-bound;
and prompt_sparse, the block-sparse prompt of TensorFold #1622's shapes: 7,936
causal rows, 24/2 heads, d 256, each row's 2,048 selected keys as 32 blocks of 64,
three-part P, whose flops count the visible selected keys only.  --next none
skips them.

value = (decode bytes / HBM peak + prompt flops / bf16 peak) / measured step time:
the step's roofline time over its measured time.  Decode bytes are the visible
K and V rows plus q and out; prompt flops are 4*d per visible (row, key, head).
Peaks come from MEASURED_PEAKS.json: the copy bandwidth and the burst bf16
figure, since each part is timed alone by CUDA events around its own calls (the
sustained figure is reported beside it).

Each part's calls are captured once in a CUDA graph and replayed in the timed region (the
three-stream parts fork and join inside it), as a serving loop would; the e2e leg calls the C
ABI eagerly with host copies.

Prints one JSON line.  --impl reference times the float64 oracle on the host
cores on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode KV-read GB/s and prompt attention TFLOP/s, as fraction of GB300 roofline"
UNIT = "fraction of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s nominal figure, printed beside the measured-copy fraction

PARTS = ("decode_sliding", "decode_linear", "prompt_causal", "prompt_dense", "prompt_dense_p32")
EXTRA_PARTS = ("decode_gqa8", "decode_gqa16_linear", "prep_dense", "prompt_sparse")
SPEC = {
    "decode_sliding": dict(caches=3, rows=64, hq=32, hkv=16, d=256, win=1024, ring=1536, pos_max=40000,
                           seed=20260003),
    "decode_linear": dict(rows=64, hq=32, hkv=16, d=256, win=0, ring=32768, seed=20260004),
    "prompt_causal": dict(n=8192, p0=0, hq=16, hkv=8, d=256, win=0, ring=8192, p32=True, seed=20260005),
    "prompt_dense": dict(N=37810, H=56, d=128, p32=False, seed=20260006),
    "prompt_dense_p32": dict(N=37810, H=56, d=128, p32=True, seed=20260006),
    "decode_gqa8": dict(caches=3, rows=64, hq=32, hkv=4, d=256, win=1024, ring=1536, pos_max=40000,
                        seed=20260007),
    "decode_gqa16_linear": dict(rows=64, hq=32, hkv=2, d=256, win=0, ring=32768, seed=20260008),
    "prep_dense": dict(N=37810, H=56, d=128, seed=20260009),
    "prompt_sparse": dict(n=7936, p0=0, hq=24, hkv=2, d=256, win=0, ring=7936, nsel=32, p32=2, seed=20260010),
}

# ncu DRAM bytes per launch of the dominant kernels, valid only while the kernel source is unchanged.
TRAFFIC = {
    "prompt_dense": {"bytes_per_launch": 2057 * 10**6, "source_sha": "68921256d3482bf8",
                     "note": "ncu at N=8192 (352.5 MB read + 93.1 MB write), scaled by N to 37,810"},
    "prompt_dense_p32": {"bytes_per_launch": 2058 * 10**6, "source_sha": "68921256d3482bf8",
                         "note": "ncu at N=8192 (352.6 MB read + 93.3 MB write), scaled by N to 37,810"},
    "prompt_causal": {"bytes_per_launch": 214 * 10**6, "source_sha": "d1f5adac0ed541b3",
                      "note": "ncu of the full launch (187.1 MB read + 26.6 MB write)"},
    "decode_gqa8": {"bytes_per_launch": 853 * 10**6, "source_sha": "2033d7ed7d9eaec4",
                    "note": "the part's three launches together, like its achieved figure: ncu at 256 rows, one cache "
                            "(1.134 GB read + 8.0 MB write for 1.072 GB algorithmic), scaled by algorithmic bytes "
                            "to the part's 801 MB"},
}


# ----------------------------------------------------------------------------- work accounting

def decode_positions(part: str):
    import torch
    s = SPEC[part]
    g = torch.Generator().manual_seed(s["seed"])
    if "caches" in s:
        out = []
        for _ in range(s["caches"]):
            p = torch.randint(0, s["pos_max"] + 1, (s["rows"],), generator=g).tolist()
            p[0] = s["pos_max"]
            out.append(p)
        return out
    p = torch.randint(0, s["ring"], (s["rows"],), generator=g).tolist()
    p[5] = s["ring"] - 1
    return [p]


def visible(p: int, win: int) -> int:
    lo = max(0, p - win + 1) if win > 0 else 0
    return p - lo + 1


def decode_bytes(pos, hq, hkv, d, win) -> int:
    """K and V rows each row reads (hkv * visible * d * 2 bytes, twice) plus q and out."""
    kv = sum(hkv * visible(p, win) * d * 2 * 2 for p in pos)
    return kv + 2 * len(pos) * hq * d * 2


def prompt_flops_rows(rows, p0, win, hi_of, hq, d) -> int:
    """4*d flops (2d for q.k, 2d for p.v) per visible (row, key, head)."""
    tot = 0
    for i in rows:
        p = p0 + i
        lo = max(0, p - win + 1) if win > 0 else 0
        tot += hi_of(i) - lo + 1
    return tot * hq * 4 * d


_SEL_CACHE: dict = {}


def sparse_selection_of(s):
    """The part's synthetic block selection [n, hkv, nsel] (CPU int32), generated once."""
    import wa_synth
    key = (s["n"], s["p0"], s["hkv"], s["nsel"], s["seed"], s["win"])
    if key not in _SEL_CACHE:
        _SEL_CACHE[key] = wa_synth.sparse_selection(s["n"], s["p0"], s["hkv"], s["nsel"], seed=s["seed"], win=s["win"])
    return _SEL_CACHE[key]


def sparse_visible_keys(s):
    """Visible selected keys per (row, key head): blocks counted once, cut to [lo, p]."""
    import numpy as np
    sel = sparse_selection_of(s).numpy().astype(np.int64)
    n = s["n"]
    p = (s["p0"] + np.arange(n))[:, None, None]
    lo = np.maximum(0, p - s["win"] + 1) if s["win"] > 0 else np.zeros_like(p)
    srt = np.sort(sel, axis=2)
    first = np.ones_like(srt, dtype=bool)
    first[:, :, 1:] = srt[:, :, 1:] != srt[:, :, :-1]
    a = np.maximum(lo, srt * 64)
    e = np.minimum(p, srt * 64 + 63)
    cnt = np.where((srt >= 0) & first & (e >= a), e - a + 1, 0)
    return cnt.sum(axis=2)


def part_work(part: str):
    s = SPEC[part]
    if part.startswith("decode"):
        return {"bytes": sum(decode_bytes(p, s["hq"], s["hkv"], s["d"], s["win"]) for p in decode_positions(part)),
                "flops": 0}
    if part == "prompt_sparse":
        vis = sparse_visible_keys(s)
        return {"bytes": 0, "flops": int(vis.sum()) * (s["hq"] // s["hkv"]) * 4 * s["d"],
                "issued_flops_factor": 2.0 if s["p32"] == 2 else (1.5 if s["p32"] else 1.0)}
    if part == "prep_dense":
        # Q and K heads read once and written once (V stays in place)
        return {"bytes": 2 * s["N"] * 2 * s["H"] * s["d"] * 2, "flops": 0}
    if part == "prompt_causal":
        n = s["n"]
        vis = n * (n + 1) // 2          # row i sees keys 0..i
        return {"bytes": 0, "flops": vis * s["hq"] * 4 * s["d"], "issued_flops_factor": 1.5 if s["p32"] else 1.0}
    N = s["N"]
    return {"bytes": 0, "flops": N * N * s["H"] * 4 * s["d"], "issued_flops_factor": 1.5 if s["p32"] else 1.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def roofline_seconds(parts, pk) -> float:
    """Seconds the parts' algorithmic work takes at the peaks: bytes at the copy bandwidth, flops at
    the burst bf16 rate (each part is timed alone, by CUDA events around its own calls)."""
    t = 0.0
    for part in parts:
        w = part_work(part)
        t += w["bytes"] / (pk["hbm_gbs"] * 1e9) + w["flops"] / (pk["bf16_tflops"] * 1e12)
    return t


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for nm, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- native arm

class Part:
    """One part of the step.  calls(stream) makes the part's C-ABI calls; in the timed region they
    are replayed as a CUDA graph captured after one eager call, so the GPU time does not include the
    host's per-call work (argument checks, tensor-map encoding).  The e2e leg calls them eagerly."""
    name = ""
    launches = 0
    graph = None

    def calls(self, stream):
        raise NotImplementedError

    def timed_calls(self, stream):
        torch = self.torch
        if self.graph is None:
            self.calls(stream)                      # eager once: device attributes, encoder lookup
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream()
            cap.wait_stream(stream)
            with torch.cuda.graph(g, stream=cap):
                self.calls(cap)
            stream.wait_stream(cap)
            self.graph = g
            return
        self.graph.replay()

    def run(self, stream, host=None):
        if host is not None:
            self.copy_in(host)
            self.k_start.record(stream)
            self.calls(stream)
            self.k_end.record(stream)
            self.copy_out(host)
            return
        self.k_start.record(stream)
        self.timed_calls(stream)
        self.k_end.record(stream)

    def collect(self):
        self.kernel_ms.append(self.k_start.elapsed_time(self.k_end))

    h2d_stream = None   # the e2e leg's one host-to-device copy stream, shared by every part

    def h2d(self, dst, src):
        """dst <- src (pinned host).  The copy goes on the shared copy stream, after the work already
        queued on the current stream, and the current stream waits for it: every part's inputs come
        in one after another, in the order the parts are issued, at the link's full rate."""
        torch = self.torch
        cur = torch.cuda.current_stream()
        cs = Part.h2d_stream
        if cs is None:
            dst.copy_(src, non_blocking=True)
            return
        ready = torch.cuda.Event()
        ready.record(cur)
        cs.wait_event(ready)
        with torch.cuda.stream(cs):
            dst.copy_(src, non_blocking=True)
        done = torch.cuda.Event()
        done.record(cs)
        cur.wait_event(done)


def _events(torch, stream, n=2):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


class DecodeSliding(Part):
    name = "decode_sliding"

    def __init__(self, torch, wa, wa_synth, dev):
        s = SPEC[self.name]
        self.torch, self.wa = torch, wa
        self.cases, self.outs, self.ws = [], [], []
        for i, pos in enumerate(decode_positions(self.name)):
            c = wa_synth.decode_case(s["rows"], s["hq"], s["hkv"], s["d"], s["win"], s["ring"], pos,
                                     seed=s["seed"] * 10 + i, device=dev, outside="keep")
            self.cases.append(c)
            self.outs.append(torch.empty_like(c["q"]))
            self.ws.append(torch.empty(wa.decode_ws_bytes(s["rows"], s["hq"], s["d"], s["win"], s["ring"]),
                                       dtype=torch.uint8, device=dev))
        self.streams = [torch.cuda.Stream(device=dev) for _ in self.cases]
        self.launches = 3 * len(self.cases)   # partial, merge, float64 re-run per cache
        self.start_ev = torch.cuda.Event(enable_timing=True)
        self.join_ev = torch.cuda.Event(enable_timing=True)
        self.end_evs = [torch.cuda.Event() for _ in self.cases]
        self.kernel_ms = []
        self.graph = None

    def _capture(self):
        """The three calls, forked to their streams and joined back, as one CUDA graph: a replay
        starts all three at once, as a serving loop would, instead of one host call after another."""
        torch, wa, s = self.torch, self.wa, SPEC[self.name]
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap):
            fork = torch.cuda.Event()
            fork.record(cap)
            for i, (c, st) in enumerate(zip(self.cases, self.streams)):
                st.wait_event(fork)
                with torch.cuda.stream(st):
                    wa.decode(c["q"], c["k"], c["v"], c["pos"], s["win"], 1.0, out=self.outs[i], ws=self.ws[i],
                              stream=st)
                done = torch.cuda.Event()
                done.record(st)
                cap.wait_event(done)
        torch.cuda.current_stream().wait_stream(cap)
        self.graph = g

    def run(self, stream, host=None):
        torch, wa, s = self.torch, self.wa, SPEC[self.name]
        if host is None and self.graph is not None:
            self.start_ev.record(stream)
            self.graph.replay()
            self.join_ev.record(stream)
            return
        self.start_ev.record(stream)
        for i, (c, st) in enumerate(zip(self.cases, self.streams)):
            st.wait_event(self.start_ev)
            with torch.cuda.stream(st):
                if host is not None:
                    for key in ("q", "k", "v", "pos"):
                        self.h2d(c[key], host[i][key])
                wa.decode(c["q"], c["k"], c["v"], c["pos"], s["win"], 1.0, out=self.outs[i], ws=self.ws[i], stream=st)
                if host is not None:
                    host[i]["out"].copy_(self.outs[i], non_blocking=True)
            self.end_evs[i].record(st)
            stream.wait_event(self.end_evs[i])
        self.join_ev.record(stream)
        if host is None and self.graph is None:
            self._capture()   # after one eager call (device attributes, tensor-map encoder)

    def collect(self):
        # wall time of the three concurrent calls, from the fork to the join on the main stream
        self.kernel_ms.append(self.start_ev.elapsed_time(self.join_ev))

    def host_buffers(self):
        hb = []
        for c, o in zip(self.cases, self.outs):
            d = {k: c[k].cpu().pin_memory() for k in ("q", "k", "v", "pos")}
            d["out"] = torch_empty_pinned_like(o)
            hb.append(d)
        return hb


def torch_empty_pinned_like(t):
    import torch
    return torch.empty(t.shape, dtype=t.dtype, pin_memory=True)


class DecodeLinear(Part):
    name = "decode_linear"

    def __init__(self, torch, wa, wa_synth, dev):
        s = SPEC[self.name]
        self.torch, self.wa = torch, wa
        pos = decode_positions(self.name)[0]
        self.c = wa_synth.decode_case(s["rows"], s["hq"], s["hkv"], s["d"], s["win"], s["ring"], pos,
                                      seed=s["seed"], device=dev, outside="keep")
        self.out = torch.empty_like(self.c["q"])
        self.ws = torch.empty(wa.decode_ws_bytes(s["rows"], s["hq"], s["d"], s["win"], s["ring"]),
                              dtype=torch.uint8, device=dev)
        self.launches = 3
        self.k_start, self.k_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.kernel_ms = []

    def calls(self, stream):
        s, c = SPEC[self.name], self.c
        self.wa.decode(c["q"], c["k"], c["v"], c["pos"], s["win"], 1.0, out=self.out, ws=self.ws, stream=stream)

    def copy_in(self, host):
        for key in ("q", "k", "v", "pos"):
            self.h2d(self.c[key], host[key])

    def copy_out(self, host):
        host["out"].copy_(self.out, non_blocking=True)

    def host_buffers(self):
        d = {k: self.c[k].cpu().pin_memory() for k in ("q", "k", "v", "pos")}
        d["out"] = torch_empty_pinned_like(self.out)
        return d


class PromptCausal(Part):
    name = "prompt_causal"

    def __init__(self, torch, wa, wa_synth, dev):
        s = SPEC[self.name]
        self.torch, self.wa = torch, wa
        self.c = wa_synth.prompt_case(s["n"], s["p0"], s["hq"], s["hkv"], s["d"], s["win"], s["ring"],
                                      seed=s["seed"], device=dev, outside="keep")
        self.out = torch.empty_like(self.c["q"])
        self.ws = torch.empty(wa.prompt_ws_bytes(s["n"], s["hq"]), dtype=torch.uint8, device=dev)
        self.launches = 2   # prompt kernel, float64 re-run
        self.k_start, self.k_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.kernel_ms = []

    def calls(self, stream):
        s, c = SPEC[self.name], self.c
        self.wa.prompt(c["q"], c["k"], c["v"], s["p0"], None, s["win"], 1.0, p32=s["p32"], out=self.out, ws=self.ws,
                       stream=stream)

    def copy_in(self, host):
        for key in ("q", "k", "v"):
            self.h2d(self.c[key], host[key])

    def copy_out(self, host):
        host["out"].copy_(self.out, non_blocking=True)

    def host_buffers(self):
        d = {k: self.c[k].cpu().pin_memory() for k in ("q", "k", "v")}
        d["out"] = torch_empty_pinned_like(self.out)
        return d


class PromptDense(Part):
    name = "prompt_dense"

    def __init__(self, torch, wa, wa_synth, dev):
        s = SPEC[self.name]
        self.torch, self.wa = torch, wa
        self.c = wa_synth.dense_qkv_case(s["N"], s["H"], s["d"], seed=s["seed"], device=dev)
        self.hi = torch.full((s["N"],), s["N"] - 1, dtype=torch.int32, device=dev)
        self.out = torch.empty((s["N"], s["H"], s["d"]), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(wa.prompt_ws_bytes(s["N"], s["H"]), dtype=torch.uint8, device=dev)
        self.launches = 2
        self.k_start, self.k_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.kernel_ms = []

    def calls(self, stream):
        s, c = SPEC[self.name], self.c
        self.wa.prompt(c["q"], c["k"], c["v"], 0, self.hi, 0, c["scale"], p32=s["p32"], out=self.out, ws=self.ws,
                       stream=stream)

    def copy_in(self, host):
        self.h2d(self.c["qkv"], host["qkv"])
        self.h2d(self.hi, host["hi"])

    def copy_out(self, host):
        host["out"].copy_(self.out, non_blocking=True)

    def host_buffers(self):
        return {"qkv": self.c["qkv"].cpu().pin_memory(), "hi": self.hi.cpu().pin_memory(),
                "out": torch_empty_pinned_like(self.out)}


class PrepDense(Part):
    name = "prep_dense"

    def __init__(self, torch, wa, wa_synth, dev):
        s = SPEC[self.name]
        self.torch, self.wa = torch, wa
        N, H, d = s["N"], s["H"], s["d"]
        W = 3 * H * d
        g = torch.Generator(device=dev).manual_seed(s["seed"])
        self.qkv = torch.randn((N, W), generator=g, device=dev).to(torch.bfloat16)   # projection rows
        self.q = self.qkv.as_strided((N, H, d), (W, d, 1), 0)
        self.k = self.qkv.as_strided((N, H, d), (W, d, 1), H * d)
        self.pos = torch.arange(N, dtype=torch.int32, device=dev)
        self.ws = torch.empty(256, dtype=torch.uint8, device=dev)
        self.launches = 1
        self.k_start, self.k_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.kernel_ms = []

    def calls(self, stream):
        self.wa.prep_append(self.qkv, self.pos, self.q, self.k, None, mode="rmsnorm", ws=self.ws, stream=stream)

    def copy_in(self, host):
        self.h2d(self.qkv, host["qkv"])

    def copy_out(self, host):
        host["out"].copy_(self.qkv, non_blocking=True)

    def host_buffers(self):
        return {"qkv": self.qkv.cpu().pin_memory(), "out": torch_empty_pinned_like(self.qkv)}


class PromptSparse(Part):
    name = "prompt_sparse"

    def __init__(self, torch, wa, wa_synth, dev):
        s = SPEC[self.name]
        self.torch, self.wa = torch, wa
        self.c = wa_synth.prompt_case(s["n"], s["p0"], s["hq"], s["hkv"], s["d"], s["win"], s["ring"],
                                      seed=s["seed"], device=dev, outside="keep")
        self.sel = sparse_selection_of(s).to(dev)
        self.out = torch.empty_like(self.c["q"])
        self.ws = torch.empty(wa.prompt_ws_bytes(s["n"], s["hq"]), dtype=torch.uint8, device=dev)
        self.launches = 2   # sparse prompt kernel, float64 re-run
        self.k_start, self.k_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.kernel_ms = []

    def calls(self, stream):
        s, c = SPEC[self.name], self.c
        self.wa.prompt_sparse(c["q"], c["k"], c["v"], s["p0"], self.sel, None, s["win"], 1.0, p32=s["p32"],
                              out=self.out, ws=self.ws, stream=stream)

    def copy_in(self, host):
        for key in ("q", "k", "v"):
            self.h2d(self.c[key], host[key])
        self.h2d(self.sel, host["sel"])

    def copy_out(self, host):
        host["out"].copy_(self.out, non_blocking=True)

    def host_buffers(self):
        d = {k: self.c[k].cpu().pin_memory() for k in ("q", "k", "v")}
        d["sel"] = self.sel.cpu().pin_memory()
        d["out"] = torch_empty_pinned_like(self.out)
        return d


class PromptDenseP32(PromptDense):
    name = "prompt_dense_p32"


class DecodeGqa8(DecodeSliding):
    name = "decode_gqa8"


class DecodeGqa16Linear(DecodeLinear):
    name = "decode_gqa16_linear"


PART_CLASSES = {"decode_sliding": DecodeSliding, "decode_linear": DecodeLinear,
                "prompt_causal": PromptCausal, "prompt_dense": PromptDense, "prompt_dense_p32": PromptDenseP32,
                "decode_gqa8": DecodeGqa8, "decode_gqa16_linear": DecodeGqa16Linear, "prep_dense": PrepDense,
                "prompt_sparse": PromptSparse}

KERNEL_OF = {"decode_sliding": "decode partial (wa_decode.cu)", "decode_linear": "decode partial (wa_decode.cu)",
             "prompt_causal": "prompt tensor-core tile, 128-key tiles (wa_prompt_d256.cuh)",
             "prompt_dense": "prompt tensor-core tiles, two query tiles a CTA (wa_prompt_pair.cuh)",
             "prompt_dense_p32": "prompt tensor-core tiles, two query tiles a CTA, two P parts (wa_prompt_pair.cuh)",
             "decode_gqa8": "tensor-core decode partial (wa_decode_tc.cu)",
             "decode_gqa16_linear": "tensor-core decode partial (wa_decode_tc.cu)",
             "prep_dense": "q/k preparation (wa_prep.cu)",
             "prompt_sparse": "block-sparse prompt tile (wa_prompt_sparse.cu)"}
SOURCE_OF = {"decode_sliding": "wa_decode.cu", "decode_linear": "wa_decode.cu",
             "prompt_causal": "wa_prompt_d256.cuh", "prompt_dense": "wa_prompt_pair.cuh",
             "prompt_dense_p32": "wa_prompt_pair.cuh",
             "decode_gqa8": "wa_decode_tc.cu", "decode_gqa16_linear": "wa_decode_tc.cu",
             "prep_dense": "wa_prep.cu", "prompt_sparse": "wa_prompt_kernel.cuh"}


def source_hash(fname: str) -> str:
    p = os.path.join(ROOT, "sliding_window_gqa_gb300", "csrc", fname)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def io_bytes(obj) -> int:
    import torch
    if isinstance(obj, torch.Tensor):
        return obj.numel() * obj.element_size()
    if isinstance(obj, dict):
        return sum(io_bytes(v) for v in obj.values())
    if isinstance(obj, (list, tuple)):
        return sum(io_bytes(v) for v in obj)
    return 0


# Pinned host-to-device rate on the GB300 machines (measured: ~211 GB/s on one stream, the same on
# several).  It only splits the parts into "copy shorter than kernel" and the rest.
H2D_GBS = 200.0


def johnson_order(copy_ms, kernel_ms):
    """Johnson's rule (1954) for two machines in series: jobs whose first stage is shorter than
    their second go first, by first stage ascending; the others after, by second stage
    descending.  Returns job indices."""
    n = len(copy_ms)
    first = sorted((i for i in range(n) if copy_ms[i] < kernel_ms[i]), key=lambda i: copy_ms[i])
    last = sorted((i for i in range(n) if copy_ms[i] >= kernel_ms[i]), key=lambda i: -kernel_ms[i])
    return first + last


def reduce_max(x: float, dist, device) -> float:
    """The maximum of x over all ranks (the slowest rank sets the time); x itself with one rank."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(t_roof_s: float, ms_per_step: float, world: int) -> float:
    """Whole-job fraction of roofline: every rank runs its own copy of the workload (no data exchange),
    so the job does world x the roofline work in the slowest rank's time."""
    return t_roof_s * world / (ms_per_step * 1e-3)


def run_native(args, parts, rank, world, dist):
    import torch

    import sliding_window_gqa_gb300 as wa
    import wa_synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wa.lib()
    objs = [PART_CLASSES[p](torch, wa, wa_synth, dev) for p in parts]
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step(host=None):
        for i, o in enumerate(objs):
            o.run(stream, None if host is None else host[i])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for o in objs:
        o.kernel_ms = []

    def barrier():
        if dist is not None:
            dist.barrier()

    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step()
        torch.cuda.synchronize()      # per-step event reads; the region stays GPU-timed end to end
        for o in objs:
            o.collect()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    total_ms = reduce_max(t_start.elapsed_time(t_end), dist, dev)
    ms_per_step = total_ms / args.steps

    # e2e: the same step through the C ABI with host buffers (H2D of inputs, D2H of outputs each
    # step).  The parts are independent, so each runs on a stream of its own: one part's kernels
    # overlap the next parts' host copies, and every step still copies all its inputs in and all
    # its results out.  All inputs come in on one copy stream, part after part, in the order that
    # minimises the span of a two-stage flow shop (copy, then kernel; Johnson's rule).
    e2e = None
    if not args.no_e2e:
        host = [o.host_buffers() for o in objs]
        part_streams = [torch.cuda.Stream(device=dev) for _ in objs]
        in_bytes = [io_bytes({k: v for k, v in h.items() if k != "out"}) if isinstance(h, dict)
                    else sum(io_bytes({k: v for k, v in x.items() if k != "out"}) for x in h) for h in host]
        e2e_order = johnson_order([b / (H2D_GBS * 1e6) for b in in_bytes],
                                  [statistics.median(o.kernel_ms) for o in objs])
        Part.h2d_stream = torch.cuda.Stream(device=dev)

        def step_e2e():
            fork = torch.cuda.Event()
            fork.record(stream)
            for i in e2e_order:
                o, ps, h = objs[i], part_streams[i], host[i]
                ps.wait_event(fork)
                with torch.cuda.stream(ps):
                    o.run(ps, h)
                done = torch.cuda.Event()
                done.record(ps)
                stream.wait_event(done)

        torch.cuda.synchronize()
        step_e2e()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ksteps = max(1, min(args.steps, args.e2e_steps))
        e0.record(stream)
        for _ in range(ksteps):
            step_e2e()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = reduce_max(e0.elapsed_time(e1) / ksteps, dist, dev)
        h2d = sum(io_bytes({k: v for k, v in h.items() if k != "out"}) if isinstance(h, dict)
                  else sum(io_bytes({k: v for k, v in x.items() if k != "out"}) for x in h) for h in host)
        d2h = sum(io_bytes(h["out"]) if isinstance(h, dict) else sum(io_bytes(x["out"]) for x in h) for h in host)
        e2e = {"ms_per_step": e_ms, "steps": ksteps, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "order": [objs[i].name for i in e2e_order]}
        Part.h2d_stream = None
        del host
    per_part_ms = {o.name: statistics.median(o.kernel_ms) for o in objs}
    launches = sum(o.launches for o in objs) * args.steps
    del objs
    nxt = time_next_parts(args, torch, wa, wa_synth, dev, stream) if args.next_parts else None
    return ms_per_step, per_part_ms, clk, e2e, launches, nxt


def time_next_parts(args, torch, wa, wa_synth, dev, stream):
    """The "next" parts, one after another: W warm-up calls, then K calls each timed by CUDA events
    on the launching stream (graph replays, as in the step), with clocks sampled meanwhile."""
    out = {}
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    for name in args.next_parts:
        o = PART_CLASSES[name](torch, wa, wa_synth, dev)
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            o.run(stream)
        torch.cuda.synchronize()
        o.kernel_ms = []
        for _ in range(args.steps):
            o.run(stream)
            torch.cuda.synchronize()
            o.collect()
        out[name] = {"ms": statistics.median(o.kernel_ms), "launches": o.launches * args.steps}
        del o
        torch.cuda.empty_cache()
    out["clocks"] = clocks.stop()
    return out


# ----------------------------------------------------------------------------- oracle (CPU) arm

_SAMPLES: dict = {}


def _sample_inputs(part: str, i: int = 0):
    """Host inputs for the oracle sample of a part, generated once and reused across steps."""
    import numpy as np
    import torch

    import wa_synth

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    key = (part, i)
    if key not in _SAMPLES:
        s = SPEC[part]
        if part.startswith("decode"):
            p = [q for ps in decode_positions(part) for q in ps][i]
            c = wa_synth.decode_case(1, s["hq"], s["hkv"], s["d"], s["win"], s["ring"], [p],
                                     seed=s["seed"] + i, outside="keep", peaked=False)
            _SAMPLES[key] = (p, bits(c["q"]), bits(c["k"]), bits(c["v"]))
        elif part == "prompt_sparse":
            c = wa_synth.prompt_case(s["n"], s["p0"], s["hq"], s["hkv"], s["d"], s["win"], s["ring"], seed=s["seed"],
                                     outside="keep", peaked=False)
            _SAMPLES[key] = (bits(c["q"]), bits(c["k"]), bits(c["v"]), sparse_selection_of(s).numpy())
        elif part == "prep_dense":
            g = torch.Generator().manual_seed(s["seed"])
            x = torch.randn((1024, 3 * s["H"] * s["d"]), generator=g).to(torch.bfloat16)
            _SAMPLES[key] = (bits(x),)
        elif part == "prompt_causal":
            c = wa_synth.prompt_case(s["n"], s["p0"], s["hq"], s["hkv"], s["d"], s["win"], s["ring"], seed=s["seed"],
                                     outside="keep", peaked=False)
            _SAMPLES[key] = (bits(c["q"]), bits(c["k"]), bits(c["v"]))
        else:
            c = wa_synth.dense_qkv_case(s["N"], 2, s["d"], seed=s["seed"])   # 2 of the heads: same per-head work
            _SAMPLES[key] = (bits(c["q"]), bits(c["k"]), bits(c["v"]), c["scale"])
    return _SAMPLES[key]


def oracle_sample(parts, budget_s: float):
    """Times the float64 oracle on a bounded sample of each part and extrapolates to the full part by work.

    Only the oracle calls are timed; the sample inputs are generated once and reused.
    Returns (seconds for the full workload, description)."""
    import numpy as np

    import oracle

    per = budget_s / max(1, len(parts))
    total, desc = 0.0, []
    for part in parts:
        s = SPEC[part]
        w = part_work(part)
        if part.startswith("decode"):
            n_rows = sum(len(ps) for ps in decode_positions(part))
            rows_done, work_done, t_used = 0, 0, 0.0
            while t_used < per and rows_done < n_rows:
                p, q, k, v = _sample_inputs(part, rows_done % 8)   # up to 8 distinct rows, cycled
                t0 = time.perf_counter()
                oracle.decode(q, k, v, [p], s["win"], s["ring"], 1.0)
                t_used += time.perf_counter() - t0
                work_done += decode_bytes([p], s["hq"], s["hkv"], s["d"], s["win"])
                rows_done += 1
            total += t_used * w["bytes"] / work_done
            desc.append(f"{part}: {rows_done} rows of {n_rows}")
        elif part == "prompt_sparse":
            q, k, v, sel = _sample_inputs(part)
            vis = sparse_visible_keys(s)
            rng = np.random.default_rng(s["seed"])
            rows_done, t_used, flops_done = 0, 0.0, 0
            while t_used < per and rows_done < 64:
                i = int(rng.integers(0, s["n"]))
                t0 = time.perf_counter()
                oracle.prompt_sparse(q, k, v, s["p0"], s["win"], s["ring"], 1.0, sel, rows=[i])
                t_used += time.perf_counter() - t0
                flops_done += int(vis[i].sum()) * (s["hq"] // s["hkv"]) * 4 * s["d"]
                rows_done += 1
            total += t_used * w["flops"] / flops_done
            desc.append(f"{part}: {rows_done} random rows of {s['n']}, all heads")
        elif part == "prep_dense":
            from oracle import prep
            (x,) = _sample_inputs(part)
            rows_done, t_used = 0, 0.0
            while t_used < per and rows_done < s["N"]:
                t0 = time.perf_counter()
                prep.prepare(x, np.arange(x.shape[0]), s["H"], s["H"], s["d"], "rmsnorm")
                t_used += time.perf_counter() - t0
                rows_done += x.shape[0]
            total += t_used * s["N"] / rows_done
            desc.append(f"{part}: {rows_done} tokens of {s['N']}")
        elif part == "prompt_causal":
            n = s["n"]
            q, k, v = _sample_inputs(part)
            rng = np.random.default_rng(s["seed"])
            rows_done, t_used, flops_done = 0, 0.0, 0
            while t_used < per and rows_done < 64:
                i = int(rng.integers(0, n))
                t0 = time.perf_counter()
                oracle.prompt(q, k, v, s["p0"], s["win"], s["ring"], 1.0, rows=[i])
                t_used += time.perf_counter() - t0
                flops_done += prompt_flops_rows([i], s["p0"], s["win"], lambda r: s["p0"] + r, s["hq"], s["d"])
                rows_done += 1
            total += t_used * w["flops"] / flops_done
            desc.append(f"{part}: {rows_done} random rows of {n}, all heads")
        else:
            # every row sees all N keys, so the oracle gathers K and V once per call: fit
            # t(rows) = a + b * rows from two sample sizes and extrapolate to all N rows
            N, H, d = s["N"], 2, s["d"]
            q, k, v, scale = _sample_inputs(part)
            hi = np.full(N, N - 1)
            ts = {}
            for nr in (32, 512):
                rows = list(range(0, N, N // nr))[:nr]
                t0 = time.perf_counter()
                oracle.prompt(q, k, v, 0, 0, N, scale, hi=hi, rows=rows)
                ts[nr] = time.perf_counter() - t0
            b = max((ts[512] - ts[32]) / 480.0, 1e-12)
            a = max(ts[32] - 32 * b, 0.0)
            total += (a + b * N) * (s["H"] / H)
            desc.append(f"{part}: 32 and 512 rows x {H} heads of {N} x {s['H']} "
                        f"(t = a + b*rows fitted, a {a:.3f} s, b {b * 1e3:.3f} ms/row)")
    return total, "; ".join(desc)


def report_part(p: str, ms: float, pk) -> dict:
    """A part's time with its algorithmic throughput and fractions of the peaks."""
    w = part_work(p)
    if w["bytes"]:
        gbs = w["bytes"] / (ms * 1e-3) / 1e9
        return {"ms": ms, "GB/s": gbs, "frac_hbm": gbs / pk["hbm_gbs"],
                "frac_hbm_nominal_8tbs": gbs / NOMINAL_HBM_GBS, "bytes": w["bytes"]}
    tf = w["flops"] / (ms * 1e-3) / 1e12
    return {"ms": ms, "TFLOP/s": tf, "frac_bf16": tf / pk["bf16_tflops"],
            "frac_bf16_sustained": tf / pk["bf16_tflops_sustained"],
            "flops": w["flops"], "issued_TFLOP/s": tf * w.get("issued_flops_factor", 1.0)}


def oracle_one_core(parts, budget_s: float):
    """The oracle sample again in a child process pinned to one core, with every math library held to
    one thread (the variables must be set before numpy loads).  None if the child fails."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[var] = "1"
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-one-core", "--cpu-budget", str(budget_s),
           "--parts", ",".join(parts), "--no-next"]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=60 + 20 * budget_s)
    except subprocess.TimeoutExpired:
        return None
    if r.returncode != 0 or not r.stdout.strip():
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_oracle_one_core(args, parts):
    """Child side of oracle_one_core: pin to the first allowed core, time the sample, print JSON."""
    try:
        cpus = sorted(os.sched_getaffinity(0))
        os.sched_setaffinity(0, {cpus[0]})
    except (AttributeError, OSError):
        pass
    t, desc = oracle_sample(parts, args.cpu_budget)
    print(json.dumps({"seconds": t, "sample": desc}), flush=True)


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, parts):
    pk = peaks()
    t_roof = roofline_seconds(parts, pk)
    times = []
    budget = args.ref_budget
    for _ in range(args.warmup):
        oracle_sample(parts, budget / 4)
    desc = ""
    for _ in range(args.steps):
        t, desc = oracle_sample(parts, budget)
        times.append(t)
    t_step = statistics.median(times)
    value = t_roof / t_step
    cores = cpu_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(parts),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc + " (per step; extrapolated to the full workload by work)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(parts):
    return {"workload": " + ".join(parts), "parts": {p: SPEC[p] for p in parts},
            "l2": "inputs larger than L2 (each step streams > 40 GB of K/V and QKV); no flush",
            "peaks": "MEASURED_PEAKS.json hbm_gbs and bf16_tflops (burst; each part is timed alone)",
            "launch": "each part's C-ABI calls replayed as a CUDA graph captured after one eager call (the "
                      "three-stream parts fork and join inside the graph); e2e calls everything eagerly with "
                      "host copies, each part on a stream of its own"}


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--parts", default="all", help="comma list of " + ",".join(PARTS + EXTRA_PARTS))
    ap.add_argument("--next", default="all", help="comma list of the parts timed after the step: "
                    + ",".join(EXTRA_PARTS) + ", or none")
    ap.add_argument("--no-next", action="store_true", help="same as --next none")
    ap.add_argument("--oracle-one-core", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=6, help="e2e steps timed (the host link's rate varies from copy to copy; the mean over these)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=4.0, help="oracle seconds per reference step")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="oracle seconds for cpu_baseline")
    ap.add_argument("--caches", type=int, default=None, help="override the decode_sliding cache count (profiling)")
    ap.add_argument("--dense-n", type=int, default=None, help="override the dense prompts' and prep_dense's row count (profiling)")
    ap.add_argument("--decode-rows", type=int, default=None, help="override every decode part's rows per cache (profiling)")
    args = ap.parse_args()
    if args.caches is not None:
        SPEC["decode_sliding"]["caches"] = args.caches
    if args.dense_n is not None:
        for name in ("prompt_dense", "prompt_dense_p32", "prep_dense"):
            SPEC[name]["N"] = args.dense_n
    if args.decode_rows is not None:
        for name, sp in SPEC.items():
            if name.startswith("decode"):
                sp["rows"] = args.decode_rows
    args.warmup = max(args.warmup, 3)
    parts = list(PARTS) if args.parts == "all" else [p for p in args.parts.split(",") if p]
    for p in parts:
        if p not in PARTS and p not in EXTRA_PARTS:
            raise SystemExit(f"unknown part {p}")
    if args.no_next or args.next == "none":
        args.next_parts = []
    else:
        args.next_parts = [p for p in (EXTRA_PARTS if args.next == "all" else args.next.split(",")) if p
                           and p not in parts]
    for p in args.next_parts:
        if p not in EXTRA_PARTS:
            raise SystemExit(f"unknown next part {p}")
    if args.oracle_one_core:
        run_oracle_one_core(args, parts)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, parts)
        return

    dist = None
    if world > 1:
        args.next_parts = []   # the next parts are a one-GPU report
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    ms_per_step, per_part_ms, clk, e2e, launches, nxt = run_native(args, parts, rank, world, dist)
    pk = peaks()
    t_roof = roofline_seconds(parts, pk)
    value = weak_scaling_value(t_roof, ms_per_step, world)

    part_report = {p: report_part(p, per_part_ms[p], pk) for p in parts}
    dom = max(parts, key=lambda p: per_part_ms[p])
    w = part_work(dom)
    ms = per_part_ms[dom]
    if w["bytes"]:
        ach = w["bytes"] / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"]}
    else:
        ach = w["flops"] / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"], "peak_sustained": pk["bf16_tflops_sustained"],
                "frac_sustained": ach / pk["bf16_tflops_sustained"]}
    tr = TRAFFIC.get(dom)
    roof["traffic"] = tr["bytes_per_launch"] if tr and tr.get("source_sha") == source_hash(SOURCE_OF[dom]) else None
    roof["kernel"] = KERNEL_OF[dom] + f", part {dom}; per-launch time from CUDA events around the C-ABI call"
    roof["peak_source"] = pk["source"] + (" (burst bf16; the part is timed alone)" if roof["bound"] == "tensor"
                                          else " (copy GB/s)")

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_block(parts),
        "parts": part_report, "roofline": roof, "clocks": clk, "gpu_launches": launches,
    }
    if nxt is not None:
        line["next_parts"] = {p: report_part(p, nxt[p]["ms"], pk) for p in args.next_parts}
        line["next_parts"]["clocks"] = nxt["clocks"]
        line["next_parts"]["note"] = ("timed after the step, outside its value; each part's graph replay "
                                      "timed by CUDA events, median of the steps")
    if e2e is not None:
        line["e2e"] = {"value": weak_scaling_value(t_roof, e2e["ms_per_step"], world), "unit": UNIT,
                       "h2d_bytes_per_step": e2e["h2d_bytes_per_step"], "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                       "ms_per_step": e2e["ms_per_step"], "steps": e2e["steps"], "order": e2e["order"]}
    # the oracle baseline is one host's figure: timed on rank 0 of a one-GPU run only
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_cpu, desc = oracle_sample(parts, args.cpu_budget)
        line["cpu_baseline"] = {"value": t_roof / t_cpu, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                                "sample": desc + "; extrapolated to the full workload by work"}
        one = oracle_one_core(parts, args.cpu_budget / 2)
        if one is not None:
            line["cpu_baseline"]["one_core"] = {"value": t_roof / one["seconds"], "cores": 1,
                                                "sample": one["sample"] + "; extrapolated to the full workload by work"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
