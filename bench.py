#!/usr/bin/env python
"""Benchmark of the masked-MHA / split-KV decode path on GB300.

One JSON line on rank 0. Headline: valid-pair TFLOP/s of the masked MHA forward
(4*d FLOPs per unmasked (q, k) pair per head) on the largest configured workload,
the Longformer-style mask with one random head (B=1, H=32, L=16384, d=128, bf16),
with its roofline against the measured GB300 peaks. The same line carries the
other configured workloads (BERT band, BigBird, the split-KV GQA decode in
KV-read GB/s) and the widening rows as secondary objects under "workloads", and
ends with a compact "summary" of every figure (value, unit, roofline fraction,
ms), so that a reader of the line's tail sees all of them.

A step is one sta_mha_fwd_splitkv call with the library's split plan and kernel
choice (mask encoded once, outside the timed region).
L2 is flushed (a 256 MiB write, then a read of another 256 MiB buffer so that
no dirty line of the flush is left to write back, outside the CUDA events)
before every timed launch. The device time is the sum of per-launch CUDA-event durations on the
launching stream, each around the replay of a CUDA graph holding one library
call (so that host-side argument handling does not sit between the events);
`e2e` repeats the step through the public API, without a graph, with the
inputs copied from pinned host memory and the outputs copied back inside the
timed region.

--impl reference times the CPU oracle (fp64, all host cores) on the same
workload: the reference arm of this comparison is the plain restatement of
the method, not a GPU system.

Multi-GPU: the path shards into independent units and the bench runs
replicas only (every rank runs the same workload on its own GPU); value is
the sum over ranks divided by the slowest rank's time.
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha(name: str) -> str:
    """sha1 (12 hex) of a kernel source and of the library's headers (the `.cuh` / `.h` files
    beside it, which every kernel file includes), comments and whitespace removed: edits to
    comments keep recorded counters valid, any code change in the file or a header invalidates
    them."""
    d = os.path.join(ROOT, "split_kv_decode_bsr_gb300", "csrc")
    files = [name] + sorted(f for f in os.listdir(d) if f.endswith((".cuh", ".h")))
    h = hashlib.sha1()
    for f in files:
        src = open(os.path.join(d, f), encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(re.sub(r"\s+", " ", src).strip().encode() + b"\0")
    return h.hexdigest()[:12]


def recorded_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_source_sha(kernel_file)
    for line in open(p):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel_file and parts[1] == workload:
            return float(parts[3]) if parts[2] == sha else None
    return None


# ---------------------------------------------------------------------------
# distributed plumbing


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist

            backend = os.environ.get("STA_BENCH_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def _dev(self):
        import torch

        if self.pg.get_backend() == "nccl":
            return torch.device("cuda", self.local)
        return torch.device("cpu")

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=self._dev())
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=self._dev())
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(self.out)):
            row = [c.strip() for c in row]
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                mx.append(float(row[2]))
            except ValueError:
                continue
            for n, v in zip(names, row[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# workloads


def host_tensor(t):
    """torch CPU tensor of a seeded input (bf16 bit patterns reinterpreted, or float32)."""
    import torch

    if t.bf16 is not None:
        return torch.from_numpy(t.bf16.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(t.f32)


def gpu_sources_for(mask_heads, dev):
    """Mask descriptions of the seeded workloads as library mask sources (data uploaded)."""
    import torch

    import split_kv_decode_bsr_gb300 as sta

    out = []
    for m in mask_heads:
        if m.kind == "pattern":
            out.append(sta.MaskSource.pattern(m.causal, m.win_lo, m.win_hi, m.n_global_cols))
        elif m.kind == "bits":
            out.append(sta.MaskSource.dense_bits(torch.from_numpy(m.data.view(np.int64)).to(dev)))
        else:
            out.append(sta.MaskSource.dense_u8(torch.from_numpy(np.ascontiguousarray(m.data)).to(dev)))
    return out


def mha_workload(name):
    import workloads as W

    return {"bert-band": W.bert_band, "bigbird": W.bigbird, "longformer": W.longformer,
            "tiny-causal": W.tiny_causal, "long-causal": W.long_causal,
            "causal-1head": lambda: W.long_causal(H=1, L=16384), "sparse-random": W.sparse_random,
            "mixed-sparse": W.mixed_sparse, "dense-square": lambda: W.square_mask("dense"),
            "part-square": lambda: W.square_mask("random")}[name]()


def algorithmic_bytes_mha(wl, mask):
    elt = 2 if wl.dtype == "bf16" else 4
    qo = 2 * wl.B * wl.H * wl.Lq * wl.d * elt
    kv = 2 * wl.B * wl.H * wl.Lk * wl.d * elt
    lse = wl.B * wl.H * wl.Lq * 4
    bitmaps = mask.n_part * 512 + (mask.n_full + mask.n_part) * 4 + 2 * (mask.Hm * mask.ot_rows + 1) * 4
    return qo + kv + lse + bitmaps


def valid_pairs(wl, mask_counts):
    # mask_counts[h] = valid elements of mask head h
    return sum(wl.B * mask_counts[wl.head_map[h]] for h in range(wl.H))


class MhaBench:
    def __init__(self, name, dev, num_splits=0):
        import torch

        import split_kv_decode_bsr_gb300 as sta

        self.sta = sta
        self.wl = wl = mha_workload(name)
        self.name = name
        self.dev = dev
        self.q, self.k, self.v = (host_tensor(t).to(dev) for t in (wl.q, wl.k, wl.v))
        self.mask = sta.sta_encode_mask(gpu_sources_for(wl.mask_heads, dev), wl.Lq, wl.Lk)
        # per-mask-head valid counts (encode each head alone: host-side bookkeeping only)
        self.head_valid = [sta.sta_encode_mask(gpu_sources_for([m], dev), wl.Lq, wl.Lk).n_valid
                           for m in wl.mask_heads]
        self.pairs = valid_pairs(wl, self.head_valid)
        self.flops = 4.0 * wl.d * self.pairs
        self.bytes = algorithmic_bytes_mha(wl, self.mask)
        # bytes of dense mask input the encoder reads (pattern heads have none)
        self.encode_input_bytes = sum(int(m.data.nbytes) for m in wl.mask_heads if m.kind in ("bits", "u8"))
        self.kernel = sta.sta_mha_select_kernel(self.mask, wl.B, wl.H, wl.d,
                                                torch.bfloat16 if wl.dtype == "bf16" else torch.float32)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((wl.B, wl.H, wl.Lq), dtype=torch.float32, device=dev)
        # split-KV plan of the block kernel (0: the library's choice from the mask's tile counts)
        self.num_splits = num_splits
        ws = sta.mha_splitkv_workspace_bytes(self.mask, wl.B, wl.H, wl.d, self.q.dtype, head_map=wl.head_map,
                                             num_splits=num_splits)
        self.split = self.kernel in ("block", "mixed") and ws > 256
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.hq, self.hk, self.hv = (x.cpu().pin_memory() for x in (self.q, self.k, self.v))
        self.ho = torch.empty_like(self.o, device="cpu").pin_memory()
        self.hlse = torch.empty_like(self.lse, device="cpu").pin_memory()

    def step(self, kernel=None):
        if kernel is not None:  # selector calibration: one kernel, no split
            self.sta.sta_mha_fwd(self.q, self.k, self.v, self.mask, head_map=self.wl.head_map, scale=self.wl.scale,
                                 kernel=kernel, o=self.o, lse=self.lse)
            return
        self.sta.sta_mha_fwd_splitkv(self.q, self.k, self.v, self.mask, head_map=self.wl.head_map,
                                     scale=self.wl.scale, num_splits=self.num_splits, o=self.o, lse=self.lse,
                                     workspace=self.ws)

    def step_e2e(self):
        self.q.copy_(self.hq, non_blocking=True)
        self.k.copy_(self.hk, non_blocking=True)
        self.v.copy_(self.hv, non_blocking=True)
        self.step()
        self.ho.copy_(self.o, non_blocking=True)
        self.hlse.copy_(self.lse, non_blocking=True)

    def pipelined_e2e(self):
        """Serving-loop form of the end-to-end step: two sets of device buffers, so that step i+1's
        inputs are copied in (one stream) while step i computes (another) and step i-1's outputs
        are copied out (a third). Every step still copies its own inputs in and its outputs out;
        returns a callable running one such step."""
        import torch

        sta, wl = self.sta, self.wl
        bufs = []
        for _ in range(2):
            bufs.append(dict(q=torch.empty_like(self.q), k=torch.empty_like(self.k), v=torch.empty_like(self.v),
                             o=torch.empty_like(self.o), lse=torch.empty_like(self.lse), ws=torch.empty_like(self.ws),
                             ho=torch.empty_like(self.ho).pin_memory(), hlse=torch.empty_like(self.hlse).pin_memory(),
                             inp=torch.cuda.Event(), comp=torch.cuda.Event(), out=torch.cuda.Event()))
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        state = {"i": 0}

        def one():
            b = bufs[state["i"] % 2]
            state["i"] += 1
            with torch.cuda.stream(s_in):
                s_in.wait_event(b["out"])  # the buffers' previous step has been copied out
                b["q"].copy_(self.hq, non_blocking=True)
                b["k"].copy_(self.hk, non_blocking=True)
                b["v"].copy_(self.hv, non_blocking=True)
                b["inp"].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(b["inp"])
                sta.sta_mha_fwd_splitkv(b["q"], b["k"], b["v"], self.mask, head_map=wl.head_map, scale=wl.scale,
                                        num_splits=self.num_splits, o=b["o"], lse=b["lse"], workspace=b["ws"],
                                        stream=s_comp)
                b["comp"].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(b["comp"])
                b["ho"].copy_(b["o"], non_blocking=True)
                b["hlse"].copy_(b["lse"], non_blocking=True)
                b["out"].record(s_out)

        return one

    @property
    def h2d_bytes(self):
        return sum(x.numel() * x.element_size() for x in (self.hq, self.hk, self.hv))

    @property
    def d2h_bytes(self):
        return sum(x.numel() * x.element_size() for x in (self.ho, self.hlse))

    def launches_per_step(self):
        # block or row kernel, or both under the per-head choice (+ the merge of split heads)
        return (2 if self.kernel == "mixed" else 1) + (1 if self.split else 0)


class DecodeBench:
    def __init__(self, dev, page_size: int = 0):
        import torch

        import split_kv_decode_bsr_gb300 as sta
        import workloads as W

        self.sta = sta
        self.wl = wl = W.gqa_decode()
        self.dev = dev
        self.q, self.k, self.v = (host_tensor(t).to(dev) for t in (wl.q, wl.k, wl.v))
        self.ind_host = wl.kv_indptr
        self.ind = torch.from_numpy(wl.kv_indptr).to(dev)
        self.T = int(wl.kv_indptr[-1])
        self.kv_bytes = self.T * wl.Hkv * wl.d * 2 * 2
        self.bytes = self.kv_bytes + 2 * wl.n_req * wl.Hq * wl.d * 2 + wl.n_req * wl.Hq * 4
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((wl.n_req, wl.Hq), dtype=torch.float32, device=dev)
        nbytes = sta.decode_workspace_bytes(self.ind_host, wl.n_req, wl.Hq, wl.Hkv, wl.d, 0, page_size)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.page_size = page_size
        if page_size:  # the same K/V values in pages of page_size tokens, in a random page order
            pk = W.page_kv(wl, page_size, seed=1)
            self.kp, self.vp = (host_tensor(t).to(dev) for t in (pk.k_pages, pk.v_pages))
            self.pind = torch.from_numpy(pk.page_indptr).to(dev)
            self.pidx = torch.from_numpy(pk.page_indices).to(dev)
            del self.k, self.v
        self.hq = self.q.cpu().pin_memory()
        self.ho = torch.empty_like(self.o, device="cpu").pin_memory()
        self.hlse = torch.empty_like(self.lse, device="cpu").pin_memory()

    def step(self):
        if self.page_size:
            self.sta.sta_decode_splitkv_paged(self.q, self.kp, self.vp, self.pind, self.pidx, self.ind, self.ind_host,
                                              scale=self.wl.scale, num_splits=0, o=self.o, lse=self.lse,
                                              workspace=self.ws)
            return
        self.sta.sta_decode_splitkv(self.q, self.k, self.v, self.ind, self.ind_host, scale=self.wl.scale,
                                    num_splits=0, o=self.o, lse=self.lse, workspace=self.ws)

    def step_e2e(self):
        # serving shape: the KV cache stays resident; the new query tokens come in, outputs go out
        self.q.copy_(self.hq, non_blocking=True)
        self.step()
        self.ho.copy_(self.o, non_blocking=True)
        self.hlse.copy_(self.lse, non_blocking=True)

    def launches_per_step(self):
        return 2


class MlaBench:
    """Decode against a shared latent KV cache (64 requests, 16 query heads, 512 + 64 entries per
    cached token, lengths 512..32768 like the GQA decode)."""

    def __init__(self, dev):
        import torch

        import split_kv_decode_bsr_gb300 as sta
        import workloads as W

        self.sta = sta
        self.wl = wl = W.mla_decode()
        self.q, self.kv = host_tensor(wl.q).to(dev), host_tensor(wl.kv).to(dev)
        self.ind_host = wl.kv_indptr
        self.ind = torch.from_numpy(wl.kv_indptr).to(dev)
        self.T = int(wl.kv_indptr[-1])
        self.kv_bytes = self.T * wl.d_qk * 2
        self.bytes = self.kv_bytes + wl.n_req * wl.Hq * (wl.d_qk + wl.d_v) * 2 + wl.n_req * wl.Hq * 4
        self.flops = 2 * wl.Hq * self.T * (wl.d_qk + wl.d_v)
        self.o = torch.empty((wl.n_req, wl.Hq, wl.d_v), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((wl.n_req, wl.Hq), dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(sta.mla_workspace_bytes(self.ind_host, wl.n_req, wl.Hq), 256), dtype=torch.uint8,
                              device=dev)
        self.hq = self.q.cpu().pin_memory()
        self.ho = torch.empty_like(self.o, device="cpu").pin_memory()

    def step(self):
        self.sta.sta_mla_decode(self.q, self.kv, self.ind, self.ind_host, scale=self.wl.scale, o=self.o, lse=self.lse,
                                workspace=self.ws)

    def step_e2e(self):  # the latent cache stays resident; query tokens in, outputs out
        self.q.copy_(self.hq, non_blocking=True)
        self.step()
        self.ho.copy_(self.o, non_blocking=True)

    kernel_desc = "mma.sync m16n8k16 bf16 (16 query heads as M)"

    def launches_per_step(self):
        return 2  # decode (+ the merge of the requests cut into chunks)


class EpilogueBench:
    """The fused bias + residual + layer norm after the output projection of a 16384-token,
    32-head x 128 attention layer: x, residual [16384, 4096] bf16, bias [4096] bf16,
    gamma, beta [4096] f32 -> y bf16."""

    def __init__(self, dev, rows=16384, n=4096):
        import torch

        import split_kv_decode_bsr_gb300 as sta
        import workloads as W

        self.sta, self.rows, self.n = sta, rows, n
        self.x = host_tensor(W.make_tensor(0, 1, (rows, n), "bf16")).to(dev)
        self.res = host_tensor(W.make_tensor(0, 2, (rows, n), "bf16", 2.0)).to(dev)
        self.bias = host_tensor(W.make_tensor(0, 3, (n,), "bf16", 0.5)).to(dev)
        self.gamma = (1.0 + torch.from_numpy(W.make_tensor(0, 4, (n,), "f32", 0.1).f32)).to(dev)
        self.beta = torch.from_numpy(W.make_tensor(0, 5, (n,), "f32", 0.1).f32).to(dev)
        self.y = torch.empty_like(self.x)
        self.bytes = rows * n * 2 * 3 + n * (2 + 4 + 4)  # x, residual read, y written; the row vectors
        self.hx = self.x.cpu().pin_memory()
        self.hy = torch.empty_like(self.y, device="cpu").pin_memory()

    def step(self):
        self.sta.sta_bias_residual_layernorm(self.x, self.bias, self.res, self.gamma, self.beta, eps=1e-5, y=self.y)

    def step_unfused(self):  # the same operators as three separate torch kernels (context only)
        import torch

        h = self.x + self.bias + self.res
        return torch.nn.functional.layer_norm(h, (self.n,), self.gamma.to(h.dtype), self.beta.to(h.dtype), 1e-5)

    def step_e2e(self):
        self.x.copy_(self.hx, non_blocking=True)
        self.step()
        self.hy.copy_(self.y, non_blocking=True)

    def launches_per_step(self):
        return 1


def graphed(fn):
    """One library call captured in a CUDA graph; returns its replay.

    The device-timed steps replay the same kernel launches without the host's
    per-call work (argument checks, planning, tensor-map encoding, ctypes), which
    would otherwise sit inside the CUDA events whenever the host is slower than
    the GPU. The end-to-end figure keeps the direct call.
    """
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g.replay


def time_device(fn, steps, warmup, dist, flush):
    import torch

    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0 = time.perf_counter()
    for a, b in evs:
        flush()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    dist.barrier()
    wall = time.perf_counter() - t0
    ms = [a.elapsed_time(b) for a, b in evs]
    return ms, wall


def timing_stats(ms, fn, steps, warmup, dist):
    """Median and minimum of the cold (L2-flushed) per-step times, and the median with L2
    left warm (no flush between steps)."""
    warm, _ = time_device(fn, steps, warmup, dist, lambda: None)
    return {"cold_median_ms": statistics.median(ms), "cold_min_ms": min(ms),
            "warm_median_ms": statistics.median(warm), "warm_min_ms": min(warm)}


def time_e2e(fn, steps, warmup, dist):
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        fn()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    return dist.max(wall)


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)


def oracle_mha_seconds(wl, repeats=1):
    import oracle

    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle.mha_fwd(wl.q.f32, wl.k.f32, wl.v.f32, wl.mask_heads, wl.head_map, wl.scale)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, flops, target_s):
    t1 = oracle_mha_seconds(wl)
    reps = max(1, int(math.ceil(target_s / max(t1, 1e-3))))
    t = oracle_mha_seconds(wl, reps) if reps > 1 else t1
    return {"value": flops * reps / t / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"full {wl.name} workload, {reps} pass(es), fp64 C oracle, {t:.1f} s"}


# ---------------------------------------------------------------------------


L2_NOTE = ("inputs of the configured workloads exceed or approach the 129 MB L2; the GPU arm flushes L2 before "
           "every timed launch (256 MiB write, then a 256 MiB read)")


def mha_config(wl, pairs, world):
    """The workload description both arms report (identical dicts, so the two lines compare)."""
    return {"workload": wl.name, "B": wl.B, "H": wl.H, "L": wl.Lq, "d": wl.d, "mask": wl.meta.get("mask", ""),
            "valid_pairs": int(pairs), "l2": L2_NOTE, "parallelism": f"replicas x{world}"}


def run_reference(args, dist):
    """Reference arm: the CPU oracle, as it stands, on the headline workload (one full pass per step)."""
    if dist.rank != 0:
        return
    wl = mha_workload(args.workload)
    import oracle

    heads_valid = [oracle.mask_count(m, wl.Lq, wl.Lk) for m in wl.mask_heads]
    pairs = valid_pairs(wl, heads_valid)
    flops = 4.0 * wl.d * pairs
    for _ in range(args.warmup):
        oracle_mha_seconds(wl)
    times = [oracle_mha_seconds(wl) for _ in range(args.steps)]
    tot = sum(times)
    value = flops * args.steps / tot / 1e12
    line = {"impl": "reference", "metric": "valid-pair TFLOP/s (masked MHA fwd)", "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": mha_config(wl, pairs, args.gpus),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"full {wl.name} workload per step, fp64 C oracle"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def roofline_obj(bound, achieved, peak, unit, traffic, which):
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": traffic, "peak_source": which}


def mha_roofline(b, t, peaks, traffic, which):
    """The bound of a masked-MHA workload is the slower of its ideal times: valid-pair FLOPs at
    the bf16 peak (tensor) or algorithmic bytes at the HBM peak (hbm); the line reports the
    achieved rate against that one. Traffic (DRAM bytes) belongs to the hbm view only."""
    t_tensor = b.flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = b.bytes / (peaks["hbm_gbs"] * 1e9)
    if t_tensor > t_hbm:
        r = roofline_obj("tensor", b.flops / t / 1e12, peaks["bf16_tflops"], "TFLOP/s", None, which)
    else:
        r = roofline_obj("hbm", b.bytes / t / 1e9, peaks["hbm_gbs"], "GB/s", traffic, which)
    r["algorithmic_bytes_per_launch"] = b.bytes
    r["valid_pair_flops_per_launch"] = b.flops
    return r


def summary_entry(d):
    """[value, unit, ms, roofline fraction, bound] of one workload object (the last two null
    without a roofline)."""
    r = d.get("roofline") or {}
    return [round(d["value"], 2), d["unit"], round(d["ms_per_step"], 4), round(r["frac"], 3) if r else None,
            r.get("bound")]


def measure_mha(name, dev, args, dist, flush, peaks, peak_src, steps):
    """One masked-MHA workload through sta_mha_fwd_splitkv (library plan): timing, roofline."""
    b = MhaBench(name, dev, args.mha_splits)
    g = graphed(b.step)
    ms, wall = time_device(g, steps, args.warmup, dist, flush)
    t = sum(ms) / len(ms) / 1e3
    kf = "mha_block.cu" if b.kernel == "block" else "mha_row.cu"
    out = {
        "metric": "valid-pair TFLOP/s (masked MHA fwd)", "value": b.flops / t / 1e12, "unit": "TFLOP/s",
        "ms_per_step": 1e3 * t, "config": mha_config(b.wl, b.pairs, dist.world),
        "launch": {"kernel": b.kernel, "split_kv": "planned" if b.split else "none", "workspace_bytes": b.ws.numel()},
        "tensor_frac": (b.flops / t / 1e12) / peaks["bf16_tflops"],
        "tensor_frac_sustained": (b.flops / t / 1e12) / peaks["bf16_tflops_sustained"],
        "roofline": mha_roofline(b, t, peaks, recorded_traffic(kf, name), peak_src),
        "gpu_launches": b.launches_per_step() * steps,
        "timing_stats": timing_stats(ms, g, steps, args.warmup, dist),
    }
    return b, out, ms, wall


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="sta", choices=["sta", "reference"])
    ap.add_argument("--workload", default="longformer",
                    help="headline masked-MHA workload (default: the Longformer + random head, the largest)")
    ap.add_argument("--extra", default="bert-band,bigbird,decode,decode-paged,long-causal,causal-1head,"
                                       "sparse-random,mixed-sparse,epilogue-ln,mha-token-major,mla-decode",
                    help="comma list of secondary workloads (bert-band, bigbird, longformer, decode, decode-paged, "
                         "long-causal, causal-1head, sparse-random, mixed-sparse, epilogue-ln, mha-token-major, "
                         "mla-decode, and the matched pair dense-square / part-square) or 'none'")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--mha-splits", type=int, default=0,
                    help="split-KV chunks per head for the block kernel (0: the library's plan)")
    ap.add_argument("--sweep-kernels", action="store_true",
                    help="also time both MHA kernels on every MHA workload (selector calibration)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
        dist.close()
        return

    import torch

    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    import split_kv_decode_bsr_gb300 as sta

    sta.lib()  # fails loudly when libsta.so is missing
    peaks, peak_src = load_peaks()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clean_buf = torch.zeros(64 << 20, dtype=torch.float32, device=dev)  # 256 MiB, summed in place

    def flush():
        # a write larger than L2 evicts everything; reading a second such buffer then evicts
        # the write's own dirty lines, so the timed launch starts from a cold L2 with nothing
        # of the flush left to write back
        flush_buf.fill_(1)
        clean_buf.sum()

    # ---- headline: masked MHA on the largest configured workload
    with ClockSampler(dist.local) as clk:
        mb, head, ms, wall = measure_mha(args.workload, dev, args, dist, flush, peaks, peak_src, args.steps)
    dev_s = dist.max(sum(ms) / 1e3)
    total_flops = dist.sum(mb.flops * args.steps)
    value = total_flops / dev_s / 1e12
    ms_per_step = 1e3 * dev_s / args.steps
    if args.sweep_kernels:
        head["launch"]["kernel_ms"] = {
            k: sum(time_device(graphed(lambda: mb.step(k)), args.steps, args.warmup, dist, flush)[0]) / args.steps
            for k in ("block", "row")}
    e2e_s = time_e2e(mb.pipelined_e2e(), args.steps, args.warmup, dist)
    e2e_value = total_flops / e2e_s / 1e12
    e2e_serial_s = time_e2e(mb.step_e2e, args.steps, args.warmup, dist)
    line = {
        "metric": "valid-pair TFLOP/s (masked MHA fwd)", "value": value, "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": head["config"],
        "launch": dict(head["launch"], timing="CUDA events around a CUDA-graph replay of one library call per step"),
        "tensor_frac": head["tensor_frac"],
        "tensor_frac_sustained": head["tensor_frac_sustained"],
        "roofline": head["roofline"],
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": mb.h2d_bytes,
                "d2h_bytes_per_step": mb.d2h_bytes,
                "form": "serving loop: step i+1's inputs copied in while step i computes and step i-1's "
                        "outputs are copied out (two device buffer sets, three streams)",
                "serial_value": total_flops / e2e_serial_s / 1e12},
        "gpu_launches": head["gpu_launches"],
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
        "timing_stats": head["timing_stats"],
    }
    if dist.rank == 0:
        line["cpu_baseline"] = cpu_baseline(mb.wl, mb.flops, args.cpu_seconds) if dist.world == 1 else None
    del mb
    torch.cuda.empty_cache()
    summary = {args.workload: summary_entry(dict(head, ms_per_step=ms_per_step, value=value))}

    # ---- secondary workloads
    extras = {}
    wanted = [] if args.extra == "none" else [x for x in args.extra.split(",") if x and x != args.workload]
    for name in wanted:
        steps = max(3, min(args.steps, 10))
        if name == "epilogue-ln":
            eb = EpilogueBench(dev)
            g = graphed(eb.step)
            ms, _ = time_device(g, steps, args.warmup, dist, flush)
            t = sum(ms) / len(ms) / 1e3
            ms_u, _ = time_device(graphed(eb.step_unfused), steps, args.warmup, dist, flush)
            e2e_s = time_e2e(eb.step_e2e, steps, args.warmup, dist)
            extras[name] = {
                "metric": "fused bias+residual+layernorm GB/s", "value": eb.bytes / t / 1e9, "unit": "GB/s",
                "ms_per_step": 1e3 * t,
                "config": {"workload": f"bias+residual+layernorm bf16 rows {eb.rows} n {eb.n}",
                           "algorithmic_bytes": eb.bytes},
                "roofline": roofline_obj("hbm", eb.bytes / t / 1e9, peaks["hbm_gbs"], "GB/s",
                                         recorded_traffic("epilogue.cu", name), peak_src),
                "unfused_torch_ms": sum(ms_u) / len(ms_u),
                "e2e": {"value": eb.bytes / (e2e_s / steps) / 1e9, "unit": "GB/s",
                        "h2d_bytes_per_step": eb.x.numel() * 2, "d2h_bytes_per_step": eb.y.numel() * 2},
                "gpu_launches": eb.launches_per_step() * steps,
                "timing_stats": timing_stats(ms, g, steps, args.warmup, dist),
            }
            del eb
        elif name == "mla-decode":
            mb2 = MlaBench(dev)
            g = graphed(mb2.step)
            ms, _ = time_device(g, steps, args.warmup, dist, flush)
            t = sum(ms) / len(ms) / 1e3
            e2e_s = time_e2e(mb2.step_e2e, steps, args.warmup, dist)
            extras[name] = {
                "metric": "MLA decode KV-read GB/s", "value": mb2.kv_bytes / t / 1e9, "unit": "GB/s",
                "ms_per_step": 1e3 * t, "tflops": mb2.flops / t / 1e12,
                "config": {"workload": mb2.wl.name, "T": mb2.T, "kv_bytes": mb2.kv_bytes, "chunking": "library",
                           "kernel": mb2.kernel_desc},
                "roofline": roofline_obj("hbm", mb2.bytes / t / 1e9, peaks["hbm_gbs"], "GB/s",
                                         recorded_traffic("mla.cu", name), peak_src),
                "e2e": {"value": mb2.kv_bytes / (e2e_s / steps) / 1e9, "unit": "GB/s",
                        "h2d_bytes_per_step": mb2.hq.numel() * 2, "d2h_bytes_per_step": mb2.ho.numel() * 2},
                "gpu_launches": mb2.launches_per_step() * steps,
                "timing_stats": timing_stats(ms, g, steps, args.warmup, dist),
            }
            del mb2
        elif name == "mha-token-major":
            b = MhaBench("longformer", dev, args.mha_splits)
            ob = torch.empty((b.wl.B, b.wl.Lq, b.wl.H, b.wl.d), dtype=b.q.dtype, device=dev)

            def step_tokens():
                b.sta.sta_mha_fwd_splitkv(b.q, b.k, b.v, b.mask, head_map=b.wl.head_map, scale=b.wl.scale,
                                          num_splits=b.num_splits, o=ob, lse=b.lse, workspace=b.ws, o_layout="blhd")

            def step_then_transpose():  # head-major output, then torch's copy into token-major (context only)
                b.step()
                ob.copy_(b.o.permute(0, 2, 1, 3))

            ms_t, _ = time_device(graphed(step_tokens), steps, args.warmup, dist, flush)
            ms_h, _ = time_device(graphed(b.step), steps, args.warmup, dist, flush)
            ms_x, _ = time_device(graphed(step_then_transpose), steps, args.warmup, dist, flush)
            t = sum(ms_t) / len(ms_t) / 1e3
            extras[name] = {
                "metric": "valid-pair TFLOP/s (masked MHA fwd, O token-major)", "value": b.flops / t / 1e12,
                "unit": "TFLOP/s", "ms_per_step": 1e3 * t,
                "config": {"workload": b.wl.name, "o_layout": "[B, L, H, d]", "kernel": b.kernel},
                "head_major_ms": sum(ms_h) / len(ms_h),
                "head_major_then_torch_transpose_ms": sum(ms_x) / len(ms_x),
                "gpu_launches": b.launches_per_step() * steps,
            }
            del b, ob
        elif name in ("decode", "decode-paged"):
            db = DecodeBench(dev, 16 if name == "decode-paged" else 0)
            g = graphed(db.step)
            ms, _ = time_device(g, steps, args.warmup, dist, flush)
            t = sum(ms) / len(ms) / 1e3
            gbs = db.kv_bytes / t / 1e9
            e2e_s = time_e2e(db.step_e2e, steps, args.warmup, dist)
            extras[name] = {
                "metric": "split-KV decode KV-read GB/s", "value": gbs, "unit": "GB/s", "ms_per_step": 1e3 * t,
                "config": {"workload": db.wl.name, "T": db.T, "kv_bytes": db.kv_bytes, "num_splits": "auto",
                           "kv_layout": f"paged, {db.page_size} tokens per page, random page order"
                           if db.page_size else "packed [T, Hkv, d]"},
                "roofline": roofline_obj("hbm", db.bytes / t / 1e9, peaks["hbm_gbs"], "GB/s",
                                         recorded_traffic("decode.cu", name), peak_src),
                "e2e": {"value": db.kv_bytes / (e2e_s / steps) / 1e9, "unit": "GB/s",
                        "h2d_bytes_per_step": db.hq.numel() * 2,
                        "d2h_bytes_per_step": db.ho.numel() * 2 + db.hlse.numel() * 4},
                "gpu_launches": db.launches_per_step() * steps,
                "timing_stats": timing_stats(ms, g, steps, args.warmup, dist),
            }
            del db
        else:
            b, extras[name], _, _ = measure_mha(name, dev, args, dist, flush, peaks, peak_src, steps)
            if b.encode_input_bytes:  # the encoder, timed apart: the fill call over the dense mask input
                ms_e, _ = time_device(graphed(b.mask.refill), steps, args.warmup, dist, flush)
                te = sum(ms_e) / len(ms_e) / 1e3
                extras[name]["encode"] = {"us": 1e6 * te, "min_us": 1e3 * min(ms_e), "input_bytes": b.encode_input_bytes,
                                          "GB/s": b.encode_input_bytes / te / 1e9,
                                          "frac_hbm": b.encode_input_bytes / te / 1e9 / peaks["hbm_gbs"]}
            if b.split:  # the planner cut some heads: time the same call unsplit for comparison
                nb = MhaBench(name, dev, 1)
                ms1, _ = time_device(graphed(nb.step), steps, args.warmup, dist, flush)
                extras[name]["unsplit_ms"] = sum(ms1) / len(ms1)
                del nb
            if args.sweep_kernels or b.kernel == "mixed":  # each kernel alone on every head, for comparison
                extras[name]["launch"]["kernel_ms"] = {
                    k: sum(time_device(graphed(lambda: b.step(k)), steps, args.warmup, dist, flush)[0]) / steps
                    for k in ("block", "row")}
            del b
        summary[name] = summary_entry(extras[name])
        torch.cuda.empty_cache()
    line["workloads"] = extras
    err = sta.sta_device_error()
    if err:
        line["device_error"] = err
    # last key: one short entry per workload, so the end of the line holds every figure
    line["summary"] = dict(summary, columns=["value", "unit", "ms", "frac", "bound"])
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
