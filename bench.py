#!/usr/bin/env python3
"""Benchmark of the next-scale VAR attention hot path on B300.

One step = one pass of every row of the path, each on its workload, all
through the C ABI:
  dense attention      var_attn_dense         1024px final scale: 2 x 16 heads x
                                              4,096 queries against 10,521 keys, D 128
  cached token pruning var_pivot_select       the 48x48 step (hidden states 2304 x 2048,
                       var_attn_pruned        keep 2/5), from the 40x40 step's output,
                       var_restore_scatter    then the 64x64 step (4096 x 2048, keep
                                              1/5) from the restored 48x48 output
  block-sparse         var_attn_blocksparse   2K final scale: 16,384 queries against
                                              42,521 keys, sinks <= 16 + a +-2 block
                                              window (12.99 % of the pairs); the mask
                                              and plan are built once on the host
`value` is the step's algorithmic TFLOP/s: the FLOPs each attention kernel
executes (4 D per computed (query, key) pair: every pair for dense, the kept
rows for pruned, the kept pairs for block-sparse) over the step time.  The
dense-equivalent "effective" figure (full dense FLOPs of every attention
variant) is reported beside it, never against the peak.  The JSON line also
carries:
  rows          per-kernel times inside the timed region (CUDA events between
                the calls) and separate measurements: the small kernels from a
                CUDA graph after an L2 flush, the fused pruned step, the
                attention-guided pivots, the dynamic sparse pattern, Branch
                Halving, the tiny and 256px workloads, the host link ceiling
  roofline      the step's dominant kernel against the measured peak
  e2e           the same step with host buffers (pinned H2D of its inputs, D2H
                of its outputs, inside the timed region)
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same work
  clocks        SM clock and throttle reasons sampled during the timed region

`--impl reference` times the CPU oracle as the reference arm.
Multi-GPU (torchrun, N>1): every rank runs the same workload on its own GPU
(weak scaling, no collective on the data path); the slowest rank's time is
used and `value` counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from var_synth import WORKLOADS, cache_len, make_inputs  # noqa: E402

METRIC = "final-scale attention ms and TFLOP/s (dense-equiv) at 1 B300; % of BF16 peak"
W1024 = "pruned_1024px"              # tensors of the 1024px schedule (CFG pair, sink) + hidden states
W2K = "blocksparse_2k"
PREV, MID, FINAL = 10, 11, 12        # the 40x40, 48x48 and 64x64 steps
KEEP = {MID: (2, 5), FINAL: (1, 5)}  # keep ratios of the pruned steps
QBLOCK, RADIUS, SINK_SIDE = 8, 2, 16
ROW_NAMES = ("attn_dense_1024px", "pivot_select_48", "attn_pruned_48", "restore_scatter_40to48",
             "pivot_select_64", "attn_pruned_64", "restore_scatter_48to64", "attn_blocksparse_2k")
LAUNCHES_PER_STEP = 12               # dense 1, (pivot 3, pruned 1, restore 1) x 2, block-sparse 1
KERNEL_NAMES = {"attn_dense_1024px": "attn_kernel<128, dense>", "attn_pruned_48": "attn_kernel<128, gather>",
                "attn_pruned_64": "attn_kernel<128, gather>", "attn_blocksparse_2k": "attn_kernel<128, sparse>",
                "pivot_select_48": "pivot kernels", "pivot_select_64": "pivot kernels",
                "restore_scatter_40to48": "restore_rows_kernel<128>",
                "restore_scatter_48to64": "restore_rows_kernel<128>"}
TRAFFIC_KEYS = {"attn_dense_1024px": "attn_kernel<128, dense>:dense_1024px_final",
                "attn_blocksparse_2k": "attn_kernel<128, sparse>:blocksparse_2k_final",
                "attn_pruned_64": "attn_kernel<128, gather>:pruned_64x64_k819"}


# ----------------------------------------------------------------------------- helpers

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained") or d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# The sources that decide what the attention kernels compute and how they are
# launched: the kernel body, its PTX wrappers and the two launchers (grid, CTA
# plan, tensor maps).  Declarations elsewhere do not change the traffic.
ATTN_SOURCES = ("visual_autoregressive_next_var_b300/csrc/attn_kernel.cuh",
                "visual_autoregressive_next_var_b300/csrc/ptx.cuh",
                "visual_autoregressive_next_var_b300/csrc/attn.cu",
                "visual_autoregressive_next_var_b300/csrc/blocksparse.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(key: str):
    """Per-launch DRAM bytes (read + write) of a kernel on a workload from the
    committed ncu summary, or None when absent or taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(key)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e["dram_bytes"]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu = gpu_index
        self.enabled = enabled
        self.proc = None
        self.file = None

    def __enter__(self):
        if not self.enabled:
            return self
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.enabled:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled (--no-clocks)"]}
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = [l.strip().split(", ") for l in open(self.file.name) if l.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def flops_attn(B, H, Nq, Lk, D) -> float:
    """QK^T and PV: 4 D FLOPs per (query, key) pair."""
    return 4.0 * B * H * Nq * Lk * D


def mask_kept_pairs(sides, row_ptr, entries, sink_len, qblock) -> int:
    """(query, key) pairs a block mask keeps, counted from its CSR."""
    pairs = 0
    for qb in range(len(row_ptr) - 1):
        nk = sink_len
        for e in entries[row_ptr[qb]:row_ptr[qb + 1]]:
            sc, u, vv = int(e) >> 24, (int(e) >> 12) & 0xFFF, int(e) & 0xFFF
            s = sides[sc]
            nk += (min(s, u * qblock + qblock) - u * qblock) * (min(s, vv * qblock + qblock) - vv * qblock)
        pairs += nk * qblock * qblock
    return pairs


class L2Flush:
    """Evicts L2 by reading a buffer twice its size (reads leave no dirty lines)."""

    def __init__(self, dev):
        self.buf = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.sum()


def time_graph(fn, iters: int, flush: L2Flush) -> float:
    """Median ms of one fn() replayed from a CUDA graph, L2 flushed before each replay."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                   # warm up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


# ----------------------------------------------------------------------------- the step

class Step:
    """Device buffers and the call sequence of one step (every row of the path)."""

    def __init__(self, V, dev, inp, inp2k, mask2k_host):
        w, w2 = WORKLOADS[W1024], WORKLOADS[W2K]
        self.V = V
        B, H, D = w.batch, w.heads, w.head_dim
        self.p = V.problem(B, H, D, w.sides, kv_capacity=inp.k.shape[2])
        self.k = inp.k.to(dev)
        self.v = inp.v.to(dev)
        self.q = {s: inp.q[s].to(dev) for s in (MID, FINAL)}
        self.x = {s: inp.x[s].to(dev) for s in (MID, FINAL)}
        self.N = {s: w.sides[s] ** 2 for s in (PREV, MID, FINAL)}
        self.L = {s: cache_len(w.sides, s) for s in (PREV, MID, FINAL)}
        self.K = {s: V.var_keep_count(self.N[s], *KEEP[s]) for s in (MID, FINAL)}
        # the 40x40 step's output, the first restore's input: dense attention, computed once
        q10 = inp.q[PREV].to(dev)
        self.prev = torch.empty_like(q10)
        V.var_attn_dense(self.p, PREV, q10, self.k, self.v, self.prev)
        del q10
        self.o_dense = torch.empty_like(self.q[FINAL])
        C = self.x[FINAL].shape[2]
        self.ws = {s: torch.empty(V.var_pivot_workspace_bytes(self.p, s, C), dtype=torch.uint8, device=dev)
                   for s in (MID, FINAL)}
        self.idx = {s: torch.empty((B, self.K[s]), dtype=torch.int32, device=dev) for s in (MID, FINAL)}
        self.oc = {s: torch.empty((B, H, self.K[s], D), dtype=torch.bfloat16, device=dev) for s in (MID, FINAL)}
        self.out = {s: torch.empty_like(self.q[s]) for s in (MID, FINAL)}
        # 2K block-sparse
        st2 = w2.steps[-1]
        self.st2 = st2
        self.p2 = V.problem(w2.batch, w2.heads, w2.head_dim, w2.sides)
        self.q2, self.k2, self.v2 = inp2k.q[st2].to(dev), inp2k.k.to(dev), inp2k.v.to(dev)
        self.o2 = torch.empty_like(self.q2)
        rp, en, sink, plan = mask2k_host
        self.mask_dev = [torch.as_tensor(rp, device=dev), torch.as_tensor(en, device=dev)] + \
                        [torch.as_tensor(a, device=dev) for a in plan]
        self.mask = V.block_mask_struct(QBLOCK, self.mask_dev[0], self.mask_dev[1], sink, self.mask_dev[2:])
        self.sparse_pairs = mask_kept_pairs(w2.sides, rp, en, sink, QBLOCK)
        self.N2, self.L2 = w2.sides[st2] ** 2, cache_len(w2.sides, st2)
        # algorithmic work per row
        self.flops = {
            "attn_dense_1024px": flops_attn(B, H, self.N[FINAL], self.L[FINAL], D),
            "attn_pruned_48": flops_attn(B, H, self.K[MID], self.L[MID], D),
            "attn_pruned_64": flops_attn(B, H, self.K[FINAL], self.L[FINAL], D),
            "attn_blocksparse_2k": 4.0 * w2.batch * w2.heads * self.sparse_pairs * w2.head_dim,
        }
        self.flops_dense_equiv = {
            "attn_dense_1024px": self.flops["attn_dense_1024px"],
            "attn_pruned_48": flops_attn(B, H, self.N[MID], self.L[MID], D),
            "attn_pruned_64": flops_attn(B, H, self.N[FINAL], self.L[FINAL], D),
            "attn_blocksparse_2k": flops_attn(w2.batch, w2.heads, self.N2, self.L2, w2.head_dim),
        }
        self.bytes = {
            "pivot_select_48": self.x[MID].numel() * 2 + self.idx[MID].numel() * 4,
            "pivot_select_64": self.x[FINAL].numel() * 2 + self.idx[FINAL].numel() * 4,
            "restore_scatter_40to48": (self.prev.numel() + self.oc[MID].numel() + self.out[MID].numel()) * 2
                                      + self.idx[MID].numel() * 4,
            "restore_scatter_48to64": (self.out[MID].numel() + self.oc[FINAL].numel() + self.out[FINAL].numel()) * 2
                                      + self.idx[FINAL].numel() * 4,
        }

    def calls(self, stream=None):
        V, p = self.V, self.p

        def pivot(s):
            return lambda: V.var_pivot_select(p, s, self.x[s], self.K[s], self.idx[s], self.ws[s], stream=stream)

        def pruned(s):
            return lambda: V.var_attn_pruned(p, s, self.q[s], self.k, self.v, self.idx[s], self.K[s], self.oc[s],
                                             stream=stream)

        def restore(s, prev):
            return lambda: V.var_restore_scatter(p, s, prev, self.oc[s], self.idx[s], self.K[s], self.out[s],
                                                 stream=stream)

        return (
            lambda: V.var_attn_dense(p, FINAL, self.q[FINAL], self.k, self.v, self.o_dense, stream=stream),
            pivot(MID), pruned(MID), restore(MID, self.prev),
            pivot(FINAL), pruned(FINAL), restore(FINAL, self.out[MID]),
            lambda: V.var_attn_blocksparse(self.p2, self.st2, self.q2, self.k2, self.v2, self.mask, self.o2,
                                           stream=stream),
        )

    def run(self, stream=None):
        for c in self.calls(stream):
            c()

    def uploads(self, host):
        """(device tensor, pinned host tensor) pairs of the step's inputs."""
        return [(self.q[FINAL], host["q64"]), (self.q[MID], host["q48"]), (self.k, host["k"]), (self.v, host["v"]),
                (self.x[MID], host["x48"]), (self.x[FINAL], host["x64"]), (self.prev, host["prev40"]),
                (self.q2, host["q2k"]), (self.k2, host["k2k"]), (self.v2, host["v2k"])]

    def results(self):
        return {"o_dense": self.o_dense, "idx48": self.idx[MID], "idx64": self.idx[FINAL],
                "out48": self.out[MID], "out64": self.out[FINAL], "o2k": self.o2}


def time_step(step: Step, steps: int, stream):
    """Total ms per step and per-row ms, CUDA events on `stream` between the calls."""
    calls = step.calls(stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(steps)]
    torch.cuda.synchronize()
    for s in range(steps):
        ev[s][0].record(stream)
        for i, c in enumerate(calls):
            c()
            ev[s][i + 1].record(stream)
    torch.cuda.synchronize()
    total = ev[0][0].elapsed_time(ev[-1][-1]) / steps
    per_row = [sum(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(steps)) / steps for i in range(len(calls))]
    return total, per_row


def build_mask_2k(V):
    """Host block mask and plan of the 2K final step: (row_ptr, entries, sink_len, plan), ms."""
    w = WORKLOADS[W2K]
    st = w.steps[-1]
    p = V.problem(w.batch, w.heads, w.head_dim, w.sides)
    t0 = time.perf_counter()
    rp, en, sink = V.var_block_mask_build(p, st, w.qblock_side, w.radius, w.sink_max_side)
    plan = V.var_block_mask_plan(p, st, w.qblock_side, rp, en, sink)
    return (rp, en, sink, plan), (time.perf_counter() - t0) * 1e3


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_sample(inp, budget_s: float, seed: int = 0):
    """Time the oracle on random query rows of the 1024px final step's dense
    attention, sized to about budget_s: (TFLOP/s, seconds, rows, threads)."""
    import oracle
    w = WORKLOADS[W1024]
    q = inp.q[FINAL]
    B, H, N, D = q.shape
    L = cache_len(w.sides, FINAL)
    oracle.attention(q, inp.k, inp.v, L, rows=np.arange(2))        # load + warm
    n = 8
    while True:
        t0 = time.perf_counter()
        oracle.attention(q, inp.k, inp.v, L, rows=np.arange(n) * (B * H * N // n))
        dt = time.perf_counter() - t0
        if dt >= 0.25 * budget_s or n >= B * H * N:
            break
        n = min(B * H * N, 4 * n)
    n_rows = int(max(1, min(B * H * N, n * budget_s / max(dt, 1e-6))))
    rows = np.sort(np.random.default_rng(seed).choice(B * H * N, size=n_rows, replace=False))
    t0 = time.perf_counter()
    oracle.attention(q, inp.k, inp.v, L, rows=rows)
    dt = time.perf_counter() - t0
    return n_rows * 4.0 * L * D / dt / 1e12, dt, n_rows, oracle.num_threads()


def step_config():
    """The `config` of both arms' JSON lines."""
    w, w2 = WORKLOADS[W1024], WORKLOADS[W2K]
    return {"workload": "var_hot_path_step: 1024px final-scale dense + pruned 48x48 and 64x64 steps "
                        "+ 2K final-scale block-sparse",
            "batch": w.batch, "heads": w.heads, "head_dim": w.head_dim,
            "dense": {"queries": w.sides[FINAL] ** 2, "keys": cache_len(w.sides, FINAL)},
            "pruned": {"48x48": {"keep": "2/5", "keys": cache_len(w.sides, MID)},
                       "64x64": {"keep": "1/5", "keys": cache_len(w.sides, FINAL)},
                       "channels": w.channels},
            "blocksparse": {"queries": w2.sides[-1] ** 2, "keys": cache_len(w2.sides, w2.steps[-1]),
                            "mask": f"qblock {QBLOCK}, radius {RADIUS}, sinks <= {SINK_SIDE}"},
            "rows": list(ROW_NAMES),
            "l2": "inputs larger than L2 (1024px Q/K/V + hidden states 0.28 GB, 2K Q/K/V 0.83 GB per step)",
            "per_gpu": "each rank runs the whole workload"}


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    inp = make_inputs(WORKLOADS[W1024], steps=(FINAL,))
    per_step = min(args.ref_seconds, 150.0 / (args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        tf, dt, n_rows, thr = oracle_sample(inp, per_step, seed=i)
        if i >= args.warmup:
            vals.append((tf, dt))
    value = statistics.median(v for v, _ in vals)
    ms = statistics.median(dt for _, dt in vals) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": step_config(),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"{n_rows} random query rows of the 1024px final step's dense attention "
                                   "per step; throughput per FLOP"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def time_events(fn, n: int, stream) -> float:
    """Mean ms of n back-to-back fn() on `stream` (CUDA events)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def extra_rows(V, dev, step: Step, inp, iters: int, peaks, host_bytes):
    """Separate measurements: the small kernels alone, the fused pruned step, the
    §8(f) rows, the tiny and 256px workloads, the host link ceiling."""
    rows = {}
    flush = L2Flush(dev)
    calls = dict(zip(ROW_NAMES, step.calls()))
    for name in ("pivot_select_48", "pivot_select_64", "restore_scatter_40to48", "restore_scatter_48to64"):
        t = time_graph(calls[name], iters, flush)
        rows[name + "_alone"] = {"ms": t, "GB/s": step.bytes[name] / t / 1e6,
                                 "frac_hbm": step.bytes[name] / t / 1e6 / peaks["hbm_gbs"],
                                 "timing": "CUDA graph replay after an L2 flush"}
    # the single-launch floor at the pivot's size: one copy of the 64x64 hidden states
    xs = step.x[FINAL]
    xd = torch.empty_like(xs)
    t = time_graph(lambda: xd.copy_(xs), iters, flush)
    rows["copy_floor_34MB_alone"] = {"ms": t, "GB/s": 2 * xs.numel() * 2 / t / 1e6,
                                     "frac_hbm": 2 * xs.numel() * 2 / t / 1e6 / peaks["hbm_gbs"],
                                     "note": "one torch copy_ launch of the 64x64 hidden states (read + write "
                                             "2 x 33.6 MB): what a single launch of this size reaches",
                                     "timing": "CUDA graph replay after an L2 flush"}
    del xd
    # the pruned 64x64 step with the outputs written in place (no compact buffer)
    p, s = step.p, FINAL

    def fused():
        # one call: the fill starts beside the attention (programmatic dependent
        # launch) on the SMs the attention leaves free; disjoint rows
        V.var_pruned_in_place(p, s, step.q[s], step.k, step.v, step.out[MID], step.idx[s], step.K[s], step.out[s])

    t = time_graph(fused, iters, flush)
    t_attn = time_graph(lambda: V.var_attn_pruned_scatter(p, s, step.q[s], step.k, step.v, step.idx[s], step.K[s],
                                                          step.out[s]), iters, flush)
    t_chain = time_graph(lambda: (calls["attn_pruned_64"](), calls["restore_scatter_48to64"]()), iters, flush)
    # the whole pruned 64x64 step: pivots, pruned attention and restore
    t_step = time_graph(lambda: V.var_pruned_step(p, s, step.x[s], step.K[s], step.q[s], step.k, step.v, step.out[MID],
                                                  step.idx[s], step.out[s], step.ws[s]), iters, flush)
    t_step_chain = time_graph(lambda: (calls["pivot_select_64"](), calls["attn_pruned_64"](),
                                       calls["restore_scatter_48to64"]()), iters, flush)
    rows["pruned_64_whole_step_one_call"] = {
        "ms": t_step, "three_calls_ms": t_step_chain,
        "note": "var_pruned_step: pivot selection, then the in-place pruned attention started beside the selection "
                "kernel, then the fill beside the attention; three calls: var_pivot_select, var_attn_pruned, "
                "var_restore_scatter",
        "timing": "CUDA graph replay after an L2 flush"}
    rows["pruned_64_attn_and_restore_fused"] = {
        "ms": t, "attn_in_place_alone_ms": t_attn, "unfused_ms": t_chain,
        "note": "var_pruned_in_place: the attention writes its rows into the full grid and the fill, started "
                "beside it, writes the rest; unfused: compact attention output, then restore + scatter",
        "timing": "CUDA graph replay after an L2 flush"}
    # attention-guided pivots (ARVAR): the 32x32 step's row statistics and saliency
    src = FINAL - 3
    q_src = inp.q[src].to(dev)
    B, H, Ns, D = q_src.shape
    o_src = torch.empty_like(q_src)
    lse = torch.empty((B, H, Ns), dtype=torch.float32, device=dev)
    sal = torch.empty((B, H, Ns), dtype=torch.float32, device=dev)
    gws = torch.empty(V.var_guided_pivot_workspace_bytes(p, FINAL), dtype=torch.uint8, device=dev)
    gidx = torch.empty_like(step.idx[FINAL])
    t_plain = time_graph(lambda: V.var_attn_dense(p, src, q_src, step.k, step.v, o_src), iters, flush)
    t_lse = time_graph(lambda: V.var_attn_dense_lse(p, src, q_src, step.k, step.v, o_src, lse), iters, flush)
    t_sal = time_graph(lambda: V.var_attn_saliency(p, src, q_src, step.k, lse, sal), iters, flush)
    t_sel = time_graph(lambda: V.var_guided_pivot_select(p, FINAL, src, sal, step.K[FINAL], gidx, gws),
                       iters, flush)
    L_src = cache_len(WORKLOADS[W1024].sides, src)
    gx_ws = torch.empty(V.var_guided_pivot_exact_workspace_bytes(p, FINAL, src), dtype=torch.uint8, device=dev)
    t_exact = time_graph(lambda: V.var_guided_pivot_select_exact(p, FINAL, src, q_src, step.k, step.K[FINAL], gidx,
                                                                 gx_ws), max(3, iters // 4), flush)
    fl_sal = 2.0 * B * H * Ns * Ns * D            # S^T = K_self Q^T
    rows["guided_pivot_from_32x32"] = {
        "ms": t_sal + t_sel, "saliency_ms": t_sal, "select_ms": t_sel,
        "saliency_TFLOP/s": fl_sal / t_sal / 1e9,
        "source_dense_ms": t_plain, "source_dense_with_lse_ms": t_lse,
        "exact_fp64_ms": t_exact,
        "note": f"source step 32x32 ({Ns} queries, {L_src} keys) -> 64x64, keep 1/5; the row "
                "statistics are written by the source step's own dense attention; exact_fp64_ms: the "
                "ranking decided in fp64 (var_guided_pivot_select_exact, from the source queries and keys)",
        "timing": "CUDA graph replay after an L2 flush"}
    # SparVAR dynamic pattern: the 32x32 step's block scores decide the 64x64 step's mask
    d_sv, tau_sv = src, 0.8
    U_sv, _ = V.var_sparvar_units(p, d_sv, SINK_SIDE)
    sv_ws = torch.empty(V.var_sparvar_workspace_bytes(p, d_sv, SINK_SIDE), dtype=torch.uint8, device=dev)
    nqb_sv = (int(round(Ns ** 0.5)) // 8) ** 2
    sv_sc = torch.empty((nqb_sv, U_sv), dtype=torch.float64, device=dev)
    sv_rs = torch.zeros(nqb_sv, dtype=torch.int32, device=dev)
    t_sc = time_graph(lambda: V.var_sparvar_scores(p, d_sv, SINK_SIDE, tau_sv, q_src, step.k, sv_ws, sv_sc,
                                                   rescored=sv_rs), iters, flush)
    n_rescored = int(sv_rs.sum().item())
    # the tensor-core scores from the decision step's row log2-sum-exp (the lse of
    # its dense attention, computed above for the guided pivots)
    sv_fast = torch.empty_like(sv_sc)
    V.var_attn_dense_lse(p, src, q_src, step.k, step.v, o_src, lse)
    t_fast = time_graph(lambda: V.var_sparvar_scores_fast(p, d_sv, SINK_SIDE, q_src, step.k, lse, sv_ws, sv_fast),
                        iters, flush)
    t_sc_all = time_graph(lambda: V.var_sparvar_scores(p, d_sv, SINK_SIDE, tau_sv, q_src, step.k, sv_ws, sv_sc,
                                                       flags=V.VAR_SPARVAR_RESCORE_ALL), iters, flush)
    V.var_sparvar_scores(p, d_sv, SINK_SIDE, tau_sv, q_src, step.k, sv_ws, sv_sc)
    t0 = time.perf_counter()
    A = sv_sc.cpu().numpy()
    rp, en, sink = V.var_sparvar_mask_build(p, d_sv, FINAL, SINK_SIDE, A, tau_sv)
    sv_plan = [torch.as_tensor(a, device=dev) for a in V.var_block_mask_plan(p, FINAL, QBLOCK, rp, en, sink)]
    t_host = (time.perf_counter() - t0) * 1e3
    sv_rp, sv_en = torch.as_tensor(rp, device=dev), torch.as_tensor(en, device=dev)
    sv_mask = V.block_mask_struct(QBLOCK, sv_rp, sv_en, sink, sv_plan)
    o_sv = torch.empty_like(step.q[FINAL])
    t_sv = time_graph(lambda: V.var_attn_blocksparse(p, FINAL, step.q[FINAL], step.k, step.v, sv_mask, o_sv),
                      iters, flush)
    pairs = mask_kept_pairs(WORKLOADS[W1024].sides, rp, en, sink, QBLOCK)
    fl_sv = 4.0 * B * H * pairs * D
    A_fast = sv_fast.cpu().numpy()
    rp_f, en_f, sink_f = V.var_sparvar_mask_build(p, d_sv, FINAL, SINK_SIDE, A_fast, tau_sv)
    same_mask = bool(np.array_equal(rp_f, rp) and np.array_equal(en_f, en) and sink_f == sink)
    rows["sparvar_dynamic_mask_32_to_64"] = {
        "scores_ms": t_sc, "blocks_rescored_fp64": n_rescored, "blocks": nqb_sv,
        "scores_fast_tensor_core_ms": t_fast, "fast_mask_equals_certified": same_mask,
        "fast_max_rel_diff": float(np.max(np.abs(A_fast - A) / np.maximum(A, 1e-12))),
        "scores_all_blocks_fp64_ms": t_sc_all, "host_select_map_plan_ms": t_host, "attn_ms": t_sv,
        "density": pairs / (step.N[FINAL] * step.L[FINAL]), "TFLOP/s": fl_sv / t_sv / 1e9,
        "effective_dense_equiv_TFLOP/s": step.flops["attn_dense_1024px"] / t_sv / 1e9, "units": U_sv, "tau": tau_sv,
        "note": "decision step 32x32: block scores (certified fp32 on the CUDA cores, fp64 re-score of the "
                "blocks the bound does not settle) -> host selection + index mapping -> block-sparse "
                "attention of the 64x64 step; scores_fast_tensor_core_ms: the same scores on the tensor cores "
                "from the decision step's row log2-sum-exp (deterministic, no error bound); "
                "fast_mask_equals_certified: the 64x64 mask built from them is the certified one",
        "timing": "CUDA graph replay after an L2 flush; host part timed once"}
    del q_src, o_src, o_sv
    # Branch Halving: the conditional half only, its rows repeated
    fd = step.flops["attn_dense_1024px"]
    t = time_graph(lambda: V.var_attn_dense_halved(p, FINAL, step.q[FINAL], step.k, step.v, step.o_dense),
                   iters, flush)
    rows["attn_dense_branch_halved"] = {"ms": t, "TFLOP/s": fd / 2 / t / 1e9,
                                        "frac_tensor": fd / 2 / t / 1e9 / peaks["bf16_tflops"],
                                        "effective_dense_equiv_TFLOP/s": fd / t / 1e9,
                                        "timing": "CUDA graph replay after an L2 flush"}
    # the tiny workload: 256 queries against 680 keys, batch 1, head_dim 64 (launch-bound)
    w = WORKLOADS["dense_tiny"]
    inp_t = make_inputs(w)
    st_t = w.steps[0]
    pt = V.problem(w.batch, w.heads, w.head_dim, w.sides)
    qt, kt, vt = inp_t.q[st_t].to(dev), inp_t.k.to(dev), inp_t.v.to(dev)
    ot = torch.empty_like(qt)
    t = time_graph(lambda: V.var_attn_dense(pt, st_t, qt, kt, vt, ot), iters, flush)
    fl = flops_attn(w.batch, w.heads, w.sides[st_t] ** 2, cache_len(w.sides, st_t), w.head_dim)
    rows["dense_tiny_256q_680k"] = {"ms": t, "TFLOP/s": fl / t / 1e9, "launches": 1,
                                    "note": "launch-bound: 0.71 GFLOP on 16 CTAs",
                                    "timing": "CUDA graph replay after an L2 flush"}
    # the whole 256px schedule, dense (launch-bound)
    w = WORKLOADS["dense_256px"]
    inp_s = make_inputs(w)
    B2, H2, D2 = w.batch, w.heads, w.head_dim
    ps = V.problem(B2, H2, D2, w.sides)
    ks, vs = inp_s.k.to(dev), inp_s.v.to(dev)
    qs = {s2: inp_s.q[s2].to(dev) for s2 in w.steps}
    os_ = {s2: torch.empty_like(qs[s2]) for s2 in w.steps}

    def sched():
        for s2 in w.steps:
            V.var_attn_dense(ps, s2, qs[s2], ks, vs, os_[s2])

    t = time_graph(sched, iters, flush)
    fl = sum(flops_attn(B2, H2, w.sides[s2] ** 2, cache_len(w.sides, s2), D2) for s2 in w.steps)
    t_last = time_graph(lambda: V.var_attn_dense(ps, w.steps[-1], qs[w.steps[-1]], ks, vs, os_[w.steps[-1]]),
                        iters, flush)
    rows["schedule_256px_dense_10_steps"] = {"ms": t, "TFLOP/s": fl / t / 1e9, "launches": len(w.steps),
                                             "final_step_ms": t_last,
                                             "timing": "CUDA graph replay after an L2 flush"}
    # the host link: one pinned copy of the e2e leg's upload and download sizes
    h_in, h_out = host_bytes
    hb = torch.empty(h_in, dtype=torch.uint8).pin_memory()
    db = torch.empty(h_in, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    t_h2d = time_events(lambda: db.copy_(hb, non_blocking=True), 3, stream)
    t_d2h = time_events(lambda: hb[:h_out].copy_(db[:h_out], non_blocking=True), 3, stream)
    rows["host_link_ceiling"] = {"h2d_GB/s": h_in / t_h2d / 1e6, "h2d_ms": t_h2d, "h2d_bytes": h_in,
                                 "d2h_GB/s": h_out / t_d2h / 1e6, "d2h_ms": t_d2h, "d2h_bytes": h_out,
                                 "note": "one cudaMemcpyAsync from/to pinned host memory of the e2e leg's "
                                         "per-step upload and download sizes"}
    del hb, db
    return rows


def run_gpu(args):
    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import visual_autoregressive_next_var_b300 as V

    inp = make_inputs(WORKLOADS[W1024], steps=(FINAL - 3, PREV, MID, FINAL))
    inp2k = make_inputs(WORKLOADS[W2K])
    mask2k, mask_ms = build_mask_2k(V)
    step = Step(V, dev, inp, inp2k, mask2k)
    stream = torch.cuda.current_stream(dev)
    flops_step = sum(step.flops.values())
    flops_equiv = sum(step.flops_dense_equiv.values())

    for _ in range(args.warmup):
        step.run(stream)
    torch.cuda.synchronize()
    barrier(ws)
    with ClockSampler(local, enabled=not args.no_clocks) as clk:
        if not args.no_clocks:
            t0 = time.perf_counter()            # keep the GPU busy (untimed) until the sampler runs
            while time.perf_counter() - t0 < 0.4:
                step.run(stream)
                torch.cuda.synchronize()
            barrier(ws)
        ms, per_row = time_step(step, args.steps, stream)
    ms_max = reduce_max(ms, ws, dev)
    st = V.var_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({V.var_status_string(st)})")
    peaks = load_peaks()
    value = ws * flops_step / ms_max / 1e9

    # per-row figures inside the timed region
    rows = {}
    for name, t in zip(ROW_NAMES, per_row):
        r = {"ms": t, "kernel": KERNEL_NAMES[name]}
        if name in step.flops:
            r["TFLOP/s"] = step.flops[name] / t / 1e9
            r["frac_tensor"] = r["TFLOP/s"] / peaks["bf16_tflops_sustained"]       # timed inside the long step
            r["frac_tensor_of_burst"] = r["TFLOP/s"] / peaks["bf16_tflops"]
            r["effective_dense_equiv_TFLOP/s"] = step.flops_dense_equiv[name] / t / 1e9
        else:
            r["GB/s"] = step.bytes[name] / t / 1e6
            r["frac_hbm"] = r["GB/s"] / peaks["hbm_gbs"]
        rows[name] = r
    rows["attn_blocksparse_2k"]["density"] = step.sparse_pairs / (step.N2 * step.L2)
    rows["block_mask_build_and_plan_2k_host_once"] = {"ms": mask_ms}
    dom = max(range(len(ROW_NAMES)), key=lambda i: per_row[i])
    dom_name = ROW_NAMES[dom]
    if dom_name in step.flops:
        achieved = step.flops[dom_name] / per_row[dom] / 1e9
        # the kernel is timed inside a step of ~3 ms of back-to-back tensor work,
        # so its peak is the sustained cuBLAS figure (the burst one is beside it)
        roof = {"kernel": KERNEL_NAMES[dom_name], "row": dom_name, "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops_sustained"],
                "peak_source": f"{peaks['source']} dense bf16 sustained (cuBLAS, seconds-long loop under the "
                               "power cap)",
                "frac_of_burst": achieved / peaks["bf16_tflops"],
                "traffic": ncu_traffic(TRAFFIC_KEYS[dom_name]) if dom_name in TRAFFIC_KEYS else None,
                "algorithmic_flops_per_launch": step.flops[dom_name], "launch_ms": per_row[dom]}
    else:
        achieved = step.bytes[dom_name] / per_row[dom] / 1e6
        roof = {"kernel": KERNEL_NAMES[dom_name], "row": dom_name, "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "peak_source": f"{peaks['source']} copy", "traffic": None,
                "algorithmic_bytes_per_launch": step.bytes[dom_name], "launch_ms": per_row[dom]}

    # end to end through the public API with host buffers: every step uploads its
    # inputs (the 1024px Q's, K/V cache and hidden states, the 40x40 output, the
    # 2K Q and K/V cache) from pinned host memory and downloads its results.
    # Pipelined over two device buffer sets and three streams, as a run of steps
    # would be: step i+1's upload and step i-1's download overlap step i's
    # kernels.  The serial order (upload, kernels, download, one stream) is
    # reported beside it.
    host = {"q64": inp.q[FINAL].pin_memory(), "q48": inp.q[MID].pin_memory(), "k": inp.k.pin_memory(),
            "v": inp.v.pin_memory(), "x48": inp.x[MID].pin_memory(), "x64": inp.x[FINAL].pin_memory(),
            "prev40": step.prev.cpu().pin_memory(), "q2k": inp2k.q[step.st2].pin_memory(),
            "k2k": inp2k.k.pin_memory(), "v2k": inp2k.v.pin_memory()}
    outs = [{k: torch.empty(t.shape, dtype=t.dtype).pin_memory() for k, t in step.results().items()}
            for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
    sets = [step, Step(V, dev, inp, inp2k, mask2k)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def upload(st, strm):
        with torch.cuda.stream(strm):
            for d, h in st.uploads(host):
                d.copy_(h, non_blocking=True)

    def download(st, o, strm):
        with torch.cuda.stream(strm):
            for k, t in st.results().items():
                o[k].copy_(t, non_blocking=True)

    def e2e_serial():
        upload(step, stream)
        step.run(stream)
        download(step, outs[0], stream)

    def e2e_pipelined(n):
        for i in range(n):
            b = i & 1
            st = sets[b]
            if i >= 2:
                s_in.wait_event(ev_comp[b])          # step i-2 has finished reading this set
            upload(st, s_in)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])         # step i-2's results are downloaded
            st.run(stream)
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            download(st, outs[b], s_out)
            ev_out[b].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    e2e_steps = max(4, min(args.steps, 10))
    for _ in range(2):
        e2e_serial()
    e2e_pipelined(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_serial()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_serial = reduce_max(e0.elapsed_time(e1) / e2e_steps, ws, dev)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    e0.record(stream)
    s_in.wait_stream(stream)                         # the uploads start after e0
    e2e_pipelined(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = reduce_max(e0.elapsed_time(e1) / e2e_steps, ws, dev)
    del sets[1]

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": step_config(),
        "value_note": f"algorithmic: {flops_step / 1e9:.1f} GFLOP executed per step (4 D per computed "
                      "(query, key) pair); the dense-equivalent effective figure "
                      f"({flops_equiv / 1e9:.1f} GFLOP: every attention variant counted as full dense "
                      f"attention) is {ws * flops_equiv / ms_max / 1e9:.1f} TFLOP/s and is not a fraction "
                      "of any peak",
        "effective_dense_equiv_TFLOP/s": ws * flops_equiv / ms_max / 1e9,
        "roofline": roof,
        "e2e": {"value": ws * flops_step / ms_e2e / 1e9, "unit": "TFLOP/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "mode": f"pipelined over {e2e_steps} steps: upload of step i+1 and download of step i-1 "
                        "overlap step i's kernels (two device buffer sets, three streams)",
                "serial_ms_per_step": ms_serial},
        "gpu_launches": args.steps * LAUNCHES_PER_STEP,
        "clocks": clk.summary(),
        "rows": rows,
    }
    if not args.no_rows:
        line["rows"].update(extra_rows(V, dev, step, inp, max(5, min(args.steps, 20)), peaks, (h2d, d2h)))
    if rank == 0 and ws == 1 and not args.no_cpu:
        tf, dt, n_rows, thr = oracle_sample(inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": f"{n_rows} random query rows of the 1024px final step's dense attention "
                                          f"(of {2 * 16 * step.N[FINAL]}), {dt:.1f} s; throughput per FLOP"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("varattn", "reference"), default="varattn")
    ap.add_argument("--no-rows", action="store_true", help="skip the separate per-kernel measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-clocks", action="store_true", help="no nvidia-smi sampling (profiler runs)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=3.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
