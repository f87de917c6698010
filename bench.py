#!/usr/bin/env python3
"""Benchmark of the next-scale VAR attention hot path on B300.

One step = the final scale of the 1024px schedule (64x64 = 4,096 queries of a
CFG pair, 16 heads, head_dim 128, attending a 10,521-token cache) taken
through every row of the hot path, all through the C ABI:
  dense attention      var_attn_dense
  pivot selection      var_pivot_select      (hidden states 4096 x 2048, keep 20 %)
  pruned attention     var_attn_pruned
  restore + scatter    var_restore_scatter   (from the 48x48 step's output)
  block-sparse         var_attn_blocksparse  (sinks <= 16, +-2 block window;
                                              the mask is built once on the host)
`value` is the step's dense-equivalent TFLOP/s: the dense FLOPs of the three
attention variants (each computes the final-scale attention) divided by the
step time.  The JSON line also carries:
  rows          per-kernel times inside the timed region (CUDA events between
                the calls) and separate measurements: the small kernels from a
                CUDA graph after an L2 flush, the 2K block-sparse workload, the
                256px schedule
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
STEP_WORKLOAD = "pruned_1024px"      # tensors of the 1024px schedule (CFG pair, sink) + hidden states
FINAL = 12                           # the 64x64 step
KEEP = (1, 5)                        # keep ratio at 64x64
QBLOCK, RADIUS, SINK_SIDE = 8, 2, 16
ROW_NAMES = ("attn_dense", "pivot_select", "attn_pruned", "restore_scatter", "attn_blocksparse")
LAUNCHES_PER_STEP = 7                # dense 1, pivot 3, pruned 1, restore 1, block-sparse 1


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
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# The sources that decide what the attention kernels do and launch: the kernel,
# its PTX wrappers, the shared header, both launchers and the public header.
ATTN_SOURCES = ("visual_autoregressive_next_var_b300/csrc/attn_kernel.cuh",
                "visual_autoregressive_next_var_b300/csrc/ptx.cuh",
                "visual_autoregressive_next_var_b300/csrc/internal.h",
                "visual_autoregressive_next_var_b300/csrc/attn.cu",
                "visual_autoregressive_next_var_b300/csrc/blocksparse.cu",
                "include/varattn.h")


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
    """Device buffers and the call sequence of one step."""

    def __init__(self, V, dev, inp):
        w = WORKLOADS[STEP_WORKLOAD]
        self.V = V
        self.w = w
        B, H, D = w.batch, w.heads, w.head_dim
        self.p = V.problem(B, H, D, w.sides, kv_capacity=inp.k.shape[2])
        self.N = w.sides[FINAL] ** 2
        self.L = cache_len(w.sides, FINAL)
        self.K = V.var_keep_count(self.N, *KEEP)
        self.q = inp.q[FINAL].to(dev)
        self.q_src = inp.q[FINAL - 3].to(dev)     # the 32x32 step whose attention guides the pivots
        self.k = inp.k.to(dev)
        self.v = inp.v.to(dev)
        self.x = inp.x[FINAL].to(dev)
        self.C = self.x.shape[2]
        # the previous (48x48) step's output: dense attention, computed once
        q11 = inp.q[FINAL - 1].to(dev)
        self.prev = torch.empty_like(q11)
        V.var_attn_dense(self.p, FINAL - 1, q11, self.k, self.v, self.prev)
        del q11
        self.o_dense = torch.empty_like(self.q)
        self.ws = torch.empty(V.var_pivot_workspace_bytes(self.p, FINAL, self.C), dtype=torch.uint8, device=dev)
        self.idx = torch.empty((B, self.K), dtype=torch.int32, device=dev)
        self.oc = torch.empty((B, H, self.K, D), dtype=torch.bfloat16, device=dev)
        self.o_pruned = torch.empty_like(self.q)
        self.o_sparse = torch.empty_like(self.q)
        t0 = time.perf_counter()
        rp, en, sink = V.var_block_mask_build(self.p, FINAL, QBLOCK, RADIUS, SINK_SIDE)
        self.rp = torch.as_tensor(rp, device=dev)
        self.en = torch.as_tensor(en, device=dev)
        self.plan = [torch.as_tensor(a, device=dev) for a in V.var_block_mask_plan(self.p, FINAL, QBLOCK, rp, en, sink)]
        self.mask_build_ms = (time.perf_counter() - t0) * 1e3
        self.mask = V.block_mask_struct(QBLOCK, self.rp, self.en, sink, self.plan)
        self.sparse_pairs = mask_kept_pairs(w.sides, rp, en, sink, QBLOCK)
        self.flops_dense = flops_attn(B, H, self.N, self.L, D)
        self.flops_pruned = flops_attn(B, H, self.K, self.L, D)
        self.flops_sparse = 4.0 * B * H * self.sparse_pairs * D
        self.bytes_pivot = self.x.numel() * 2 + self.idx.numel() * 4
        self.bytes_restore = (self.prev.numel() + self.oc.numel() + self.o_pruned.numel()) * 2 + self.idx.numel() * 4

    def calls(self, stream=None):
        V, p = self.V, self.p
        return (
            lambda: V.var_attn_dense(p, FINAL, self.q, self.k, self.v, self.o_dense, stream=stream),
            lambda: V.var_pivot_select(p, FINAL, self.x, self.K, self.idx, self.ws, stream=stream),
            lambda: V.var_attn_pruned(p, FINAL, self.q, self.k, self.v, self.idx, self.K, self.oc, stream=stream),
            lambda: V.var_restore_scatter(p, FINAL, self.prev, self.oc, self.idx, self.K, self.o_pruned,
                                          stream=stream),
            lambda: V.var_attn_blocksparse(p, FINAL, self.q, self.k, self.v, self.mask, self.o_sparse,
                                           stream=stream),
        )

    def run(self, stream=None):
        for c in self.calls(stream):
            c()


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


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_sample(inp, budget_s: float, seed: int = 0):
    """Time the oracle on random query rows of the final step's dense attention,
    sized to about budget_s: (TFLOP/s, seconds, rows, threads)."""
    import oracle
    w = WORKLOADS[STEP_WORKLOAD]
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


def step_config(inp):
    w = WORKLOADS[STEP_WORKLOAD]
    q = inp.q[FINAL]
    B, H, N, D = q.shape
    return {"workload": "final_step_1024px", "schedule": list(w.sides), "batch": B, "heads": H,
            "head_dim": D, "queries": N, "keys": cache_len(w.sides, FINAL), "channels": w.channels,
            "keep": f"{KEEP[0]}/{KEEP[1]}", "block_mask": f"qblock {QBLOCK}, radius {RADIUS}, sinks <= {SINK_SIDE}",
            "rows": list(ROW_NAMES)}


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    inp = make_inputs(WORKLOADS[STEP_WORKLOAD], steps=(FINAL,))
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
        "data": "synthetic", "config": step_config(inp),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"{n_rows} random query rows of the final step's dense attention "
                                   "per step; throughput per FLOP"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def extra_rows(V, dev, step: Step, iters: int, peaks):
    """Separate measurements: small kernels alone, the 2K block-sparse workload,
    the 256px schedule."""
    rows = {}
    flush = L2Flush(dev)
    calls = step.calls()
    t = time_graph(calls[1], iters, flush)
    rows["pivot_select_64x64_alone"] = {"ms": t, "GB/s": step.bytes_pivot / t / 1e6,
                                        "frac_hbm": step.bytes_pivot / t / 1e6 / peaks["hbm_gbs"],
                                        "timing": "CUDA graph replay after an L2 flush"}
    t = time_graph(calls[3], iters, flush)
    rows["restore_scatter_48to64_alone"] = {"ms": t, "GB/s": step.bytes_restore / t / 1e6,
                                            "frac_hbm": step.bytes_restore / t / 1e6 / peaks["hbm_gbs"],
                                            "timing": "CUDA graph replay after an L2 flush"}
    # the pruned step with the outputs written in place (no compact buffer)
    def fused():
        step.V.var_attn_pruned_scatter(step.p, FINAL, step.q, step.k, step.v, step.idx, step.K, step.o_pruned)
        step.V.var_restore_fill(step.p, FINAL, step.prev, step.idx, step.K, step.o_pruned)

    side = torch.cuda.Stream()

    def fused_overlapped():
        # disjoint rows: the HBM-bound fill runs on a second stream beside the attention
        cur = torch.cuda.current_stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            step.V.var_restore_fill(step.p, FINAL, step.prev, step.idx, step.K, step.o_pruned)
        step.V.var_attn_pruned_scatter(step.p, FINAL, step.q, step.k, step.v, step.idx, step.K, step.o_pruned)
        cur.wait_stream(side)

    t = time_graph(fused, iters, flush)
    t_ov = time_graph(fused_overlapped, iters, flush)
    t_chain = time_graph(lambda: (calls[2](), calls[3]()), iters, flush)
    rows["pruned_attn_and_restore_fused"] = {"ms": t, "overlapped_ms": t_ov, "unfused_ms": t_chain,
                                             "dense_equiv_TFLOP/s": step.flops_dense / t_ov / 1e9,
                                             "timing": "CUDA graph replay after an L2 flush; overlapped = "
                                                       "fill on a second stream beside the attention"}
    # attention-guided pivots (ARVAR): the 32x32 step's row statistics and saliency
    src = FINAL - 3
    B, H, Ns, D = step.q_src.shape
    o_src = torch.empty_like(step.q_src)
    lse = torch.empty((B, H, Ns), dtype=torch.float32, device=dev)
    sal = torch.empty((B, H, Ns), dtype=torch.float32, device=dev)
    gws = torch.empty(step.V.var_guided_pivot_workspace_bytes(step.p, FINAL), dtype=torch.uint8, device=dev)
    gidx = torch.empty_like(step.idx)
    t_plain = time_graph(lambda: step.V.var_attn_dense(step.p, src, step.q_src, step.k, step.v, o_src), iters, flush)
    t_lse = time_graph(lambda: step.V.var_attn_dense_lse(step.p, src, step.q_src, step.k, step.v, o_src, lse),
                       iters, flush)
    t_sal = time_graph(lambda: step.V.var_attn_saliency(step.p, src, step.q_src, step.k, lse, sal), iters, flush)
    t_sel = time_graph(lambda: step.V.var_guided_pivot_select(step.p, FINAL, src, sal, step.K, gidx, gws),
                       iters, flush)
    L_src = cache_len(WORKLOADS[STEP_WORKLOAD].sides, src)
    fl_sal = 2.0 * B * H * Ns * Ns * D            # S^T = K_self Q^T
    rows["guided_pivot_from_32x32"] = {
        "ms": t_sal + t_sel, "saliency_ms": t_sal, "select_ms": t_sel,
        "saliency_TFLOP/s": fl_sal / t_sal / 1e9,
        "source_dense_ms": t_plain, "source_dense_with_lse_ms": t_lse,
        "note": f"source step 32x32 ({Ns} queries, {L_src} keys) -> 64x64, keep 1/5; the row "
                "statistics are written by the source step's own dense attention",
        "timing": "CUDA graph replay after an L2 flush"}
    # SparVAR dynamic pattern: the 32x32 step's block scores decide the 64x64 step's mask
    d_sv, tau_sv = FINAL - 3, 0.8
    U_sv, _ = step.V.var_sparvar_units(step.p, d_sv, SINK_SIDE)
    sv_ws = torch.empty(step.V.var_sparvar_workspace_bytes(step.p, d_sv), dtype=torch.uint8, device=dev)
    nqb_sv = (int(round(step.q_src.shape[2] ** 0.5)) // 8) ** 2
    sv_sc = torch.empty((nqb_sv, U_sv), dtype=torch.float64, device=dev)
    t_sc = time_graph(lambda: step.V.var_sparvar_scores(step.p, d_sv, SINK_SIDE, step.q_src, step.k, sv_ws, sv_sc),
                      iters, flush)
    t0 = time.perf_counter()
    A = sv_sc.cpu().numpy()
    rp, en, sink = step.V.var_sparvar_mask_build(step.p, d_sv, FINAL, SINK_SIDE, A, tau_sv)
    sv_plan = [torch.as_tensor(a, device=dev) for a in step.V.var_block_mask_plan(step.p, FINAL, QBLOCK, rp, en, sink)]
    t_host = (time.perf_counter() - t0) * 1e3
    sv_rp, sv_en = torch.as_tensor(rp, device=dev), torch.as_tensor(en, device=dev)
    sv_mask = step.V.block_mask_struct(QBLOCK, sv_rp, sv_en, sink, sv_plan)
    t_sv = time_graph(lambda: step.V.var_attn_blocksparse(step.p, FINAL, step.q, step.k, step.v, sv_mask,
                                                           step.o_sparse), iters, flush)
    pairs = mask_kept_pairs(WORKLOADS[STEP_WORKLOAD].sides, rp, en, sink, QBLOCK)
    fl_sv = 4.0 * step.q.shape[0] * step.q.shape[1] * pairs * step.q.shape[3]
    rows["sparvar_dynamic_mask_32_to_64"] = {
        "scores_ms": t_sc, "host_select_map_plan_ms": t_host, "attn_ms": t_sv,
        "density": pairs / (step.N * step.L), "TFLOP/s": fl_sv / t_sv / 1e9,
        "dense_equiv_TFLOP/s": step.flops_dense / t_sv / 1e9, "units": U_sv, "tau": tau_sv,
        "note": "decision step 32x32: block scores (dense attention on unit-indicator values, "
                f"{U_sv} units) -> host selection + index mapping -> block-sparse attention of the 64x64 step",
        "timing": "CUDA graph replay after an L2 flush; host part timed once"}
    # Branch Halving: the conditional half only, its rows repeated
    t = time_graph(lambda: step.V.var_attn_dense_halved(step.p, FINAL, step.q, step.k, step.v, step.o_dense),
                   iters, flush)
    rows["attn_dense_branch_halved"] = {"ms": t, "TFLOP/s": step.flops_dense / 2 / t / 1e9,
                                        "frac_tensor": step.flops_dense / 2 / t / 1e9 / peaks["bf16_tflops"],
                                        "dense_equiv_TFLOP/s": step.flops_dense / t / 1e9,
                                        "timing": "CUDA graph replay after an L2 flush"}
    # block-sparse attention on the 2K schedule (its own workload)
    w = WORKLOADS["blocksparse_2k"]
    st = w.steps[-1]
    B, H, D = w.batch, w.heads, w.head_dim
    p = V.problem(B, H, D, w.sides)
    rp, en, sink = V.var_block_mask_build(p, st, w.qblock_side, w.radius, w.sink_max_side)
    inp = make_inputs(w)
    q, k, v = inp.q[st].to(dev), inp.k.to(dev), inp.v.to(dev)
    del inp
    o = torch.empty_like(q)
    plan = [torch.as_tensor(a, device=dev) for a in V.var_block_mask_plan(p, st, w.qblock_side, rp, en, sink)]
    m = V.block_mask_struct(w.qblock_side, torch.as_tensor(rp, device=dev), torch.as_tensor(en, device=dev), sink,
                            plan)
    stream = torch.cuda.current_stream(dev)

    def bs():
        V.var_attn_blocksparse(p, st, q, k, v, m, o, stream=stream)

    for _ in range(3):
        bs()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(5, iters)
    e0.record(stream)
    for _ in range(n):
        bs()
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / n
    N, L = q.shape[2], cache_len(w.sides, st)
    pairs = mask_kept_pairs(w.sides, rp, en, sink, w.qblock_side)
    fl = 4.0 * B * H * pairs * D
    rows["attn_blocksparse_2k"] = {"ms": t, "TFLOP/s": fl / t / 1e9, "frac_tensor": fl / t / 1e9 / peaks["bf16_tflops"],
                                   "dense_equiv_TFLOP/s": flops_attn(B, H, N, L, D) / t / 1e9,
                                   "density": pairs / (N * L)}
    del q, k, v, o
    # the whole 256px schedule, dense (launch-bound)
    w = WORKLOADS["dense_256px"]
    inp = make_inputs(w)
    B, H, D = w.batch, w.heads, w.head_dim
    p = V.problem(B, H, D, w.sides)
    k, v = inp.k.to(dev), inp.v.to(dev)
    qs = {s: inp.q[s].to(dev) for s in w.steps}
    os_ = {s: torch.empty_like(qs[s]) for s in w.steps}

    def sched():
        for s in w.steps:
            V.var_attn_dense(p, s, qs[s], k, v, os_[s])

    t = time_graph(sched, iters, flush)
    fl = sum(flops_attn(B, H, w.sides[s] ** 2, cache_len(w.sides, s), D) for s in w.steps)
    rows["schedule_256px_dense_10_steps"] = {"ms": t, "TFLOP/s": fl / t / 1e9, "launches": len(w.steps),
                                             "timing": "CUDA graph replay after an L2 flush"}
    return rows


def run_gpu(args):
    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import visual_autoregressive_next_var_b300 as V

    inp = make_inputs(WORKLOADS[STEP_WORKLOAD], steps=(FINAL - 3, FINAL - 1, FINAL))
    step = Step(V, dev, inp)
    stream = torch.cuda.current_stream(dev)
    flops_equiv = 3.0 * step.flops_dense
    flops_exec = step.flops_dense + step.flops_pruned + step.flops_sparse

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
    value = ws * flops_equiv / ms_max / 1e9

    # per-row figures inside the timed region
    row_flops = {"attn_dense": step.flops_dense, "attn_pruned": step.flops_pruned,
                 "attn_blocksparse": step.flops_sparse}
    row_bytes = {"pivot_select": step.bytes_pivot, "restore_scatter": step.bytes_restore}
    rows = {}
    for name, t in zip(ROW_NAMES, per_row):
        r = {"ms": t}
        if name in row_flops:
            r["TFLOP/s"] = row_flops[name] / t / 1e9
            r["frac_tensor"] = r["TFLOP/s"] / peaks["bf16_tflops"]
            r["dense_equiv_TFLOP/s"] = step.flops_dense / t / 1e9
        else:
            r["GB/s"] = row_bytes[name] / t / 1e6
            r["frac_hbm"] = r["GB/s"] / peaks["hbm_gbs"]
        rows[name] = r
    rows["attn_blocksparse"]["density"] = step.sparse_pairs / (step.N * step.L)
    rows["block_mask_build_and_plan_host_once"] = {"ms": step.mask_build_ms}
    dom = max(range(len(ROW_NAMES)), key=lambda i: per_row[i])
    dom_name = ROW_NAMES[dom]
    kernel_names = {"attn_dense": "attn_kernel<128, dense>", "attn_pruned": "attn_kernel<128, gather>",
                    "attn_blocksparse": "attn_kernel<128, sparse>", "pivot_select": "pivot kernels",
                    "restore_scatter": "restore_scatter_kernel<128>"}
    if dom_name in row_flops:
        achieved = row_flops[dom_name] / per_row[dom] / 1e9
        roof = {"kernel": kernel_names[dom_name], "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "peak_source": f"{peaks['source']} dense bf16 burst (cuBLAS)",
                "traffic": ncu_traffic(f"{kernel_names[dom_name]}:final_step_1024px"),
                "algorithmic_flops_per_launch": row_flops[dom_name],
                "launch_ms": per_row[dom]}
    else:
        achieved = row_bytes[dom_name] / per_row[dom] / 1e6
        roof = {"kernel": kernel_names[dom_name], "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} copy",
                "traffic": ncu_traffic(f"{kernel_names[dom_name]}:final_step_1024px"),
                "algorithmic_bytes_per_launch": row_bytes[dom_name], "launch_ms": per_row[dom]}

    # end to end through the public API with host buffers: every step uploads its
    # inputs (Q, the whole K/V cache, X, the previous step's output) from pinned
    # host memory and downloads its results.  Pipelined over two device buffer
    # sets and three streams, as a run of steps would be: step i+1's upload and
    # step i-1's download overlap step i's kernels.  The serial order (upload,
    # kernels, download, one stream) is reported beside it.
    host = {"q": inp.q[FINAL].pin_memory(), "k": inp.k.pin_memory(), "v": inp.v.pin_memory(),
            "x": inp.x[FINAL].pin_memory(), "prev": step.prev.cpu().pin_memory()}
    outs = [{"o_dense": torch.empty(step.o_dense.shape, dtype=torch.bfloat16).pin_memory(),
             "idx": torch.empty(step.idx.shape, dtype=torch.int32).pin_memory(),
             "o_pruned": torch.empty(step.o_pruned.shape, dtype=torch.bfloat16).pin_memory(),
             "o_sparse": torch.empty(step.o_sparse.shape, dtype=torch.bfloat16).pin_memory()} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
    sets = [step, Step(V, dev, inp)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def upload(st, strm):
        with torch.cuda.stream(strm):
            st.q.copy_(host["q"], non_blocking=True)
            st.k.copy_(host["k"], non_blocking=True)
            st.v.copy_(host["v"], non_blocking=True)
            st.x.copy_(host["x"], non_blocking=True)
            st.prev.copy_(host["prev"], non_blocking=True)

    def download(st, o, strm):
        with torch.cuda.stream(strm):
            o["o_dense"].copy_(st.o_dense, non_blocking=True)
            o["idx"].copy_(st.idx, non_blocking=True)
            o["o_pruned"].copy_(st.o_pruned, non_blocking=True)
            o["o_sparse"].copy_(st.o_sparse, non_blocking=True)

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

    cfg = step_config(inp)
    cfg["l2"] = "inputs larger than L2 (Q/K/V 206 MB + X 34 MB per step)"
    cfg["per_gpu"] = "each rank runs the whole workload"
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "value_note": "dense-equivalent: 3 x the final-scale dense attention FLOPs per step "
                      f"({flops_equiv / 1e9:.1f} GFLOP); executed algorithmic FLOPs "
                      f"{flops_exec / 1e9:.1f} GFLOP -> {ws * flops_exec / ms_max / 1e9:.1f} TFLOP/s",
        "roofline": roof,
        "e2e": {"value": ws * flops_equiv / ms_e2e / 1e9, "unit": "TFLOP/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "mode": f"pipelined over {e2e_steps} steps: upload of step i+1 and download of step i-1 "
                        "overlap step i's kernels (two device buffer sets, three streams)",
                "serial_ms_per_step": ms_serial},
        "gpu_launches": args.steps * LAUNCHES_PER_STEP,
        "clocks": clk.summary(),
        "rows": rows,
    }
    if not args.no_rows:
        line["rows"].update(extra_rows(V, dev, step, max(5, min(args.steps, 20)), peaks))
    if rank == 0 and ws == 1 and not args.no_cpu:
        tf, dt, n_rows, thr = oracle_sample(inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": f"{n_rows} random query rows of the final step's dense attention "
                                          f"(of {step.q.shape[0] * step.q.shape[1] * step.N}), {dt:.1f} s; "
                                          "throughput per FLOP"}
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
