#!/usr/bin/env python3
"""Benchmark of the next-scale VAR attention hot path on B300.

Headline (one JSON line on rank 0): final-scale attention of the 1024px
schedule -- 4,096 queries (64x64 grid) of a CFG pair (batch 2), 16 heads,
head_dim 128, attending a 10,521-token cache -- in ms and TFLOP/s through the
C ABI (var_attn_dense), with:
  roofline      the attention kernel against the measured dense bf16 peak
  e2e           the same call with host buffers (pinned H2D of Q/K/V and D2H
                of O inside the timed region)
  rows          every other hot-path kernel on its own workload's final scale
                (pivot select + pruned attention + restore at 64x64 r=0.2;
                block-sparse attention of the 2K schedule), each timed alone
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload
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
HEADLINE = "dense_1024px"


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


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "visual_autoregressive_next_var_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, units: float):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, scaled
    to `units` of work, or None when absent or taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e["dram_bytes"] * units / e["units"]


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


def time_loop(fn, steps: int, stream) -> float:
    """Mean ms per call of fn() over `steps` calls, CUDA events on `stream`."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_calibrate(w, inp, step, budget_s: float):
    """Number of query rows of `step` the oracle computes in about budget_s."""
    import oracle
    q = inp.q[step]
    B, H, N, D = q.shape
    L = cache_len(w.sides, step)
    oracle.attention(q, inp.k, inp.v, L, rows=np.arange(2))        # load + warm
    n = 8
    while True:
        t0 = time.perf_counter()
        oracle.attention(q, inp.k, inp.v, L, rows=np.arange(n) * (B * H * N // n))
        dt = time.perf_counter() - t0
        if dt >= 0.25 * budget_s or n >= B * H * N:
            return int(max(1, min(B * H * N, n * budget_s / max(dt, 1e-6))))
        n = min(B * H * N, 4 * n)


def oracle_run(w, inp, step, n_rows: int, seed: int = 0):
    """Time the oracle on n_rows random query rows of `step`: (TFLOP/s, s, threads)."""
    import oracle
    q = inp.q[step]
    B, H, N, D = q.shape
    L = cache_len(w.sides, step)
    rows = np.sort(np.random.default_rng(seed).choice(B * H * N, size=n_rows, replace=False))
    t0 = time.perf_counter()
    oracle.attention(q, inp.k, inp.v, L, rows=rows)
    dt = time.perf_counter() - t0
    return n_rows * 4.0 * L * D / dt / 1e12, dt, oracle.num_threads()


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    step = w.steps[-1]
    inp = make_inputs(w, steps=(step,))
    per_step = min(args.ref_seconds, 150.0 / (args.steps + args.warmup))
    n_rows = oracle_calibrate(w, inp, step, per_step)
    vals = []
    for i in range(args.warmup + args.steps):
        tf, dt, thr = oracle_run(w, inp, step, n_rows, seed=i)
        if i >= args.warmup:
            vals.append((tf, dt))
    value = statistics.median(v for v, _ in vals)
    ms = statistics.median(dt for _, dt in vals) * 1e3
    q = inp.q[step]
    B, H, N, D = q.shape
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": B, "heads": H, "head_dim": D, "queries": N,
                   "keys": cache_len(w.sides, step)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"{n_rows} random query rows of the final step per step "
                                   f"(of {B * H * N}); throughput scaled per FLOP"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def bench_rows(V, dev, stream, steps: int):
    """Time every non-headline kernel of the hot path on its own workload."""
    rows = {}
    peaks = load_peaks()
    # --- pruned final step of the 1024px schedule: pivot + pruned attention + restore
    w = WORKLOADS["pruned_1024px"]
    inp = make_inputs(w, steps=(11, 12))
    B, H, D = w.batch, w.heads, w.head_dim
    p = V.problem(B, H, D, w.sides)
    step = 12
    x = inp.x[step].to(dev)
    N, Cc = x.shape[1], x.shape[2]
    K = V.var_keep_count(N, 1, 5)
    q = inp.q[step].to(dev)
    k, v = inp.k.to(dev), inp.v.to(dev)
    prev = torch.randn((B, H, 48 * 48, D), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16).to(dev)
    wsb = torch.empty(V.var_pivot_workspace_bytes(p, step, Cc), dtype=torch.uint8, device=dev)
    idx = torch.empty((B, K), dtype=torch.int32, device=dev)
    oc = torch.empty((B, H, K, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    L = cache_len(w.sides, step)

    def piv():
        V.var_pivot_select(p, step, x, K, idx, wsb, stream=stream)

    def pru():
        V.var_attn_pruned(p, step, q, k, v, idx, K, oc, stream=stream)

    def res():
        V.var_restore_scatter(p, step, prev, oc, idx, K, out, stream=stream)

    for f in (piv, pru, res):
        for _ in range(3):
            f()
    t_piv = time_loop(piv, steps, stream)
    t_pru = time_loop(pru, steps, stream)
    t_res = time_loop(res, steps, stream)
    fl_pru = 4.0 * B * H * K * L * D
    fl_dense_eq = 4.0 * B * H * N * L * D
    piv_bytes = x.numel() * 2 + B * K * 4
    res_bytes = (prev.numel() + oc.numel() + out.numel()) * 2 + B * K * 4
    rows["pivot_select_64x64"] = {"ms": t_piv, "bytes": piv_bytes, "GB/s": piv_bytes / t_piv / 1e6,
                                  "frac_hbm": piv_bytes / t_piv / 1e6 / peaks["hbm_gbs"]}
    rows["attn_pruned_64x64_r0.2"] = {"ms": t_pru, "TFLOP/s": fl_pru / t_pru / 1e9,
                                      "frac_tensor": fl_pru / t_pru / 1e9 / peaks["bf16_tflops"],
                                      "dense_equiv_TFLOP/s": fl_dense_eq / t_pru / 1e9}
    rows["restore_scatter_48to64"] = {"ms": t_res, "bytes": res_bytes, "GB/s": res_bytes / t_res / 1e6,
                                      "frac_hbm": res_bytes / t_res / 1e6 / peaks["hbm_gbs"]}
    t_chain = t_piv + t_pru + t_res
    rows["pruned_step_64x64_total"] = {"ms": t_chain, "dense_equiv_TFLOP/s": fl_dense_eq / t_chain / 1e9}
    del x, q, k, v, prev, wsb, idx, oc, out
    # --- block-sparse final step of the 2K schedule
    w = WORKLOADS["blocksparse_2k"]
    step = w.steps[-1]
    B, H, D = w.batch, w.heads, w.head_dim
    p = V.problem(B, H, D, w.sides)
    try:
        row_ptr, entries, sink_len = V.var_block_mask_build(p, step, w.qblock_side, w.radius, w.sink_max_side)
        inp = make_inputs(w)
        q, k, v = inp.q[step].to(dev), inp.k.to(dev), inp.v.to(dev)
        o = torch.empty_like(q)
        rp = torch.as_tensor(row_ptr, device=dev)
        en = torch.as_tensor(entries, device=dev)
        m = V.block_mask_struct(w.qblock_side, rp, en, sink_len)

        def bs():
            V.var_attn_blocksparse(p, step, q, k, v, m, o, stream=stream)

        for _ in range(3):
            bs()
        t_bs = time_loop(bs, steps, stream)
        N = q.shape[2]
        L = cache_len(w.sides, step)
        # algorithmic FLOPs: 4*D per kept (query, key) pair, from the CSR
        kept_pairs = 0
        sides = w.sides
        for qb in range(len(row_ptr) - 1):
            nk = sink_len
            for e in entries[row_ptr[qb]:row_ptr[qb + 1]]:
                sc, u, vv = e >> 24, (e >> 12) & 0xFFF, e & 0xFFF
                s = sides[sc]
                nk += (min(s, u * 8 + 8) - u * 8) * (min(s, vv * 8 + 8) - vv * 8)
            kept_pairs += nk * 64
        fl = 4.0 * B * H * kept_pairs * D
        rows["attn_blocksparse_2k"] = {"ms": t_bs, "TFLOP/s": fl / t_bs / 1e9,
                                       "frac_tensor": fl / t_bs / 1e9 / peaks["bf16_tflops"],
                                       "dense_equiv_TFLOP/s": 4.0 * B * H * N * L * D / t_bs / 1e9,
                                       "density": kept_pairs / (N * L)}
    except V.VarError as e:
        rows["attn_blocksparse_2k"] = {"unavailable": str(e)}
    return rows


def run_gpu(args):
    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import visual_autoregressive_next_var_b300 as V

    w = WORKLOADS[args.workload]
    step = w.steps[-1]
    inp = make_inputs(w, steps=(step,))
    q_h = inp.q[step]
    B, H, N, D = q_h.shape
    L = cache_len(w.sides, step)
    p = V.problem(B, H, D, w.sides, kv_capacity=inp.k.shape[2])
    q, k, v = q_h.to(dev), inp.k.to(dev), inp.v.to(dev)
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    flops = 4.0 * B * H * N * L * D
    in_bytes = (q.numel() + k.numel() + v.numel()) * 2

    def step_fn():
        V.var_attn_dense(p, step, q, k, v, o, stream=stream)

    for _ in range(args.warmup):
        step_fn()
    torch.cuda.synchronize()
    barrier(ws)
    with ClockSampler(local, enabled=not args.no_clocks) as clk:
        if not args.no_clocks:
            # keep the GPU busy (untimed) until the sampler is producing, then time
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < 0.4:
                step_fn()
                torch.cuda.synchronize()
            barrier(ws)
        ms = time_loop(step_fn, args.steps, stream)
    ms_max = reduce_max(ms, ws, dev)
    st = V.var_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({V.var_status_string(st)})")
    peaks = load_peaks()
    achieved = flops / ms / 1e9                      # TFLOP/s of this rank's kernel
    value = ws * flops / ms_max / 1e9

    # end to end through the public API with host buffers
    qp = q_h.pin_memory()
    kp = inp.k.pin_memory()
    vp = inp.v.pin_memory()
    op = torch.empty(o.shape, dtype=o.dtype).pin_memory()

    def e2e_fn():
        q.copy_(qp, non_blocking=True)
        k.copy_(kp, non_blocking=True)
        v.copy_(vp, non_blocking=True)
        V.var_attn_dense(p, step, q, k, v, o, stream=stream)
        op.copy_(o, non_blocking=True)

    for _ in range(2):
        e2e_fn()
    e2e_steps = max(3, min(args.steps, 10))
    ms_e2e = reduce_max(time_loop(e2e_fn, e2e_steps, stream), ws, dev)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": B, "heads": H, "head_dim": D, "queries": N,
                   "keys": L, "kv_tokens_total": inp.k.shape[2],
                   "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB of Q/K/V)",
                   "per_gpu": "each rank runs the whole workload"},
        "roofline": {"kernel": "attn_kernel<128, dense>", "bound": "tensor", "achieved": achieved,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"],
                     "peak_source": f"{peaks['source']} dense bf16 burst (cuBLAS)",
                     "traffic": ncu_traffic("attn_kernel<128, dense>:" + w.name, 1.0),
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": ws * flops / ms_e2e / 1e9, "unit": "TFLOP/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": o.numel() * 2},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_rows:
        line["rows"] = bench_rows(V, dev, stream, max(5, args.steps // 2))
    if rank == 0 and ws == 1 and not args.no_cpu:
        n_rows = oracle_calibrate(w, inp, step, args.cpu_seconds)
        tf, dt, thr = oracle_run(w, inp, step, n_rows)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": f"{n_rows} random query rows of the final step "
                                          f"(of {B * H * N}), {dt:.1f} s; throughput per FLOP"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("varattn", "reference"), default="varattn")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--no-rows", action="store_true", help="skip the per-kernel rows")
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
