"""bench.py's host side on CPU: the reference (oracle) arm's JSON line and the
kept-pair count behind the block-sparse FLOP figures."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import oracle
import visual_autoregressive_next_var_b300 as V

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-seconds", "0.3"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("var_hot_path_step")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_kept_pairs_equal_the_oracle_token_mask():
    sides = (1, 2, 4, 6, 8, 12, 16, 20, 24, 32)
    step = len(sides) - 1
    p = V.problem(1, 1, 64, sides)
    for radius, sink in ((1, 8), (2, 16)):
        rp, en, sink_len = V.var_block_mask_build(p, step, 8, radius, sink)
        keep = oracle.block_mask_rows(oracle.mask_spec(sides, step, 8, radius, sink), 0, sides[step] ** 2)
        assert bench.mask_kept_pairs(sides, rp, en, sink_len, 8) == int(keep.sum())


def test_flops_attn_closed_form():
    assert bench.flops_attn(2, 16, 4096, 10521, 128) == 4.0 * 2 * 16 * 4096 * 10521 * 128
    assert abs(bench.flops_attn(2, 16, 4096, 10521, 128) - 706.05e9) < 0.01e9
