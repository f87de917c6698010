"""The debug build (-DVAR_DEBUG): it compiles, loads, exports every declared
entry point, and -- on a GPU -- reports a bad index list through the call's
status word instead of clamping or skipping it silently."""
import ctypes as C
import importlib.util
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build_debug():
    spec = importlib.util.spec_from_file_location(
        "_varattn_build", os.path.join(ROOT, "visual_autoregressive_next_var_b300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(debug=True)


def test_debug_build_compiles_and_exports_every_symbol():
    path = _build_debug()
    assert os.path.exists(path)
    import visual_autoregressive_next_var_b300 as V
    lib = C.CDLL(path)
    for name in V.header_functions():
        assert hasattr(lib, name), name


CHILD = r"""
import sys, torch
sys.path.insert(0, %r)
import visual_autoregressive_next_var_b300 as V
assert V.LIB_PATH.endswith("libvarattn_debug.so")
from var_synth import randn_bf16
dev = torch.device("cuda", 0)
sides, B, H, D = (1, 2, 4, 8, 16), 2, 2, 64
p = V.problem(B, H, D, sides)
L, N = 341, 256
q, k, v = (randn_bf16(s, 5 + i).to(dev) for i, s in enumerate(((B, H, N, D), (B, H, L, D), (B, H, L, D))))
word = torch.zeros(1, dtype=torch.int32, device=dev)
p.status = word.data_ptr()
ok = torch.tensor([[1, 5, 9], [0, 2, 255]], dtype=torch.int32, device=dev)
oc = torch.empty((B, H, 3, D), dtype=torch.bfloat16, device=dev)
V.var_attn_pruned(p, 4, q, k, v, ok, 3, oc)
assert V.var_check_status(word) == 0
bad = torch.tensor([[1, 5, 9], [0, 2, 256]], dtype=torch.int32, device=dev)         # 256 is past N
V.var_attn_pruned(p, 4, q, k, v, bad, 3, oc)
assert V.var_check_status(word) == V.VAR_ERR_INVALID_ARG
prev = randn_bf16((B, H, 64, D), 9).to(dev)
out = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
unsorted = torch.tensor([[1, 9, 5], [0, 2, 3]], dtype=torch.int32, device=dev)       # not ascending
V.var_restore_scatter(p, 4, prev, oc, unsorted, 3, out)
assert V.var_check_status(word) == V.VAR_ERR_INVALID_ARG
V.var_restore_scatter(p, 4, prev, oc, ok, 3, out)
assert V.var_check_status(word) == 0
assert V.var_device_status() == 0
print("DEBUG_OK")
"""


@pytest.mark.gpu
def test_debug_build_reports_bad_index_lists():
    _build_debug()
    env = dict(os.environ, VARATTN_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", CHILD % ROOT], capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0 and "DEBUG_OK" in r.stdout, r.stderr[-3000:]
