"""The allocation-free pivot selection (var_pivot_select_noalloc) through the C
ABI, against the CPU oracle and the workspace version (var_pivot_select).

This entry point serves callers that cannot allocate device memory where they
select pivots (an engine that owns all device memory and passes a plug-in no
workspace; a latency-critical stream where cudaMalloc, which may synchronise
the device, is not allowed).  Two calls in a row on different inputs check
that the shared static scratch carries nothing over from one call to the
next.  This file sorts last so a run that stops at the first failure has run
every other test first; it also passes alone in a fresh process."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import randn_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _with_workspace(p, step, x, K):
    B, N, Cc = x.shape
    ws = torch.empty(V.var_pivot_workspace_bytes(p, step, Cc), dtype=torch.uint8, device=DEV)
    idx = torch.full((B, max(K, 1)), -1, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, N), dtype=torch.float32, device=DEV)
    V.var_pivot_select(p, step, x, K, idx, ws, sc)
    return idx, sc


def _no_alloc(p, step, x, K, want_scores=True):
    B, N, Cc = x.shape
    idx = torch.full((B, max(K, 1)), -1, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, N), dtype=torch.float32, device=DEV) if want_scores else None
    rc = V.lib().var_pivot_select_noalloc(C.byref(p), step, C.c_void_p(x.data_ptr()), Cc, K,
                                          C.c_void_p(idx.data_ptr()),
                                          None if sc is None else C.c_void_p(sc.data_ptr()),
                                          C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == V.VAR_OK, V.var_status_string(rc)
    return idx, sc


def test_no_alloc_pivot_select_matches_oracle_and_workspace_version_twice():
    sides = (1, 2, 4, 6, 8, 12, 16, 20, 24, 32, 40, 48, 64)
    p = V.problem(2, 16, 128, sides)
    cases = [(12, randn_bf16((2, 4096, 2048), 901), 819),    # 64x64 grid, keep 20 %
             (11, randn_bf16((2, 2304, 2048), 902), 921)]    # 48x48 grid, keep 40 %
    for step, x_cpu, K in cases:
        x = x_cpu.to(DEV)
        ref_idx, ref_sc = _with_workspace(p, step, x, K)
        got_idx, got_sc = _no_alloc(p, step, x, K)
        torch.cuda.synchronize()
        assert torch.equal(got_idx, ref_idx)                 # indices: bit for bit
        assert torch.equal(got_sc, ref_sc)
        o_idx, o_sc = oracle.pivot_select(x_cpu, K)          # the fp64 definition
        assert np.array_equal(got_idx.cpu().numpy(), o_idx)
        assert np.max(np.abs(got_sc.cpu().double().numpy() - o_sc) / o_sc) < 1e-4
    assert V.var_device_status() == 0


def test_no_alloc_without_scores_and_with_keep_zero():
    p = V.problem(2, 16, 128, (1, 2, 4, 6, 8, 12, 16, 20, 24, 32, 40, 48, 64))
    x_cpu = randn_bf16((2, 4096, 2048), 903)
    x = x_cpu.to(DEV)
    idx, _ = _no_alloc(p, 12, x, 819, want_scores=False)     # scores = NULL
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), oracle.pivot_select(x_cpu, 819)[0])
    idx0, sc0 = _no_alloc(p, 12, x, 0)                       # keep nothing: scores only
    torch.cuda.synchronize()
    _, o_sc = oracle.pivot_select(x_cpu, 0)
    assert np.max(np.abs(sc0.cpu().double().numpy() - o_sc) / o_sc) < 1e-4
    assert torch.all(idx0 == -1)                             # the index buffer is not touched
    assert V.var_device_status() == 0


def test_no_alloc_rejects_problems_beyond_its_scratch():
    p = V.problem(8, 1, 128, (1, 16))                        # batch 8 > 4
    x = torch.zeros((8, 256, 64), dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros((8, 4), dtype=torch.int32, device=DEV)
    rc = V.lib().var_pivot_select_noalloc(C.byref(p), 1, C.c_void_p(x.data_ptr()), 64, 4,
                                          C.c_void_p(idx.data_ptr()), None, None)
    assert rc == V.VAR_ERR_WORKSPACE
    q = V.problem(1, 1, 128, (1, 16))
    y = torch.zeros((1, 256, 8192), dtype=torch.bfloat16, device=DEV)   # channels 8192 > 4096
    rc = V.lib().var_pivot_select_noalloc(C.byref(q), 1, C.c_void_p(y.data_ptr()), 8192, 4,
                                          C.c_void_p(idx.data_ptr()), None, None)
    assert rc == V.VAR_ERR_WORKSPACE
