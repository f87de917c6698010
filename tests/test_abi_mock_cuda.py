"""Every VAR_ERR_CUDA branch of the C ABI, on the CPU.

The library reaches the CUDA runtime through one function table; the test hook
var_test_mock_cuda (include/varattn_test.h) swaps it for a mock that fakes a
device, runs no kernel and makes its n-th call fail.  For each entry point the
child process below counts the calls a valid invocation makes (none failing:
VAR_OK), then fails each of them in turn and records the status returned.
Every one must be VAR_ERR_CUDA: no CUDA failure may be swallowed, turned into
another code, or crash the host.  The mock runs in a child process so that no
fake value reaches a process that makes real CUDA calls."""
import ctypes as C
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FAKE = 0x7f0000100000          # a 256-byte-aligned address the mock never dereferences


def _cases(V):
    """(name, thunk) pairs: valid calls with fake device pointers."""
    L = V.lib()
    f = C.c_void_p(FAKE)
    fs = C.c_void_p(FAKE + 0x1000)                   # a caller-owned status word
    sides = (1, 2, 4, 6, 8, 12, 16, 20, 24, 32)
    p = V.problem(2, 4, 128, sides)
    p_st = V.problem(2, 4, 128, sides)
    p_st.status = FAKE + 0x1000
    p64 = V.problem(1, 3, 64, sides)
    ws_piv = L.var_pivot_workspace_bytes(C.byref(p), 9, 256)
    ws_gd = L.var_guided_pivot_workspace_bytes(C.byref(p), 9)
    ws_gx = L.var_guided_pivot_exact_workspace_bytes(C.byref(p), 9, 8)
    ws_sv = L.var_sparvar_workspace_bytes(C.byref(p), 9, 16)
    m = V.var_block_mask()
    m.qblock_side, m.n_qblocks, m.sink_len, m.nnz = 8, 16, 521, 64
    m.row_ptr, m.entries = FAKE, FAKE
    mp = V.var_block_mask()
    C.pointer(mp)[0] = m
    mp.n_squares, mp.plan_units = 4, 40
    mp.sq_ptr, mp.sq_units, mp.sq_order = FAKE, FAKE, FAKE
    out = C.c_int32()
    return [
        ("var_attn_dense", lambda: L.var_attn_dense(C.byref(p), 9, f, f, f, f, None)),
        ("var_attn_dense_d64", lambda: L.var_attn_dense(C.byref(p64), 9, f, f, f, f, None)),
        ("var_attn_dense_own_status", lambda: L.var_attn_dense(C.byref(p_st), 9, f, f, f, f, None)),
        ("var_attn_dense_lse", lambda: L.var_attn_dense_lse(C.byref(p), 9, f, f, f, f, f, None)),
        ("var_attn_dense_halved", lambda: L.var_attn_dense_halved(C.byref(p), 9, f, f, f, f, None)),
        ("var_pivot_select", lambda: L.var_pivot_select(C.byref(p), 9, f, 256, 204, f, f, f, ws_piv, None)),
        ("var_pivot_select_noalloc", lambda: L.var_pivot_select_noalloc(C.byref(p), 9, f, 256, 204, f, None, None)),
        ("var_attn_pruned", lambda: L.var_attn_pruned(C.byref(p), 9, f, f, f, f, 204, f, None)),
        ("var_attn_pruned_scatter", lambda: L.var_attn_pruned_scatter(C.byref(p), 9, f, f, f, f, 204, f, None)),
        ("var_restore_scatter", lambda: L.var_restore_scatter(C.byref(p), 9, f, f, f, 204, f, None)),
        ("var_restore_fill", lambda: L.var_restore_fill(C.byref(p), 9, f, f, 204, f, None)),
        ("var_pruned_in_place", lambda: L.var_pruned_in_place(C.byref(p), 9, f, f, f, f, f, 204, f, None)),
        ("var_pruned_in_place_fill_only", lambda: L.var_pruned_in_place(C.byref(p), 9, None, None, None, f, None,
                                                                        0, f, None)),
        ("var_pruned_step", lambda: L.var_pruned_step(C.byref(p), 9, f, 256, 204, f, f, f, f, f, f, f, ws_piv,
                                                      None)),
        ("var_pruned_step_fill_only", lambda: L.var_pruned_step(C.byref(p), 9, f, 256, 0, None, None, None, f,
                                                                None, f, None, 0, None)),
        ("var_attn_saliency", lambda: L.var_attn_saliency(C.byref(p), 8, f, f, f, f, None)),
        ("var_guided_pivot_select", lambda: L.var_guided_pivot_select(C.byref(p), 9, 8, f, 204, f, None, f, ws_gd,
                                                                      None)),
        ("var_guided_pivot_select_exact", lambda: L.var_guided_pivot_select_exact(C.byref(p), 9, 8, f, f, 204, f, f,
                                                                                  f, ws_gx, None)),
        ("var_attn_blocksparse", lambda: L.var_attn_blocksparse(C.byref(p), 9, f, f, f, C.byref(m), f, None)),
        ("var_attn_blocksparse_plan", lambda: L.var_attn_blocksparse(C.byref(p), 9, f, f, f, C.byref(mp), f, None)),
        ("var_sparvar_scores", lambda: L.var_sparvar_scores(C.byref(p), 9, 16, 0.8, 0, f, f, f, ws_sv, f, fs, None)),
        ("var_sparvar_scores_fast", lambda: L.var_sparvar_scores_fast(C.byref(p), 9, 16, f, f, f, f, ws_sv, f, None)),
        ("var_selftest_wait_timeout", lambda: L.var_selftest_wait_timeout(1000, fs, None)),
        ("var_device_status", lambda: L.var_device_status(C.byref(out), 1)),
        ("var_check_status", lambda: L.var_check_status(fs, C.byref(out), 1, None)),
    ]


def child():
    """Runs in its own process: {name: [status with no failure, then per failing call]}."""
    sys.path.insert(0, ROOT)
    import visual_autoregressive_next_var_b300 as V
    L = V.lib()
    res = {}
    for name, call in _cases(V):
        L.var_test_mock_cuda(1, 0)
        ok = call()
        n = L.var_test_mock_calls()
        codes = []
        for i in range(1, n + 1):
            L.var_test_mock_cuda(1, i)
            codes.append(call())
        L.var_test_mock_cuda(0, 0)
        res[name] = {"ok": ok, "calls": n, "codes": codes}
    print(json.dumps(res))


@pytest.fixture(scope="module")
def mock_results():
    r = subprocess.run([sys.executable, "-c", "import tests.test_abi_mock_cuda as m; m.child()"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_every_entry_point_succeeds_on_the_mock_device(mock_results):
    for name, r in mock_results.items():
        assert r["ok"] == 0, (name, r["ok"])
        assert r["calls"] >= 1, name


def test_every_cuda_failure_returns_var_err_cuda(mock_results):
    VAR_ERR_CUDA = 3
    for name, r in mock_results.items():
        assert len(r["codes"]) == r["calls"]
        bad = [(i + 1, c) for i, c in enumerate(r["codes"]) if c != VAR_ERR_CUDA]
        assert not bad, f"{name}: failing call -> status {bad}"


def test_launching_entry_points_reach_a_launch(mock_results):
    # each compute entry point makes at least: current device, status-word lookup
    # or attribute, and its launch(es)
    for name in ("var_attn_dense", "var_pivot_select", "var_attn_blocksparse", "var_sparvar_scores"):
        assert mock_results[name]["calls"] >= 3, name
