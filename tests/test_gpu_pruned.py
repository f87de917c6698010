"""GPU parity: cached token pruning -- pivot selection (bit-exact indices),
pruned attention, restore + scatter, and the chained 1024px pruned steps."""
import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import WORKLOADS, cache_len, make_inputs, randn_bf16
from tests._util import assert_close, check_device_status, sample_rows, to_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_pivot(p, step, x, keep_k, want_scores=False):
    B, N, Cc = x.shape
    ws = torch.empty(V.var_pivot_workspace_bytes(p, step, Cc), dtype=torch.uint8, device=DEV)
    idx = torch.full((B, max(keep_k, 1)), -1, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, N), dtype=torch.float32, device=DEV) if want_scores else None
    V.var_pivot_select(p, step, x.to(DEV), keep_k, idx, ws, sc)
    torch.cuda.synchronize()
    return idx[:, :keep_k].cpu().numpy(), (sc.cpu().numpy() if want_scores else None)


# ---------------------------------------------------------------- pivot selection

@pytest.mark.parametrize("step,num,den", [(11, 2, 5), (12, 1, 5)])
def test_pivot_workload_bit_exact(step, num, den):
    w = WORKLOADS["pruned_1024px"]
    inp = make_inputs(w)
    x = inp.x[step]
    B, N, Cc = x.shape
    K = V.var_keep_count(N, num, den)
    p = V.problem(w.batch, w.heads, w.head_dim, w.sides)
    got, sc = gpu_pivot(p, step, x, K, want_scores=True)
    ref, ref_sc = oracle.pivot_select(x, K)
    assert np.array_equal(got, ref)
    assert np.max(np.abs(sc - ref_sc) / ref_sc) < 1e-4
    check_device_status()


@pytest.mark.parametrize("N,Cc,K,seed", [(64, 32, 10, 0), (100, 64, 99, 1), (169, 256, 1, 2),
                                          (256, 2048, 128, 3), (400, 96, 200, 4), (1024, 512, 1024, 5)])
def test_pivot_random_shapes(N, Cc, K, seed):
    s = int(round(N ** 0.5))
    p = V.problem(2, 1, 64, (1, s))
    x = randn_bf16((2, N, Cc), 50 + seed)
    got, _ = gpu_pivot(p, 1, x, K)
    ref, _ = oracle.pivot_select(x, K)
    assert np.array_equal(got, ref)
    check_device_status()


def test_pivot_ties_and_degenerate_grids():
    p = V.problem(2, 1, 64, (1, 16))
    const = torch.full((2, 256, 64), 0.375).to(torch.bfloat16)
    got, _ = gpu_pivot(p, 1, const, 37)
    assert np.array_equal(got, np.tile(np.arange(37), (2, 1)))          # all tied: lowest indices
    x = randn_bf16((2, 256, 64), 60)
    x[:, 200] = 4.0
    x[:, 17] = 4.0                                                      # identical extreme rows
    got, _ = gpu_pivot(p, 1, x, 1)
    assert np.array_equal(got, [[17], [17]])
    got2, _ = gpu_pivot(p, 1, x, 2)
    assert np.array_equal(got2, [[17, 200], [17, 200]])
    dup = randn_bf16((2, 16, 64), 61).repeat(1, 16, 1)                  # 16 copies of 16 rows
    got3, _ = gpu_pivot(p, 1, dup, 40)
    ref3, _ = oracle.pivot_select(dup, 40)
    assert np.array_equal(got3, ref3)
    got4, _ = gpu_pivot(p, 1, x, 256)
    assert np.array_equal(got4, np.tile(np.arange(256), (2, 1)))
    got0, _ = gpu_pivot(p, 1, x, 0)
    assert got0.shape == (2, 0)
    check_device_status()


def test_pivot_outliers_and_tiny_values():
    """Elements at or beyond the fast summation window (|x| >= 512) and far below
    it (|x| < 2^-29, zeros) must still give the oracle's exact ranking."""
    p = V.problem(2, 1, 64, (1, 24))
    x = randn_bf16((2, 576, 160), 62).float()
    x[0, 5, 3] = 1000.0
    x[0, 300, 100] = -700.0
    x[1, 17, 0] = 512.0
    x[1, 200, :] = 3e-10
    x[1, 201, 7] = 0.0
    x[0, 400:410, 40] = 1e-12
    x = x.to(torch.bfloat16)
    for K in (1, 57, 300):
        got, sc = gpu_pivot(p, 1, x, K, want_scores=True)
        ref, ref_sc = oracle.pivot_select(x, K)
        assert np.array_equal(got, ref), K
        assert np.max(np.abs(sc - ref_sc) / np.maximum(ref_sc, 1.0)) < 1e-4
    check_device_status()


def test_pivot_single_token_and_large_grid():
    p = V.problem(1, 1, 64, (1, 2))
    x1 = randn_bf16((1, 1, 32), 63)
    got, _ = gpu_pivot(p, 0, x1, 1)
    assert np.array_equal(got, [[0]])
    sides = (1, 2, 4, 8, 16, 32, 64, 128)
    q = V.problem(1, 1, 64, sides)
    x = randn_bf16((1, 16384, 256), 64)
    got, _ = gpu_pivot(q, 7, x, 3277)
    ref, _ = oracle.pivot_select(x, 3277)
    assert np.array_equal(got, ref)
    check_device_status()


# ---------------------------------------------------------------- fused pruned step

@pytest.mark.parametrize("order", ["attn_then_fill", "fill_then_attn", "one_call", "whole_step"])
def test_fused_pruned_step_equals_chain(order):
    """var_attn_pruned_scatter + var_restore_fill (in either order),
    var_pruned_in_place (the fill started beside the attention) and
    var_pruned_step (pivots, attention and fill chained in one call) write the
    same output as var_attn_pruned + var_restore_scatter, bit for bit."""
    w = WORKLOADS["pruned_1024px"]
    inp = make_inputs(w, steps=(12,))
    step = 12
    q = inp.q[step]
    B, H, N, D = q.shape
    L = cache_len(w.sides, step)
    K = V.var_keep_count(N, 1, 5)
    p = V.problem(B, H, D, w.sides)
    qd, kd, vd = q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    x = inp.x[step].to(DEV)
    ws = torch.empty(V.var_pivot_workspace_bytes(p, step, x.shape[2]), dtype=torch.uint8, device=DEV)
    idx = torch.empty((B, K), dtype=torch.int32, device=DEV)
    V.var_pivot_select(p, step, x, K, idx, ws)
    prev_c = randn_bf16((B, H, 48 * 48, D), 77)
    prev = prev_c.to(DEV)
    oc = torch.empty((B, H, K, D), dtype=torch.bfloat16, device=DEV)
    chain = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=DEV)
    V.var_attn_pruned(p, step, qd, kd, vd, idx, K, oc)
    V.var_restore_scatter(p, step, prev, oc, idx, K, chain)
    fused = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    if order == "fill_then_attn":
        V.var_restore_fill(p, step, prev, idx, K, fused)
        V.var_attn_pruned_scatter(p, step, qd, kd, vd, idx, K, fused)
    elif order == "attn_then_fill":
        V.var_attn_pruned_scatter(p, step, qd, kd, vd, idx, K, fused)
        V.var_restore_fill(p, step, prev, idx, K, fused)
    elif order == "one_call":
        V.var_pruned_in_place(p, step, qd, kd, vd, prev, idx, K, fused)
    else:
        idx2 = torch.full_like(idx, -1)
        V.var_pruned_step(p, step, x, K, qd, kd, vd, prev, idx2, fused, ws)
        torch.cuda.synchronize()
        assert torch.equal(idx2, idx)
    torch.cuda.synchronize()
    assert torch.equal(fused, chain)
    # against the oracle's own step: its pivots (equal to the GPU's, bit for
    # bit), its pruned rows stored as bf16, and its restore of the synthetic prev
    ref_idx, _ = oracle.pivot_select(inp.x[step], K)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    qrows = (np.arange(B * H)[:, None] * N + ref_idx[np.arange(B * H) // H]).reshape(-1)
    oc_ref = to_bf16(oracle.attention(q, inp.k, inp.v, L, rows=qrows)).reshape(B, H, K, D)
    ref = oracle.restore_scatter(prev_c, oc_ref, ref_idx, 64)
    assert_close(fused, ref, "fused step, every row")
    check_device_status()


def test_fused_pruned_step_head_dim_64_ragged():
    """head_dim 64, a 23x23 grid (ragged tiles), random kept set; fused == chain."""
    sides, D, B, H = (1, 2, 4, 6, 9, 14, 20, 23), 64, 2, 3
    step = len(sides) - 1
    L, N = cache_len(sides, step), sides[step] ** 2
    qc, kc, vc = randn_bf16((B, H, N, D), 91), randn_bf16((B, H, L, D), 92), randn_bf16((B, H, L, D), 93)
    prev_c = randn_bf16((B, H, 20 * 20, D), 94)
    q, k, v, prev = qc.to(DEV), kc.to(DEV), vc.to(DEV), prev_c.to(DEV)
    K = 101
    g = torch.Generator().manual_seed(95)
    idx_c = torch.stack([torch.sort(torch.randperm(N, generator=g)[:K])[0] for _ in range(B)]).to(torch.int32)
    idx = idx_c.to(DEV)
    p = V.problem(B, H, D, sides)
    oc = torch.empty((B, H, K, D), dtype=torch.bfloat16, device=DEV)
    chain = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=DEV)
    V.var_attn_pruned(p, step, q, k, v, idx, K, oc)
    V.var_restore_scatter(p, step, prev, oc, idx, K, chain)
    fused = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    V.var_attn_pruned_scatter(p, step, q, k, v, idx, K, fused)
    V.var_restore_fill(p, step, prev, idx, K, fused)
    one = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    V.var_pruned_in_place(p, step, q, k, v, prev, idx, K, one)
    torch.cuda.synchronize()
    assert torch.equal(fused, chain)
    assert torch.equal(one, chain)
    # keep_k = 0: the upsampled grid alone, equal to a restore with nothing kept
    empty = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    V.var_pruned_in_place(p, step, None, None, None, prev, None, 0, empty)
    up = torch.empty_like(chain)
    V.var_restore_scatter(p, step, prev, oc, idx, 0, up)
    torch.cuda.synchronize()
    assert torch.equal(empty, up)
    # every row against the oracle: kept rows are attention rows, the rest the upsample
    ic = idx_c.numpy()
    qrows = (np.arange(B * H)[:, None] * N + ic[np.arange(B * H) // H]).reshape(-1)
    oc_ref = oracle.attention(qc, kc, vc, L, rows=qrows)
    assert_close(oc.reshape(-1, D), oc_ref, "pruned rows, head_dim 64")
    ref = oracle.restore_scatter(prev_c, to_bf16(oc_ref).reshape(B, H, K, D), ic, sides[step])
    assert_close(fused, ref, "fused step head_dim 64, every row")
    check_device_status()


# ---------------------------------------------------------------- pruned attention

@pytest.mark.parametrize("K", [1, 130, 819, 4096])
def test_pruned_attention_sampled(K):
    w = WORKLOADS["pruned_1024px"]
    inp = make_inputs(w, steps=(12,))
    step = 12
    q = inp.q[step]
    B, H, N, D = q.shape
    L = cache_len(w.sides, step)
    g = torch.Generator().manual_seed(K)
    idx = torch.stack([torch.sort(torch.randperm(N, generator=g)[:K])[0] for _ in range(B)]).to(torch.int32)
    p = V.problem(B, H, D, w.sides)
    oc = torch.empty((B, H, K, D), dtype=torch.bfloat16, device=DEV)
    V.var_attn_pruned(p, step, q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), idx.to(DEV), K, oc)
    torch.cuda.synchronize()
    # compact row (b, h, j) is query row (b, h, idx[b, j])
    crow = sample_rows(B, H, K, 96, seed=K)
    bh, j = crow // K, crow % K
    b = bh // H
    qrows = bh * N + idx.numpy()[b, j]
    ref = oracle.attention(q, inp.k, inp.v, L, rows=qrows)
    got = oc.reshape(-1, D)[torch.as_tensor(crow, device=DEV)]
    assert_close(got, ref, f"pruned K={K}")
    check_device_status()


def test_pruned_keep_all_equals_dense():
    sides, D, B, H = (1, 2, 4, 6, 9, 14, 20), 128, 2, 2
    step, N, L = 6, 400, cache_len(sides, 6)
    q = randn_bf16((B, H, N, D), 70)
    k = randn_bf16((B, H, L, D), 71)
    v = randn_bf16((B, H, L, D), 72)
    p = V.problem(B, H, D, sides)
    idx = torch.arange(N, dtype=torch.int32).repeat(B, 1).to(DEV)
    oc = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=DEV)
    od = torch.empty_like(oc)
    V.var_attn_pruned(p, step, q.to(DEV), k.to(DEV), v.to(DEV), idx, N, oc)
    V.var_attn_dense(p, step, q.to(DEV), k.to(DEV), v.to(DEV), od)
    torch.cuda.synchronize()
    assert torch.equal(oc, od)
    check_device_status()


@pytest.mark.parametrize("keep", [(1, 5), (1, 529), (1, 1)])
def test_pruned_step_one_call_head_dim_64_ragged(keep):
    """var_pruned_step at head_dim 64 on a 23x23 grid (keep 1/5, a single
    token, every token): its indices equal the oracle's pivots bit for bit and
    its output equals var_pivot_select + var_attn_pruned + var_restore_scatter
    bit for bit."""
    sides, D, B, H, C_ = (1, 2, 4, 6, 9, 14, 20, 23), 64, 2, 3, 96
    step = len(sides) - 1
    L, N = cache_len(sides, step), sides[step] ** 2
    qc, kc, vc = randn_bf16((B, H, N, D), 191), randn_bf16((B, H, L, D), 192), randn_bf16((B, H, L, D), 193)
    prev_c = randn_bf16((B, H, 20 * 20, D), 194)
    x_c = randn_bf16((B, N, C_), 195)
    q, k, v, prev, x = qc.to(DEV), kc.to(DEV), vc.to(DEV), prev_c.to(DEV), x_c.to(DEV)
    K = V.var_keep_count(N, *keep)
    p = V.problem(B, H, D, sides)
    ws = torch.empty(V.var_pivot_workspace_bytes(p, step, C_), dtype=torch.uint8, device=DEV)
    idx = torch.empty((B, K), dtype=torch.int32, device=DEV)
    V.var_pivot_select(p, step, x, K, idx, ws)
    oc = torch.empty((B, H, K, D), dtype=torch.bfloat16, device=DEV)
    chain = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=DEV)
    V.var_attn_pruned(p, step, q, k, v, idx, K, oc)
    V.var_restore_scatter(p, step, prev, oc, idx, K, chain)
    one = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    idx1 = torch.full_like(idx, -1)
    V.var_pruned_step(p, step, x, K, q, k, v, prev, idx1, one, ws)
    torch.cuda.synchronize()
    assert np.array_equal(idx1.cpu().numpy(), oracle.pivot_select(x_c, K)[0])
    assert torch.equal(idx1, idx)
    assert torch.equal(one, chain)
    # nothing kept: the upsampled grid alone
    up = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    V.var_pruned_step(p, step, x, 0, None, None, None, prev, None, up, None)
    ref = torch.empty_like(chain)
    V.var_restore_scatter(p, step, prev, None, None, 0, ref)
    torch.cuda.synchronize()
    assert torch.equal(up, ref)
    check_device_status()


# ---------------------------------------------------------------- restore + scatter

@pytest.mark.parametrize("sp,s,K,D", [(48, 64, 819, 128), (40, 48, 921, 128), (13, 16, 0, 64),
                                      (13, 16, 256, 64), (5, 6, 7, 128), (64, 64, 100, 128),
                                      (96, 128, 6554, 64),      # index list longer than 4096: row searches
                                      (64, 80, 6400, 64),       # every token kept, searched rows full
                                      (24, 32, 1024, 128),      # every token kept, whole-list reads
                                      (1, 2, 1, 128),           # the first restore: one source token
                                      (8, 5, 3, 128)])          # a coarser output grid (ratio 1.6)
def test_restore_scatter(sp, s, K, D):
    B, H = 2, 3
    sides = (1, sp, s) if sp != s else (1, s, s)
    p = V.problem(B, H, D, sides)
    prev = randn_bf16((B, H, sp * sp, D), 80 + s)
    oc = randn_bf16((B, H, max(K, 1), D), 81 + s)[:, :, :K].contiguous()
    g = torch.Generator().manual_seed(K + s)
    idx = torch.stack([torch.sort(torch.randperm(s * s, generator=g)[:K])[0] for _ in range(B)]).to(torch.int32)
    out = torch.empty((B, H, s * s, D), dtype=torch.bfloat16, device=DEV)
    V.var_restore_scatter(p, 2, prev.to(DEV), oc.to(DEV) if K else None, idx.to(DEV) if K else None, K, out)
    torch.cuda.synchronize()
    ref = oracle.restore_scatter(prev, oc, idx.numpy(), s)
    assert_close(out, ref, f"restore {sp}->{s} K={K}")
    outc = out.cpu()
    for b in range(B):
        assert torch.equal(outc[b][:, idx[b].long()], oc[b])          # kept rows: exact copies
    check_device_status()


# ---------------------------------------------------------------- the chained pruned steps

def test_pruned_chain_1024px():
    """40x40 dense -> 48x48 pruned (r=0.4) + restore -> 64x64 pruned (r=0.2) + restore.
    The oracle runs the same chain on its own results, each stage's output
    stored as bf16 as the GPU stores it; the pivot indices are compared bit for
    bit at both steps and every output row of each stage against the oracle's."""
    w = WORKLOADS["pruned_1024px"]
    inp = make_inputs(w)
    B, H, D = w.batch, w.heads, w.head_dim
    p = V.problem(B, H, D, w.sides, kv_capacity=w.n_tokens)   # one cache for every step
    k, v = inp.k.to(DEV), inp.v.to(DEV)
    # step 10: dense 40x40
    q10 = inp.q[10]
    o10 = torch.empty_like(q10, device=DEV)
    V.var_attn_dense(p, 10, q10.to(DEV), k, v, o10)
    torch.cuda.synchronize()
    ref10 = oracle.attention(q10, inp.k, inp.v, cache_len(w.sides, 10))
    assert_close(o10, ref10, "chain step 10")
    prev, prev_ref = o10, to_bf16(ref10)
    for step, num, den in ((11, 2, 5), (12, 1, 5)):
        x = inp.x[step]
        N = x.shape[1]
        L = cache_len(w.sides, step)
        K = V.var_keep_count(N, num, den)
        idx_g, _ = gpu_pivot(p, step, x, K)
        idx_ref, _ = oracle.pivot_select(x, K)
        assert np.array_equal(idx_g, idx_ref), f"pivot indices differ at step {step}"
        idx_d = torch.as_tensor(idx_g, device=DEV)
        oc = torch.empty((B, H, K, D), dtype=torch.bfloat16, device=DEV)
        V.var_attn_pruned(p, step, inp.q[step].to(DEV), k, v, idx_d, K, oc)
        out = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=DEV)
        V.var_restore_scatter(p, step, prev, oc, idx_d, K, out)
        torch.cuda.synchronize()
        qrows = (np.arange(B * H)[:, None] * N + idx_ref[np.arange(B * H) // H]).reshape(-1)
        oc_ref = oracle.attention(inp.q[step], inp.k, inp.v, L, rows=qrows)
        assert_close(oc.reshape(-1, D), oc_ref, f"chain pruned rows {step}")
        ref = oracle.restore_scatter(prev_ref, to_bf16(oc_ref).reshape(B, H, K, D), idx_ref, w.sides[step])
        assert_close(out, ref, f"chain restore step {step}, every row")
        prev, prev_ref = out, to_bf16(ref)
    check_device_status()
