"""GPU parity: the SparVAR dynamic sparse pattern -- decision-step block scores
(dense attention kernel on unit-indicator values + ordered reduction), the host
selection and index mapping, and block-sparse attention under the resulting
mask -- against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import WORKLOADS, cache_len, make_inputs, randn_bf16
from tests._util import assert_close, check_device_status

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = (1, 2, 4, 8, 16, 24, 32, 40, 48)      # sinks: the 1, 2, 4 scales at sink_max_side 4


def gpu_scores(p, d, sink, q, k):
    U, _ = V.var_sparvar_units(p, d, sink)
    nqb = (int(round(q.shape[2] ** 0.5)) // 8) ** 2
    ws = torch.empty(V.var_sparvar_workspace_bytes(p, d), dtype=torch.uint8, device=DEV)
    sc = torch.empty((nqb, U), dtype=torch.float64, device=DEV)
    V.var_sparvar_scores(p, d, sink, q, k, ws, sc)
    torch.cuda.synchronize()
    return sc.cpu().numpy()


def check_scores(got, ref):
    # each per-row unit mass is rounded to bf16 (relative 2^-9) before the average
    assert np.all(np.abs(got - ref) <= 4e-3 * ref + 1e-7), np.max(np.abs(got - ref) / (ref + 1e-12))
    assert np.allclose(got.sum(axis=1), 1.0, rtol=0, atol=4e-3)


@pytest.mark.parametrize("d,D", [(5, 128), (5, 64), (8, 64)])   # (8, 64): 92 units, two passes
def test_scores_match_oracle(d, D):
    B, H, sink = 2, 2, 4
    L, N = cache_len(SMALL, d), SMALL[d] ** 2
    q = randn_bf16((B, H, N, D), 1101 + d)
    k = randn_bf16((B, H, L + 64, D), 1102 + d)              # spare cache capacity
    p = V.problem(B, H, D, SMALL, kv_capacity=L + 64)
    got = gpu_scores(p, d, sink, q.to(DEV), k.to(DEV))
    check_scores(got, oracle.sparvar_scores(q, k, SMALL, d, sink))
    check_device_status()


@pytest.mark.parametrize("tau", [0.5, 0.9])
def test_dynamic_mask_attention_small(tau):
    B, H, D, sink, d, ks = 2, 2, 128, 4, 5, 7                 # 24 x 24 decides the 40 x 40 step
    L = cache_len(SMALL, ks)
    q_d = randn_bf16((B, H, SMALL[d] ** 2, D), 1111)
    q = randn_bf16((B, H, SMALL[ks] ** 2, D), 1112)
    k = randn_bf16((B, H, L, D), 1113)
    v = randn_bf16((B, H, L, D), 1114)
    p = V.problem(B, H, D, SMALL, kv_capacity=L)             # the cache holds the target step's keys
    kd, vd = k.to(DEV), v.to(DEV)
    A = gpu_scores(p, d, sink, q_d.to(DEV), kd)
    rp, en, sink_len = V.var_sparvar_mask_build(p, d, ks, sink, A, tau)
    plan = [torch.as_tensor(x, device=DEV) for x in V.var_block_mask_plan(p, ks, 8, rp, en, sink_len)]
    mask = V.block_mask_struct(8, torch.as_tensor(rp, device=DEV), torch.as_tensor(en, device=DEV), sink_len, plan)
    o = torch.empty_like(q, device=DEV)
    V.var_attn_blocksparse(p, ks, q.to(DEV), kd, vd, mask, o)
    torch.cuda.synchronize()
    _, units, ns = oracle.sparvar_units(SMALL, d, sink)
    keep = oracle.sparvar_keep_mask(SMALL, d, ks, units, oracle.sparvar_select(A, ns, tau), sink)
    assert keep.mean() < 1.0
    assert_close(o, oracle.attention_keep(q, k, v, L, keep), f"dynamic mask tau {tau}")
    check_device_status()


def test_dynamic_mask_1024px_decision_32_target_64():
    w = WORKLOADS["pruned_1024px"]
    d, ks, sink, tau = 9, 12, 16, 0.8
    inp = make_inputs(w, steps=(d, ks))
    B, H, D = w.batch, w.heads, w.head_dim
    p = V.problem(B, H, D, w.sides, kv_capacity=inp.k.shape[2])
    kd, vd = inp.k.to(DEV), inp.v.to(DEV)
    A = gpu_scores(p, d, sink, inp.q[d].to(DEV), kd)
    check_scores(A, oracle.sparvar_scores(inp.q[d], inp.k, w.sides, d, sink))
    rp, en, sink_len = V.var_sparvar_mask_build(p, d, ks, sink, A, tau)
    plan = [torch.as_tensor(x, device=DEV) for x in V.var_block_mask_plan(p, ks, 8, rp, en, sink_len)]
    mask = V.block_mask_struct(8, torch.as_tensor(rp, device=DEV), torch.as_tensor(en, device=DEV), sink_len, plan)
    q = inp.q[ks]
    o = torch.empty_like(q, device=DEV)
    V.var_attn_blocksparse(p, ks, q.to(DEV), kd, vd, mask, o)
    torch.cuda.synchronize()
    L = cache_len(w.sides, ks)
    _, units, ns = oracle.sparvar_units(w.sides, d, sink)
    keep = oracle.sparvar_keep_mask(w.sides, d, ks, units, oracle.sparvar_select(A, ns, tau), sink)
    # one query of every 8x8 block of the 64x64 grid, plus the last
    rows = np.array(sorted({(8 * by + (by + bx) % 8) * 64 + 8 * bx + (3 * by) % 8
                            for by in range(8) for bx in range(8)} | {4095}), dtype=np.int64)
    ref = oracle.attention_keep(q[:, :, torch.as_tensor(rows)].contiguous(), inp.k, inp.v, L, keep[rows])
    assert_close(o[:, :, torch.as_tensor(rows, device=DEV)], ref, "dynamic mask 1024px")
    check_device_status()


def test_dynamic_mask_head_dim_64_single_batch():
    B, H, D, sink, d, ks, tau = 1, 3, 64, 4, 6, 8, 0.7        # 32 x 32 decides the 48 x 48 step
    L = cache_len(SMALL, ks)
    q_d = randn_bf16((B, H, SMALL[d] ** 2, D), 1121)
    q = randn_bf16((B, H, SMALL[ks] ** 2, D), 1122)
    k = randn_bf16((B, H, L, D), 1123)
    v = randn_bf16((B, H, L, D), 1124)
    p = V.problem(B, H, D, SMALL, kv_capacity=L)
    kd, vd = k.to(DEV), v.to(DEV)
    A = gpu_scores(p, d, sink, q_d.to(DEV), kd)
    check_scores(A, oracle.sparvar_scores(q_d, k, SMALL, d, sink))
    rp, en, sink_len = V.var_sparvar_mask_build(p, d, ks, sink, A, tau)
    mask = V.block_mask_struct(8, torch.as_tensor(rp, device=DEV), torch.as_tensor(en, device=DEV), sink_len)
    o = torch.empty_like(q, device=DEV)
    V.var_attn_blocksparse(p, ks, q.to(DEV), kd, vd, mask, o)   # without a plan: the kernel merges the lists
    torch.cuda.synchronize()
    _, units, ns = oracle.sparvar_units(SMALL, d, sink)
    keep = oracle.sparvar_keep_mask(SMALL, d, ks, units, oracle.sparvar_select(A, ns, tau), sink)
    assert_close(o, oracle.attention_keep(q, k, v, L, keep), "dynamic mask D 64")
    check_device_status()


def test_scores_two_passes_head_dim_128():
    sides, sink, d = (1, 2, 4, 8, 16, 24, 32, 40, 48, 64), 4, 9        # 156 units > 128: two passes
    B, H, D = 1, 1, 128
    L, N = cache_len(sides, d), sides[d] ** 2
    q = randn_bf16((B, H, N, D), 1131)
    k = randn_bf16((B, H, L, D), 1132)
    p = V.problem(B, H, D, sides)
    U, _ = V.var_sparvar_units(p, d, sink)
    assert U > 128
    got = gpu_scores(p, d, sink, q.to(DEV), k.to(DEV))
    check_scores(got, oracle.sparvar_scores(q, k, sides, d, sink))
    check_device_status()
