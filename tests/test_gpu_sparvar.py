"""GPU parity: the SparVAR dynamic sparse pattern -- the decision step's block
scores (certified fp32, fp64 re-score of unsettled blocks), the host selection
and index mapping, and block-sparse attention under the resulting mask --
against the oracle's own pipeline: the mask the GPU path builds must equal,
token for token, the mask the oracle builds from its own fp64 scores.  The
tensor-core scores (no error bound) are checked against the oracle's values
within the fp32 accuracy, for determinism, and for the same masks on these
inputs."""
import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import WORKLOADS, cache_len, make_inputs, randn_bf16
from tests._util import assert_close, check_device_status, csr_to_token_mask

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = (1, 2, 4, 8, 16, 24, 32, 40, 48)      # sinks: the 1, 2, 4 scales at sink_max_side 4


def gpu_scores(p, d, sink, tau, q, k, flags=0):
    U, _ = V.var_sparvar_units(p, d, sink)
    nqb = (int(round(q.shape[2] ** 0.5)) // 8) ** 2
    ws = torch.empty(V.var_sparvar_workspace_bytes(p, d, sink), dtype=torch.uint8, device=DEV)
    sc = torch.empty((nqb, U), dtype=torch.float64, device=DEV)
    rs = torch.full((nqb,), -1, dtype=torch.int32, device=DEV)
    V.var_sparvar_scores(p, d, sink, tau, q, k, ws, sc, rescored=rs, flags=flags)
    torch.cuda.synchronize()
    return sc.cpu().numpy(), rs.cpu().numpy()


def gpu_mask(p, sides, d, ks, sink, A, tau):
    rp, en, sink_len = V.var_sparvar_mask_build(p, d, ks, sink, A, tau)
    return csr_to_token_mask(sides, ks, 8, rp, en, sink_len), (rp, en, sink_len)


def oracle_mask(sides, d, ks, sink, A_ref, tau):
    _, units, ns = oracle.sparvar_units(sides, d, sink)
    return oracle.sparvar_keep_mask(sides, d, ks, units, oracle.sparvar_select(A_ref, ns, tau), sink).astype(bool)


def check_scores(got, rescored, ref):
    """Certified blocks: within the fp32 path's accuracy; re-scored blocks: the
    fp64 definition up to the last bits of exp."""
    assert set(np.unique(rescored)) <= {0, 1}
    for qb in range(got.shape[0]):
        rel = np.abs(got[qb] - ref[qb]) / np.maximum(ref[qb], 1e-300)
        if rescored[qb]:
            assert np.max(rel) < 1e-13, (qb, np.max(rel))
        else:
            assert np.max(np.abs(got[qb] - ref[qb]) - 1e-4 * ref[qb]) <= 1e-12, (qb, np.max(rel))
    assert np.allclose(got.sum(axis=1), 1.0, rtol=0, atol=1e-6)


@pytest.mark.parametrize("d,D", [(5, 128), (5, 64), (8, 64)])   # (8, 64): 92 units
def test_scores_match_oracle(d, D):
    B, H, sink = 2, 2, 4
    L, N = cache_len(SMALL, d), SMALL[d] ** 2
    q = randn_bf16((B, H, N, D), 1101 + d)
    k = randn_bf16((B, H, L + 64, D), 1102 + d)              # spare cache capacity
    p = V.problem(B, H, D, SMALL, kv_capacity=L + 64)
    ref = oracle.sparvar_scores(q, k, SMALL, d, sink)
    got, rs = gpu_scores(p, d, sink, 0.7, q.to(DEV), k.to(DEV))
    check_scores(got, rs, ref)
    forced, rs2 = gpu_scores(p, d, sink, 0.7, q.to(DEV), k.to(DEV), flags=V.VAR_SPARVAR_RESCORE_ALL)
    assert np.all(rs2 == 1)
    check_scores(forced, rs2, ref)
    check_device_status()


@pytest.mark.parametrize("tau", [0.5, 0.9])
def test_dynamic_mask_equals_oracle_and_attention_small(tau):
    B, H, D, sink, d, ks = 2, 2, 128, 4, 5, 7                 # 24 x 24 decides the 40 x 40 step
    L = cache_len(SMALL, ks)
    q_d = randn_bf16((B, H, SMALL[d] ** 2, D), 1111)
    q = randn_bf16((B, H, SMALL[ks] ** 2, D), 1112)
    k = randn_bf16((B, H, L, D), 1113)
    v = randn_bf16((B, H, L, D), 1114)
    p = V.problem(B, H, D, SMALL, kv_capacity=L)             # the cache holds the target step's keys
    kd, vd = k.to(DEV), v.to(DEV)
    A, _ = gpu_scores(p, d, sink, tau, q_d.to(DEV), kd)
    got_mask, (rp, en, sink_len) = gpu_mask(p, SMALL, d, ks, sink, A, tau)
    ref_mask = oracle_mask(SMALL, d, ks, sink, oracle.sparvar_scores(q_d, k, SMALL, d, sink), tau)
    assert ref_mask.mean() < 1.0
    assert np.array_equal(got_mask, ref_mask)
    plan = [torch.as_tensor(x, device=DEV) for x in V.var_block_mask_plan(p, ks, 8, rp, en, sink_len)]
    mask = V.block_mask_struct(8, torch.as_tensor(rp, device=DEV), torch.as_tensor(en, device=DEV), sink_len, plan)
    o = torch.empty_like(q, device=DEV)
    V.var_attn_blocksparse(p, ks, q.to(DEV), kd, vd, mask, o)
    torch.cuda.synchronize()
    assert_close(o, oracle.attention_keep(q, k, v, L, ref_mask), f"dynamic mask tau {tau}")
    check_device_status()


def test_dynamic_mask_1024px_decision_32_target_64():
    w = WORKLOADS["pruned_1024px"]
    d, ks, sink = 9, 12, 16
    inp = make_inputs(w, steps=(d, ks))
    B, H, D = w.batch, w.heads, w.head_dim
    p = V.problem(B, H, D, w.sides, kv_capacity=inp.k.shape[2])
    kd, vd = inp.k.to(DEV), inp.v.to(DEV)
    qd_d = inp.q[d].to(DEV)
    A_ref = oracle.sparvar_scores(inp.q[d], inp.k, w.sides, d, sink)
    for tau in (0.5, 0.8, 0.95):
        A, rs = gpu_scores(p, d, sink, tau, qd_d, kd)
        check_scores(A, rs, A_ref)
        got_mask, (rp, en, sink_len) = gpu_mask(p, w.sides, d, ks, sink, A, tau)
        ref_mask = oracle_mask(w.sides, d, ks, sink, A_ref, tau)
        assert np.array_equal(got_mask, ref_mask), f"tau {tau}: {np.sum(got_mask != ref_mask)} tokens differ"
    # attention of the 64x64 step under the tau = 0.8 mask, on sampled rows
    tau = 0.8
    A, _ = gpu_scores(p, d, sink, tau, qd_d, kd)
    _, (rp, en, sink_len) = gpu_mask(p, w.sides, d, ks, sink, A, tau)
    ref_mask = oracle_mask(w.sides, d, ks, sink, A_ref, tau)
    plan = [torch.as_tensor(x, device=DEV) for x in V.var_block_mask_plan(p, ks, 8, rp, en, sink_len)]
    mask = V.block_mask_struct(8, torch.as_tensor(rp, device=DEV), torch.as_tensor(en, device=DEV), sink_len, plan)
    q = inp.q[ks]
    o = torch.empty_like(q, device=DEV)
    V.var_attn_blocksparse(p, ks, q.to(DEV), kd, vd, mask, o)
    torch.cuda.synchronize()
    L = cache_len(w.sides, ks)
    # one query of every 8x8 block of the 64x64 grid, plus the last
    rows = np.array(sorted({(8 * by + (by + bx) % 8) * 64 + 8 * bx + (3 * by) % 8
                            for by in range(8) for bx in range(8)} | {4095}), dtype=np.int64)
    ref = oracle.attention_keep(q[:, :, torch.as_tensor(rows)].contiguous(), inp.k, inp.v, L, ref_mask[rows])
    assert_close(o[:, :, torch.as_tensor(rows, device=DEV)], ref, "dynamic mask 1024px")
    check_device_status()


def test_exact_ties_go_to_the_lower_unit():
    """q = 0: every key gets probability 1/L exactly, so units of equal size tie
    exactly.  The fp32 bounds cannot order them; the fp64 re-score reproduces
    the ties and the lower unit is taken first, as in the oracle."""
    B, H, D, sink, d, ks = 1, 2, 64, 4, 6, 7                  # 32 x 32 decides 40 x 40
    L = cache_len(SMALL, ks)
    q_d = torch.zeros((B, H, SMALL[d] ** 2, D), dtype=torch.bfloat16)
    k = randn_bf16((B, H, L, D), 1141)
    p = V.problem(B, H, D, SMALL, kv_capacity=L)
    A_ref = oracle.sparvar_scores(q_d, k, SMALL, d, sink)
    for tau in (0.3, 0.61):
        A, rs = gpu_scores(p, d, sink, tau, q_d.to(DEV), k.to(DEV))
        assert np.all(rs == 1)                                # every block has ties at its cut
        assert np.array_equal(A, A_ref)
        got_mask, _ = gpu_mask(p, SMALL, d, ks, sink, A, tau)
        assert np.array_equal(got_mask, oracle_mask(SMALL, d, ks, sink, A_ref, tau))
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
    A, rs = gpu_scores(p, d, sink, tau, q_d.to(DEV), kd)
    A_ref = oracle.sparvar_scores(q_d, k, SMALL, d, sink)
    check_scores(A, rs, A_ref)
    got_mask, (rp, en, sink_len) = gpu_mask(p, SMALL, d, ks, sink, A, tau)
    ref_mask = oracle_mask(SMALL, d, ks, sink, A_ref, tau)
    assert np.array_equal(got_mask, ref_mask)
    mask = V.block_mask_struct(8, torch.as_tensor(rp, device=DEV), torch.as_tensor(en, device=DEV), sink_len)
    o = torch.empty_like(q, device=DEV)
    V.var_attn_blocksparse(p, ks, q.to(DEV), kd, vd, mask, o)   # without a plan: the kernel merges the lists
    torch.cuda.synchronize()
    assert_close(o, oracle.attention_keep(q, k, v, L, ref_mask), "dynamic mask D 64")
    check_device_status()


def test_scores_many_units_head_dim_128():
    sides, sink, d = (1, 2, 4, 8, 16, 24, 32, 40, 48, 64), 4, 9        # 156 units
    B, H, D = 1, 1, 128
    L, N = cache_len(sides, d), sides[d] ** 2
    q = randn_bf16((B, H, N, D), 1131)
    k = randn_bf16((B, H, L, D), 1132)
    p = V.problem(B, H, D, sides)
    U, _ = V.var_sparvar_units(p, d, sink)
    assert U > 128
    A_ref = oracle.sparvar_scores(q, k, sides, d, sink)
    for tau in (0.4, 0.85):
        got, rs = gpu_scores(p, d, sink, tau, q.to(DEV), k.to(DEV))
        check_scores(got, rs, A_ref)
        for ks in (9,):
            got_mask, _ = gpu_mask(p, sides, d, ks, sink, got, tau)
            assert np.array_equal(got_mask, oracle_mask(sides, d, ks, sink, A_ref, tau))
    check_device_status()


def gpu_scores_fast(p, d, sink, q, k):
    """Tensor-core block scores from the decision step's row log2-sum-exp."""
    B, H, N, D = q.shape
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    o = torch.empty_like(q)
    V.var_attn_dense_lse(p, d, q, k, k, o, lse)            # the values do not enter the row statistics
    U, _ = V.var_sparvar_units(p, d, sink)
    ws = torch.empty(V.var_sparvar_workspace_bytes(p, d, sink), dtype=torch.uint8, device=DEV)
    sc = torch.full(((int(round(N ** 0.5)) // 8) ** 2, U), -1.0, dtype=torch.float64, device=DEV)
    V.var_sparvar_scores_fast(p, d, sink, q, k, lse, ws, sc)
    torch.cuda.synchronize()
    return sc.cpu().numpy()


@pytest.mark.parametrize("d,D", [(5, 128), (5, 64), (8, 64)])
def test_fast_scores_close_to_oracle(d, D):
    B, H, sink = 2, 2, 4
    L, N = cache_len(SMALL, d), SMALL[d] ** 2
    q = randn_bf16((B, H, N, D), 1201 + d)
    k = randn_bf16((B, H, L + 64, D), 1202 + d)
    p = V.problem(B, H, D, SMALL, kv_capacity=L + 64)
    ref = oracle.sparvar_scores(q, k, SMALL, d, sink)
    qd, kd = q.to(DEV), k.to(DEV)
    got = gpu_scores_fast(p, d, sink, qd, kd)
    assert np.all(np.isfinite(got))
    assert np.allclose(got, ref, rtol=2e-3, atol=1e-7), np.max(np.abs(got - ref) / np.maximum(ref, 1e-7))
    assert np.allclose(got.sum(axis=1), 1.0, rtol=0, atol=1e-3)
    again = gpu_scores_fast(p, d, sink, qd, kd)
    assert np.array_equal(got, again)                          # fixed summation order: deterministic
    check_device_status()


def test_fast_mask_1024px_decision_32_target_64():
    w = WORKLOADS["pruned_1024px"]
    d, ks, sink = 9, 12, 16
    inp = make_inputs(w, steps=(d, ks))
    B, H, D = w.batch, w.heads, w.head_dim
    p = V.problem(B, H, D, w.sides, kv_capacity=inp.k.shape[2])
    kd = inp.k.to(DEV)
    A_ref = oracle.sparvar_scores(inp.q[d], inp.k, w.sides, d, sink)
    A = gpu_scores_fast(p, d, sink, inp.q[d].to(DEV), kd)
    assert np.allclose(A, A_ref, rtol=2e-3, atol=1e-7)
    for tau in (0.5, 0.8, 0.95):
        got_mask, _ = gpu_mask(p, w.sides, d, ks, sink, A, tau)
        ref_mask = oracle_mask(w.sides, d, ks, sink, A_ref, tau)
        assert np.array_equal(got_mask, ref_mask), f"tau {tau}: {np.sum(got_mask != ref_mask)} tokens differ"
    check_device_status()
