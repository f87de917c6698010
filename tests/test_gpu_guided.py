"""GPU parity: attention-guided pivot selection (ARVAR attention retrospect) --
row statistics of the source step, the saliency kernel, and the upsampled
Top-K -- against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import WORKLOADS, cache_len, make_inputs, randn_bf16
from tests._util import check_device_status

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _source(sides, src, B, H, D, seed):
    L = cache_len(sides, src)
    N = sides[src] ** 2
    q = randn_bf16((B, H, N, D), seed)
    k = randn_bf16((B, H, L, D), seed + 1)
    v = randn_bf16((B, H, L, D), seed + 2)
    return q, k, v, L, N


@pytest.mark.parametrize("sides,src,D,B,H", [
    ((1, 2, 4, 6, 9, 14), 5, 128, 2, 2),        # 196 source tokens: a partial key and query tile
    ((1, 2, 3, 5, 8, 12), 5, 64, 1, 3),
    ((2, 4, 8, 16), 3, 128, 2, 1),              # 256: exactly two tiles
])
def test_lse_and_saliency_small(sides, src, D, B, H):
    q, k, v, L, N = _source(sides, src, B, H, D, 401)
    p = V.problem(B, H, D, sides)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    V.var_attn_dense_lse(p, src, qd, kd, vd, o, lse)
    o_plain = torch.empty_like(qd)
    V.var_attn_dense(p, src, qd, kd, vd, o_plain)
    sal = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    V.var_attn_saliency(p, src, qd, kd, lse, sal)
    torch.cuda.synchronize()
    assert torch.equal(o, o_plain)                       # the statistics change nothing else
    ref_lse = oracle.attention_lse(q, k, L)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) < 2e-3
    ref = oracle.saliency(q, k, L)
    got = sal.cpu().double().numpy()
    assert np.max(np.abs(got - ref) / np.maximum(ref, 1e-3)) < 2e-3
    check_device_status()


def test_guided_pivot_1024px_retrospect():
    """Source step 32x32 (T - 3) guiding the 64x64 step, keep 20 %."""
    w = WORKLOADS["pruned_1024px"]
    src, step = 9, 12
    inp = make_inputs(w, steps=(src,))
    q = inp.q[src]
    B, H, N, D = q.shape
    L = cache_len(w.sides, src)
    p = V.problem(B, H, D, w.sides, kv_capacity=inp.k.shape[2])     # the whole schedule's cache
    qd, kd, vd = q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    sal = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    V.var_attn_dense_lse(p, src, qd, kd, vd, o, lse)
    V.var_attn_saliency(p, src, qd, kd, lse, sal)
    s = w.sides[step]
    K = V.var_keep_count(s * s, 1, 5)
    ws = torch.empty(V.var_guided_pivot_workspace_bytes(p, step), dtype=torch.uint8, device=DEV)
    idx = torch.empty((B, K), dtype=torch.int32, device=DEV)
    vals = torch.empty((B, s * s), dtype=torch.float32, device=DEV)
    V.var_guided_pivot_select(p, step, src, sal, K, idx, ws, vals)
    torch.cuda.synchronize()
    got_idx, got_v = idx.cpu().numpy(), vals.cpu().numpy()
    # the selection is exact on the kernel's own fp32 values (a plain sort here)
    for b in range(B):
        order = np.lexsort((np.arange(s * s), -got_v[b].astype(np.float64)))
        assert np.array_equal(got_idx[b], np.sort(order[:K]))
    # against the fp64 pipeline: values to 2e-3, and only near-ties at the K-th
    # value may differ (the fast path ranks fp32 values; the exact path below
    # reproduces the fp64 ranking)
    sal_np = sal.cpu().double().numpy()
    ref_sal = oracle.saliency(q, inp.k, L)
    assert np.max(np.abs(sal_np - ref_sal) / np.maximum(ref_sal, 1e-3)) < 2e-3
    ref_idx, ref_v = oracle.guided_pivot(ref_sal, s, K)
    assert np.max(np.abs(got_v - ref_v) / np.abs(ref_v)) < 2e-3
    for b in range(B):
        vk = np.sort(ref_v[b])[::-1][K - 1]
        delta = 2e-3 * abs(vk)
        chosen = set(got_idx[b].tolist())
        assert len(chosen) == K
        assert all(ref_v[b, i] >= vk - delta for i in chosen)
        assert all(i in chosen for i in np.nonzero(ref_v[b] > vk + delta)[0])
        assert len(chosen ^ set(ref_idx[b].tolist())) <= 0.02 * K
    check_device_status()


def test_guided_pivot_ties_keep_lower_index():
    # a constant saliency map: every interpolated value ties, so the first K tokens win
    B, H, sides = 2, 4, (1, 4, 8)              # 4 heads x 16 tokens: the mean is exact
    p = V.problem(B, H, 64, sides)
    sal = torch.full((B, H, 16), 0.25, dtype=torch.float32, device=DEV)
    ws = torch.empty(V.var_guided_pivot_workspace_bytes(p, 2), dtype=torch.uint8, device=DEV)
    for K in (1, 13, 64):
        idx = torch.empty((B, K), dtype=torch.int32, device=DEV)
        V.var_guided_pivot_select(p, 2, 1, sal, K, idx, ws)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(K), (B, 1)))
    check_device_status()


def _exact(p, step, src, q_src, k, K, B, N):
    ws = torch.empty(V.var_guided_pivot_exact_workspace_bytes(p, step, src), dtype=torch.uint8, device=DEV)
    idx = torch.full((B, max(K, 1)), -1, dtype=torch.int32, device=DEV)
    vals = torch.empty((B, N), dtype=torch.float64, device=DEV)
    V.var_guided_pivot_select_exact(p, step, src, q_src, k, K, idx, ws, vals)
    torch.cuda.synchronize()
    return idx[:, :K].cpu().numpy(), vals.cpu().numpy()


def test_guided_pivot_exact_1024px_matches_oracle_bit_for_bit():
    """Source step 32x32 guiding the 64x64 step, keep 20 %: the fp64 path's kept
    indices equal the oracle's, and its values equal the oracle's fp64 values
    up to the last bits of exp."""
    w = WORKLOADS["pruned_1024px"]
    src, step = 9, 12
    inp = make_inputs(w, steps=(src,))
    q = inp.q[src]
    B, H, N, D = q.shape
    L = cache_len(w.sides, src)
    p = V.problem(B, H, D, w.sides, kv_capacity=inp.k.shape[2])
    s = w.sides[step]
    K = V.var_keep_count(s * s, 1, 5)
    got_idx, got_v = _exact(p, step, src, q.to(DEV), inp.k.to(DEV), K, B, s * s)
    ref_idx, ref_v = oracle.guided_pivot(oracle.saliency(q, inp.k, L), s, K)
    assert np.max(np.abs(got_v - ref_v) / np.abs(ref_v)) < 1e-13
    assert np.array_equal(got_idx, ref_idx)
    check_device_status()


@pytest.mark.parametrize("sides,src,step,D,B,H,num,den", [
    ((1, 2, 4, 6, 9, 14, 20), 5, 6, 64, 1, 3, 2, 5),        # 14x14 guides 20x20, ragged
    ((1, 2, 4, 8, 16, 24), 4, 5, 128, 2, 2, 1, 3),          # 16x16 guides 24x24
    ((1, 2, 4, 8, 16, 24), 3, 5, 128, 2, 2, 1, 1),          # keep everything
])
def test_guided_pivot_exact_small(sides, src, step, D, B, H, num, den):
    L = cache_len(sides, src)
    N_src = sides[src] ** 2
    q = randn_bf16((B, H, N_src, D), 421 + src)
    k = randn_bf16((B, H, cache_len(sides, step), D), 422 + src)
    p = V.problem(B, H, D, sides, kv_capacity=k.shape[2])
    s = sides[step]
    K = V.var_keep_count(s * s, num, den)
    got_idx, got_v = _exact(p, step, src, q.to(DEV), k.to(DEV), K, B, s * s)
    ref_idx, ref_v = oracle.guided_pivot(oracle.saliency(q, k, L), s, K)
    assert np.max(np.abs(got_v - ref_v) / np.abs(ref_v)) < 1e-13
    assert np.array_equal(got_idx, ref_idx)
    check_device_status()


def test_guided_pivot_exact_ties_keep_lower_index():
    # q = 0: every key receives 1/L' from every query, so the source map is
    # constant and the interpolated values tie wherever the bilinear weights
    # round alike; ties go to the lower index on both sides
    sides, src, step, B, H, D = (1, 2, 4, 8), 2, 3, 2, 2, 64
    L = cache_len(sides, src)
    q = torch.zeros((B, H, 16, D), dtype=torch.bfloat16)
    k = randn_bf16((B, H, cache_len(sides, step), D), 431)
    p = V.problem(B, H, D, sides, kv_capacity=k.shape[2])
    for K in (0, 1, 13, 64):
        got_idx, got_v = _exact(p, step, src, q.to(DEV), k.to(DEV), K, B, 64)
        ref_idx, ref_v = oracle.guided_pivot(oracle.saliency(q, k, L), 8, K)
        assert np.array_equal(got_v, ref_v)
        assert np.array_equal(got_idx, ref_idx)
        assert len(np.unique(ref_v)) < ref_v.size // 4          # the case has many exact ties
    check_device_status()
