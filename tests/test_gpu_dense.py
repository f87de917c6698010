"""GPU parity: dense cross-scale attention (var_attn_dense) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import WORKLOADS, cache_len, make_inputs, randn_bf16
from tests._util import assert_close, check_device_status, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_dense(p, step, q, k, v):
    o = torch.empty_like(q, device=DEV)
    V.var_attn_dense(p, step, q.to(DEV), k.to(DEV), v.to(DEV), o)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("sides,D,B,H", [
    ((1, 2, 3, 5, 7, 11), 64, 2, 3),          # one partial query tile, partial KV tile
    ((1, 2, 3, 5, 7, 11), 128, 2, 3),
    ((1, 2, 4, 6, 9, 14, 20, 23), 64, 1, 2),  # 529 queries: three pairs, ragged tail
    ((1, 2, 4, 6, 9, 14, 20, 23), 128, 2, 2),
    ((1,), 128, 1, 1),                        # a single token
    ((3, 16), 128, 1, 2),                     # exactly one full query pair, L = 265
])
def test_dense_small_shapes(sides, D, B, H):
    step = len(sides) - 1
    L, N = cache_len(sides, step), sides[step] ** 2
    q = randn_bf16((B, H, N, D), 1)
    k = randn_bf16((B, H, L, D), 2)
    v = randn_bf16((B, H, L, D), 3)
    p = V.problem(B, H, D, sides)
    o = run_dense(p, step, q, k, v)
    assert_close(o, oracle.attention(q, k, v, L), f"dense {sides} D{D}")
    check_device_status()


def test_dense_tiny_workload_full():
    w = WORKLOADS["dense_tiny"]
    inp = make_inputs(w)
    step = w.steps[0]
    L = cache_len(w.sides, step)
    p = V.problem(w.batch, w.heads, w.head_dim, w.sides)
    o = run_dense(p, step, inp.q[step], inp.k, inp.v)
    assert_close(o, oracle.attention(inp.q[step], inp.k, inp.v, L), "dense_tiny")
    check_device_status()


def test_dense_256px_every_step_on_one_cache():
    w = WORKLOADS["dense_256px"]
    inp = make_inputs(w)
    # one cache buffer of the full schedule; step k reads its first L_k rows
    p = V.problem(w.batch, w.heads, w.head_dim, w.sides, kv_capacity=w.n_tokens)
    k, v = inp.k.to(DEV), inp.v.to(DEV)
    for step in w.steps:
        L = cache_len(w.sides, step)
        q = inp.q[step]
        o = torch.empty_like(q, device=DEV)
        V.var_attn_dense(p, step, q.to(DEV), k, v, o)
        torch.cuda.synchronize()
        assert_close(o, oracle.attention(q, inp.k, inp.v, L), f"dense_256px step {step}")
    check_device_status()


def test_dense_1024px_every_row_and_determinism():
    """The 1024px final step (2 x 16 x 4,096 queries against 10,521 keys), every
    output row against the oracle, and two runs bit for bit."""
    w = WORKLOADS["dense_1024px"]
    inp = make_inputs(w)
    step = w.steps[0]
    L = cache_len(w.sides, step)
    q = inp.q[step]
    p = V.problem(w.batch, w.heads, w.head_dim, w.sides)
    qd, kd, vd = q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    o1 = torch.empty_like(qd)
    o2 = torch.empty_like(qd)
    V.var_attn_dense(p, step, qd, kd, vd, o1)
    V.var_attn_dense(p, step, qd, kd, vd, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2), "two runs on the same inputs differ"
    assert_close(o1, oracle.attention(q, inp.k, inp.v, L), "dense_1024px every row")
    check_device_status()


def test_dense_split_tail_ctas_every_row():
    """160 pair slots on 148 SMs: the last 12 slots run as 24 one-tile CTAs whose
    two softmax groups take alternate key tiles and merge at the end; check
    every row of the (b, h) those CTAs cover, and of the first (b, h)."""
    sides, D, B, H = (1, 2, 4, 8, 16, 32), 128, 2, 20
    step = len(sides) - 1
    L, N = cache_len(sides, step), sides[step] ** 2
    q = randn_bf16((B, H, N, D), 11)
    k = randn_bf16((B, H, L, D), 12)
    v = randn_bf16((B, H, L, D), 13)
    p = V.problem(B, H, D, sides)
    o = run_dense(p, step, q, k, v)
    bhs = [0, B * H - 3, B * H - 2, B * H - 1]
    rows = np.concatenate([np.arange(bh * N, (bh + 1) * N) for bh in bhs])
    ref = oracle.attention(q, k, v, L, rows=rows)
    got = o.reshape(-1, D)[torch.as_tensor(rows, device=DEV)]
    assert_close(got, ref, "dense split tail")
    check_device_status()


@pytest.mark.parametrize("sides,D,B,H", [
    ((1, 2, 4, 8, 16, 24), 128, 2, 3),     # CFG pair
    ((1, 2, 3, 5, 7, 11), 64, 4, 2),       # two pairs (cond 0,1 ; uncond 2,3)
])
def test_dense_branch_halved(sides, D, B, H):
    step = len(sides) - 1
    L, N = cache_len(sides, step), sides[step] ** 2
    q = randn_bf16((B, H, N, D), 31)
    k = randn_bf16((B, H, L, D), 32)
    v = randn_bf16((B, H, L, D), 33)
    p = V.problem(B, H, D, sides)
    o = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    V.var_attn_dense_halved(p, step, q.to(DEV), k.to(DEV), v.to(DEV), o)
    torch.cuda.synchronize()
    assert torch.equal(o[B // 2:], o[: B // 2])                  # the repeat is exact
    assert_close(o, oracle.branch_halved_attention(q, k, v, L), f"halved {sides}")
    check_device_status()


def test_dense_invariants_on_gpu():
    # identical value rows -> that row; all-equal keys -> mean of values
    B, H, D, sides = 1, 2, 128, (1, 2, 4, 8, 16)
    step, L, N = 4, 341, 256
    q = randn_bf16((B, H, N, D), 7)
    k = randn_bf16((B, H, L, D), 8)
    row = randn_bf16((D,), 9)
    v = row.expand(B, H, L, D).contiguous()
    p = V.problem(B, H, D, sides)
    o = run_dense(p, step, q, k, v)
    assert_close(o, np.broadcast_to(row.double().numpy(), (B, H, N, D)), "identical V", 1e-2, 1e-3)
    kz = torch.zeros_like(k)
    v2 = randn_bf16((B, H, L, D), 10)
    o2 = run_dense(p, step, q, kz, v2)
    mean = v2.double().mean(dim=2, keepdim=True).expand(B, H, N, D).numpy()
    assert_close(o2, mean, "uniform keys")
    check_device_status()
