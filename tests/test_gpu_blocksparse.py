"""GPU parity: block-sparse cross-scale attention (var_attn_blocksparse) against
the oracle's token-level mask rule."""
import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import WORKLOADS, cache_len, make_inputs, randn_bf16
from tests._util import assert_close, check_device_status

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_sparse(p, step, q, k, v, radius, sink_max, entries_fix=None):
    rp, ent, sink = V.var_block_mask_build(p, step, 8, radius, sink_max)
    if entries_fix is not None:
        ent = entries_fix(rp, ent.copy())
    m = V.block_mask_struct(8, torch.as_tensor(rp, device=DEV), torch.as_tensor(ent, device=DEV), sink)
    o = torch.empty_like(q, device=DEV)
    V.var_attn_blocksparse(p, step, q.to(DEV), k.to(DEV), v.to(DEV), m, o)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("sides,D,B,H,radius,sink", [
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32), 128, 2, 2, 1, 8),   # partial key blocks at 12 and 20
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32), 64, 1, 3, 2, 16),
    ((1, 2, 4, 8, 16, 24, 40), 128, 1, 2, 2, 4),             # 5x5 query blocks: half-empty squares,
                                                             # sink of 21 tokens (partial chunk)
    ((1, 2, 4, 6, 8, 12, 16), 128, 2, 2, 0, 4),              # the smoke-test shape
    ((2, 3, 8, 16, 48), 128, 1, 1, 3, 3),                    # sink 13 tokens, three local scales
])
def test_blocksparse_small_full(sides, D, B, H, radius, sink):
    step = len(sides) - 1
    L, N = cache_len(sides, step), sides[step] ** 2
    q = randn_bf16((B, H, N, D), 11)
    k = randn_bf16((B, H, L, D), 12)
    v = randn_bf16((B, H, L, D), 13)
    p = V.problem(B, H, D, sides)
    o = run_sparse(p, step, q, k, v, radius, sink)
    ref = oracle.attention(q, k, v, L, mask=oracle.mask_spec(sides, step, 8, radius, sink))
    assert_close(o, ref, f"blocksparse {sides} r{radius} sink{sink} D{D}")
    check_device_status()


@pytest.mark.parametrize("sides,D,B,H,radius,sink", [
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32), 128, 2, 2, 1, 8),
    ((1, 2, 4, 8, 16, 24, 40), 128, 1, 2, 2, 4),             # partial squares at the edge
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32, 40, 48, 64), 64, 1, 2, 2, 16),
])
def test_blocksparse_plan_equals_in_kernel_merge(sides, D, B, H, radius, sink):
    """The host-built plan (merged unit lists, heaviest squares first) gives the
    same output, bit for bit, as the kernel's own per-CTA merge."""
    step = len(sides) - 1
    L, N = cache_len(sides, step), sides[step] ** 2
    q = randn_bf16((B, H, N, D), 41)
    k = randn_bf16((B, H, L, D), 42)
    v = randn_bf16((B, H, L, D), 43)
    p = V.problem(B, H, D, sides)
    rp, ent, sink_len = V.var_block_mask_build(p, step, 8, radius, sink)
    plan = [torch.as_tensor(a, device=DEV) for a in V.var_block_mask_plan(p, step, 8, rp, ent, sink_len)]
    rp_d, ent_d = torch.as_tensor(rp, device=DEV), torch.as_tensor(ent, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1 = torch.empty_like(qd)
    o2 = torch.empty_like(qd)
    V.var_attn_blocksparse(p, step, qd, kd, vd, V.block_mask_struct(8, rp_d, ent_d, sink_len), o1)
    V.var_attn_blocksparse(p, step, qd, kd, vd, V.block_mask_struct(8, rp_d, ent_d, sink_len, plan), o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    ref = oracle.attention(q, k, v, L, mask=oracle.mask_spec(sides, step, 8, radius, sink))
    assert_close(o2, ref, f"planned blocksparse {sides}")
    check_device_status()


def test_blocksparse_covering_window_equals_dense():
    sides, D, B, H = (1, 2, 4, 8, 16, 32), 128, 2, 2
    step, L, N = 5, cache_len(sides, 5), 1024
    q = randn_bf16((B, H, N, D), 21)
    k = randn_bf16((B, H, L, D), 22)
    v = randn_bf16((B, H, L, D), 23)
    p = V.problem(B, H, D, sides)
    o = run_sparse(p, step, q, k, v, 100, 4)
    od = torch.empty_like(o)
    V.var_attn_dense(p, step, q.to(DEV), k.to(DEV), v.to(DEV), od)
    torch.cuda.synchronize()
    ref = oracle.attention(q, k, v, L)
    assert_close(o, ref, "covering window")
    assert (o.float() - od.float()).abs().max().item() <= 2e-2
    check_device_status()


def test_blocksparse_2k_sampled_two_whole_heads_and_deterministic():
    w = WORKLOADS["blocksparse_2k"]
    inp = make_inputs(w)
    step = w.steps[0]
    q = inp.q[step]
    B, H, N, D = q.shape
    L = cache_len(w.sides, step)
    p = V.problem(B, H, D, w.sides)
    o1 = run_sparse(p, step, q, inp.k, inp.v, w.radius, w.sink_max_side)
    o2 = run_sparse(p, step, q, inp.k, inp.v, w.radius, w.sink_max_side)
    assert torch.equal(o1, o2), "two runs on the same inputs differ"
    g = np.random.default_rng(4)
    rows = set(int(r) for r in g.integers(0, B * H * N, size=96))
    for bh in (0, B * H - 1):
        for (y, x) in ((0, 0), (0, 127), (127, 0), (127, 127), (64, 64), (7, 8), (8, 7), (63, 64)):
            rows.add(bh * N + y * 128 + x)
    rows = np.array(sorted(rows), dtype=np.int64)
    ref = oracle.attention(q, inp.k, inp.v, L, rows=rows,
                           mask=oracle.mask_spec(w.sides, step, w.qblock_side, w.radius, w.sink_max_side))
    got = o1.reshape(-1, D)[torch.as_tensor(rows, device=DEV)]
    assert_close(got, ref, "blocksparse 2k sampled")
    # every row of two whole (b, h): the first and the last
    spec = oracle.mask_spec(w.sides, step, w.qblock_side, w.radius, w.sink_max_side)
    for bh in (0, B * H - 1):
        rows = np.arange(bh * N, (bh + 1) * N, dtype=np.int64)
        ref = oracle.attention(q, inp.k, inp.v, L, rows=rows, mask=spec)
        assert_close(o1.reshape(-1, D)[bh * N:(bh + 1) * N], ref, f"blocksparse 2k (b,h) {bh} every row")
    check_device_status()


def test_blocksparse_malformed_entry_is_reported():
    sides, D = (1, 2, 4, 8, 16, 32), 128
    step, L, N = 5, cache_len(sides, 5), 1024
    q = randn_bf16((1, 1, N, D), 31)
    k = randn_bf16((1, 1, L, D), 32)
    v = randn_bf16((1, 1, L, D), 33)
    p = V.problem(1, 1, D, sides)

    def corrupt(rp, ent):
        ent[rp[1] - 1] = 31 << 24            # last entry of block 0: a scale with no tensor map
        return ent

    run_sparse(p, step, q, k, v, 1, 4, corrupt)
    assert V.var_device_status(clear=True) == V.VAR_ERR_INVALID_ARG
    check_device_status()
