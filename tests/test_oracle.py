"""Pins for the CPU oracle: each check ties it to something other than itself
(brute force, closed forms, invariants, hand-derived fixtures, a library
routine), chosen so that a dropped term, a wrong sign or index, or a transposed
operand fails at least one of them."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from var_synth import randn_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def bf(a) -> torch.Tensor:
    return torch.tensor(a, dtype=torch.float64).to(torch.bfloat16)


def cum(sides, step):
    return sum(s * s for s in sides[: step + 1])


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("sides,D", [((1, 2, 3), 4), ((1, 2, 4), 8), ((1, 3, 5), 8)])
def test_attention_matches_bruteforce(sides, D):
    B, H = 2, 2
    step = len(sides) - 1
    L, N = cum(sides, step), sides[step] ** 2
    q = randn_bf16((B, H, N, D), 11)
    k = randn_bf16((B, H, L, D), 12)
    v = randn_bf16((B, H, L, D), 13)
    got = oracle.attention(q, k, v, L)
    for b in range(B):
        for h in range(H):
            ref = brute.attention(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), 1 / np.sqrt(D))
            assert np.max(np.abs(got[b, h] - ref)) < 1e-12


# ---------------------------------------------------------------- attention retrospect (ARVAR)

def _np_bits(t):
    return t.float().double().numpy()


def test_attention_lse_and_saliency_match_bruteforce():
    B, H, D = 2, 2, 16
    sides = (2, 3)                       # cache: 4 + 9 tokens; the source grid is the 3x3 scale
    L, N = 13, 9
    q = randn_bf16((B, H, N, D), 311)
    k = randn_bf16((B, H, L, D), 312)
    scale = 1.0 / np.sqrt(D)
    s = np.einsum("bhnd,bhld->bhnl", _np_bits(q), _np_bits(k)) * scale
    lse_ref = np.log2(np.exp(s).sum(-1))
    assert np.allclose(oracle.attention_lse(q, k, L), lse_ref, rtol=0, atol=1e-12)
    P = np.exp(s - s.max(-1, keepdims=True))
    P /= P.sum(-1, keepdims=True)
    sal_ref = P[..., L - N:].sum(axis=2)               # per (b, h, source key): sum over queries
    assert np.allclose(oracle.saliency(q, k, L), sal_ref, rtol=0, atol=1e-12)


def test_saliency_closed_forms():
    B, H, D, N, L = 1, 2, 8, 16, 21
    zero_q = torch.zeros((B, H, N, D), dtype=torch.bfloat16)
    k = randn_bf16((B, H, L, D), 313)
    # zero queries: every key gets 1/L from every query
    assert np.allclose(oracle.saliency(zero_q, k, L), N / L, rtol=0, atol=1e-12)
    # a cache that is only the source scale: each query's mass (1) all lands in it
    q = randn_bf16((B, H, N, D), 314)
    kk = randn_bf16((B, H, N, D), 315)
    assert np.allclose(oracle.saliency(q, kk, N).sum(-1), N, rtol=0, atol=1e-9)


@pytest.mark.parametrize("sp,s", [(3, 5), (4, 8), (32, 64), (5, 5), (7, 3)])
def test_bilinear_map_matches_library_interpolate(sp, s):
    m = np.random.default_rng(sp * 100 + s).standard_normal((2, sp * sp))
    ref = torch.nn.functional.interpolate(torch.from_numpy(m).reshape(2, 1, sp, sp), size=(s, s),
                                          mode="bilinear", align_corners=False).reshape(2, s * s).numpy()
    assert np.allclose(oracle.bilinear_map(m, s), ref, rtol=0, atol=1e-12)


def test_top_k_ascending_ties_and_order():
    v = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.5]])
    assert np.array_equal(oracle.top_k_ascending(v, 2), [[1, 2]])      # ties: lower index first
    assert np.array_equal(oracle.top_k_ascending(v, 4), [[1, 2, 3, 4]])
    assert np.array_equal(oracle.top_k_ascending(np.zeros((2, 7)), 3), [[0, 1, 2], [0, 1, 2]])
    idx, vals = oracle.guided_pivot(np.ones((2, 3, 4)), 4, 5)            # constant map: all tie
    assert np.array_equal(idx, [[0, 1, 2, 3, 4]] * 2) and np.allclose(vals, 1.0 / 4)


def test_guided_pivot_values_follow_the_stated_order():
    """The interpolated values are the head sum (heads added in order), divided
    by H N', then the bilinear formula term by term: bit for bit equal to the
    same operations on Python floats."""
    sal = np.random.default_rng(7).random((2, 3, 16))
    sp, s = 4, 6
    _, v = oracle.guided_pivot(sal, s, 5)
    for b in range(2):
        m = []
        for j in range(16):
            acc = 0.0
            for h in range(3):
                acc += float(sal[b, h, j])
            m.append(acc / (3 * 16))
        for y in range(s):
            for x in range(s):
                def ax(d):
                    src = max((d + 0.5) * sp / s - 0.5, 0.0)
                    i0 = min(int(np.floor(src)), sp - 1)
                    return i0, min(i0 + 1, sp - 1), src - i0
                y0, y1, ly = ax(y)
                x0, x1, lx = ax(x)
                top = m[y0 * sp + x0] * (1 - lx) + m[y0 * sp + x1] * lx
                bot = m[y1 * sp + x0] * (1 - lx) + m[y1 * sp + x1] * lx
                assert v[b, y * s + x] == top * (1 - ly) + bot * ly


def test_branch_halved_attention_repeats_the_conditional_half():
    # the conditional half is the plain attention of those batch elements; the
    # unconditional half carries the same values, whatever its own inputs
    sides, B, H, D = (1, 2, 3), 4, 2, 8
    L, N = 14, 9
    q = randn_bf16((B, H, N, D), 301)
    k = randn_bf16((B, H, L, D), 302)
    v = randn_bf16((B, H, L, D), 303)
    out = oracle.branch_halved_attention(q, k, v, L)
    full = oracle.attention(q, k, v, L)
    assert np.array_equal(out[:2], full[:2])
    assert np.array_equal(out[2:], full[:2])
    assert not np.allclose(out[2:], full[2:])       # not the unconditional branch's own attention


def test_attention_two_keys_golden():
    g = json.load(open(os.path.join(GOLDEN, "attention_two_keys.json")))
    q = bf(g["q"]).reshape(1, 1, 1, 2)
    k = bf(g["k"]).reshape(1, 1, 2, 2)
    v = bf(g["v"]).reshape(1, 1, 2, 2)
    got = oracle.attention(q, k, v, 2, scale=g["scale"])[0, 0]
    assert np.allclose(got, np.array(g["o"]), rtol=0, atol=1e-15)


def test_attention_rows_sum_to_one():
    # a value column that is 1 everywhere comes out as exactly the row sum of P
    q = randn_bf16((1, 2, 9, 8), 1)
    k = randn_bf16((1, 2, 14, 8), 2)
    v = randn_bf16((1, 2, 14, 8), 3)
    v[..., 3] = 1.0
    o = oracle.attention(q, k, v, 14)
    assert np.max(np.abs(o[..., 3] - 1.0)) < 1e-14


def test_attention_identical_values_and_zero_query():
    q = randn_bf16((1, 1, 4, 8), 4)
    k = randn_bf16((1, 1, 5, 8), 5)
    row = randn_bf16((8,), 6)
    v = row.expand(1, 1, 5, 8).contiguous()
    o = oracle.attention(q, k, v, 5)
    assert np.max(np.abs(o - f64(row))) < 1e-14
    # q = 0: uniform weights -> plain mean of the value rows
    v2 = randn_bf16((1, 1, 5, 8), 7)
    o2 = oracle.attention(torch.zeros_like(q), k, v2, 5)
    assert np.max(np.abs(o2[0, 0] - f64(v2[0, 0]).mean(axis=0))) < 1e-14


def test_attention_single_key_and_cache_prefix():
    q = randn_bf16((2, 2, 3, 8), 8)
    k = randn_bf16((2, 2, 6, 8), 9)
    v = randn_bf16((2, 2, 6, 8), 10)
    o = oracle.attention(q, k, v, 1)       # only the first cached key is visible
    assert np.max(np.abs(o - f64(v[:, :, :1]))) < 1e-15
    # the prefix of a larger cache equals a cache of exactly that length
    o3 = oracle.attention(q, k, v, 4)
    o4 = oracle.attention(q, k[:, :, :4].contiguous(), v[:, :, :4].contiguous(), 4)
    assert np.array_equal(o3, o4)


def test_attention_key_permutation_invariance():
    q = randn_bf16((1, 2, 16, 8), 14)
    k = randn_bf16((1, 2, 21, 8), 15)
    v = randn_bf16((1, 2, 21, 8), 16)
    perm = torch.randperm(21, generator=torch.Generator().manual_seed(0))
    o = oracle.attention(q, k, v, 21)
    op = oracle.attention(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), 21)
    assert np.max(np.abs(o - op)) < 1e-13


def test_attention_row_sampling_equals_full():
    q = randn_bf16((2, 2, 9, 8), 17)
    k = randn_bf16((2, 2, 14, 8), 18)
    v = randn_bf16((2, 2, 14, 8), 19)
    full = oracle.attention(q, k, v, 14).reshape(-1, 8)
    rows = np.array([0, 5, 17, 35, 20])
    part = oracle.attention(q, k, v, 14, rows=rows)
    assert np.array_equal(part, full[rows])


# ---------------------------------------------------------------- block mask

@pytest.mark.parametrize("sides,qbs,radius,sink", [
    ((1, 2, 4, 6, 8, 12, 16), 4, 1, 4),
    ((1, 2, 4, 8, 12, 16, 24, 32), 8, 1, 8),
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32), 8, 2, 16),
    ((1, 3, 5, 10, 15, 20), 5, 1, 5),
])
def test_block_mask_matches_bruteforce(sides, qbs, radius, sink):
    step = len(sides) - 1
    m = oracle.mask_spec(sides, step, qbs, radius, sink)
    got = oracle.block_mask_rows(m, 0, sides[step] ** 2).astype(bool)
    ref = brute.block_mask(sides, step, qbs, radius, sink)
    assert np.array_equal(got, ref)


def test_block_mask_own_scale_is_plus_minus_radius_blocks():
    sides = (1, 2, 4, 8, 16, 32)
    m = oracle.mask_spec(sides, 5, 4, 2, 4)
    mask = oracle.block_mask_rows(m, 0, 32 * 32).astype(bool)
    off = cum(sides, 4)
    for qi in (0, 5 * 32 + 17, 31 * 32 + 31, 12 * 32 + 3):
        by, bx = (qi // 32) // 4, (qi % 32) // 4
        own = mask[qi, off:].reshape(32, 32)
        ky, kx = np.nonzero(own)
        assert set(ky // 4) == set(range(max(0, by - 2), min(8, by + 3)))
        assert set(kx // 4) == set(range(max(0, bx - 2), min(8, bx + 3)))
        assert mask[qi, :cum(sides, 2)].all()       # sink scales (side <= 4) whole


def test_block_mask_huge_radius_is_dense():
    sides = (1, 2, 4, 8, 16)
    m = oracle.mask_spec(sides, 4, 4, 100, 2)
    assert oracle.block_mask_rows(m, 0, 256).all()


def test_masked_attention_is_dense_attention_on_kept_keys():
    sides = (1, 2, 4, 8, 16)
    step, D = 4, 8
    L, N = cum(sides, step), 256
    m = oracle.mask_spec(sides, step, 4, 1, 2)
    q = randn_bf16((1, 2, N, D), 20)
    k = randn_bf16((1, 2, L, D), 21)
    v = randn_bf16((1, 2, L, D), 22)
    got = oracle.attention(q, k, v, L, mask=m)
    keep = oracle.block_mask_rows(m, 0, N).astype(bool)
    for h in range(2):
        for qi in (0, 37, 130, 255):
            kk = k[0, h, keep[qi]].reshape(1, 1, -1, D).contiguous()
            vv = v[0, h, keep[qi]].reshape(1, 1, -1, D).contiguous()
            ref = oracle.attention(q[0:1, h:h + 1, qi:qi + 1].contiguous(), kk, vv, kk.shape[2])
            assert np.max(np.abs(got[0, h, qi] - ref[0, 0, 0])) < 1e-13
    # a window that covers everything reproduces dense attention
    big = oracle.mask_spec(sides, step, 4, 100, 2)
    assert np.max(np.abs(oracle.attention(q, k, v, L, mask=big) - oracle.attention(q, k, v, L))) < 1e-13


# ---------------------------------------------------------------- pivot selection

@pytest.mark.parametrize("N,Cc,K,seed", [(16, 8, 5, 0), (25, 6, 10, 1), (36, 4, 1, 2),
                                          (40, 16, 39, 3), (9, 32, 9, 4), (30, 5, 0, 5)])
def test_pivot_matches_exact_rational_ranking(N, Cc, K, seed):
    x = randn_bf16((2, N, Cc), 100 + seed)
    idx, _ = oracle.pivot_select(x, K)
    for b in range(2):
        assert list(idx[b]) == brute.pivot_ranking_exact(f64(x[b]), K)


def test_pivot_mean_is_exact_for_bf16_grid():
    from fractions import Fraction
    x = randn_bf16((1, 64, 4), 7)
    m = oracle.pivot_mean(x)
    xs = f64(x[0])
    for c in range(4):
        exact = sum(Fraction(float(t)) for t in xs[:, c]) / 64
        assert m[0, c] == float(exact)


def test_pivot_scores_closed_form():
    # one non-zero channel: score_i = (t_i - mean t)^2 exactly
    t = torch.tensor([3.0, -1.0, 0.5, 2.0, -4.0, 0.0, 1.0, 6.0])
    x = torch.zeros(1, 8, 16)
    x[0, :, 5] = t
    x = x.to(torch.bfloat16)
    sc = oracle.pivot_scores(x)[0]
    mean = float(t.mean())
    assert np.array_equal(sc, ((t.double() - mean) ** 2).numpy())
    idx, _ = oracle.pivot_select(x, 3)
    assert list(idx[0]) == [0, 4, 7]       # |t - 0.9375|: 2.06, 4.94, 5.06 largest


def test_pivot_constant_grid_and_ties():
    x = torch.full((2, 20, 8), 0.75).to(torch.bfloat16)
    idx, sc = oracle.pivot_select(x, 6)
    assert (sc == 0).all()
    assert (idx == np.arange(6)).all()       # all tied: lowest indices
    y = randn_bf16((1, 20, 8), 9)
    y[0, 13] = 5.0
    y[0, 4] = 5.0                             # rows 4 and 13 identical and extreme
    idx, sc = oracle.pivot_select(y, 1)
    assert sc[0, 4] == sc[0, 13]
    assert list(idx[0]) == [4]
    idx2, _ = oracle.pivot_select(y, 2)
    assert list(idx2[0]) == [4, 13]


def test_pivot_keep_all_and_none():
    x = randn_bf16((2, 12, 8), 10)
    idx, _ = oracle.pivot_select(x, 12)
    assert (idx == np.arange(12)).all()
    idx0, _ = oracle.pivot_select(x, 0)
    assert idx0.shape == (2, 0)


# ---------------------------------------------------------------- restore + scatter

def test_restore_bilinear_golden():
    g = json.load(open(os.path.join(GOLDEN, "bilinear_2x2_to_4x4.json")))
    prev = bf(g["prev"]).reshape(1, 1, 4, 1)
    oc = torch.zeros(1, 1, 0, 1, dtype=torch.bfloat16)
    out = oracle.restore_scatter(prev, oc, np.zeros((1, 0), np.int32), 4)
    assert np.array_equal(out.reshape(4, 4), np.array(g["out"]))


@pytest.mark.parametrize("sp,s", [(2, 3), (3, 5), (40, 48), (48, 64), (5, 5), (6, 13)])
def test_restore_matches_library_interpolate(sp, s):
    D = 4
    prev = randn_bf16((1, 2, sp * sp, D), sp * 100 + s)
    oc = torch.zeros(1, 2, 0, D, dtype=torch.bfloat16)
    out = oracle.restore_scatter(prev, oc, np.zeros((1, 0), np.int32), s)
    g = prev.double().reshape(1, 2, sp, sp, D).permute(0, 1, 4, 2, 3).reshape(2, D, sp, sp)
    ref = torch.nn.functional.interpolate(g, size=(s, s), mode="bilinear", align_corners=False,
                                          antialias=False)
    ref = ref.reshape(1, 2, D, s * s).permute(0, 1, 3, 2).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12
    if sp == s:
        assert np.array_equal(out, f64(prev))


def test_restore_constant_and_affine():
    sp, s, D = 6, 13, 2
    prev = torch.full((1, 1, sp * sp, D), 1.5).to(torch.bfloat16)
    out = oracle.restore_scatter(prev, torch.zeros(1, 1, 0, D, dtype=torch.bfloat16),
                                 np.zeros((1, 0), np.int32), s)
    assert np.all(out == 1.5)
    # affine ramp a + b*y + c*x is reproduced exactly where no clamping happens
    yy, xx = np.meshgrid(np.arange(sp), np.arange(sp), indexing="ij")
    ramp = (0.5 + 0.25 * yy - 0.125 * xx).reshape(sp * sp, 1)
    prev = torch.tensor(np.repeat(ramp, D, axis=1)).reshape(1, 1, sp * sp, D).to(torch.bfloat16)
    assert np.array_equal(f64(prev)[0, 0, :, 0], ramp[:, 0])
    out = oracle.restore_scatter(prev, torch.zeros(1, 1, 0, D, dtype=torch.bfloat16),
                                 np.zeros((1, 0), np.int32), s)
    for y in range(s):
        for x in range(s):
            sy = (y + 0.5) * sp / s - 0.5
            sx = (x + 0.5) * sp / s - 0.5
            if 0 <= sy <= sp - 1 and 0 <= sx <= sp - 1:
                assert abs(out[0, 0, y * s + x, 0] - (0.5 + 0.25 * sy - 0.125 * sx)) < 1e-14


def test_restore_scatter_overwrites_and_bruteforce():
    B, H, sp, s, D, K = 2, 3, 5, 8, 4, 17
    prev = randn_bf16((B, H, sp * sp, D), 30)
    oc = randn_bf16((B, H, K, D), 31)
    g = torch.Generator().manual_seed(32)
    idx = np.stack([np.sort(torch.randperm(s * s, generator=g)[:K].numpy()) for _ in range(B)])
    out = oracle.restore_scatter(prev, oc, idx.astype(np.int32), s)
    for b in range(B):
        for h in range(H):
            ref = brute.restore_scatter(f64(prev[b, h]), f64(oc[b, h]), idx[b], s)
            assert np.max(np.abs(out[b, h] - ref)) < 1e-13
            assert np.array_equal(out[b, h, idx[b]], f64(oc[b, h]))   # overwrite, not add
    # K = N: the output is exactly the compact rows
    full = np.tile(np.arange(s * s, dtype=np.int32), (B, 1))
    oc_all = randn_bf16((B, H, s * s, D), 33)
    assert np.array_equal(oracle.restore_scatter(prev, oc_all, full, s), f64(oc_all))


def test_restore_rejects_bad_indices():
    prev = randn_bf16((1, 1, 4, 2), 40)
    oc = randn_bf16((1, 1, 2, 2), 41)
    with pytest.raises(ValueError):
        oracle.restore_scatter(prev, oc, np.array([[3, 3]], np.int32), 3)   # duplicate
    with pytest.raises(ValueError):
        oracle.restore_scatter(prev, oc, np.array([[0, 9]], np.int32), 3)   # out of range


# ---------------------------------------------------------------- dynamic pattern (SparVAR)

SV_SIDES = (1, 2, 4, 8, 16, 24, 32)      # sinks: the 1, 2, 4 scales (21 tokens) at sink_max_side 4
SV_SINK = 4


def _np_probs(q, k, L):
    D = q.shape[-1]
    s = np.einsum("bhnd,bhld->bhnl", _np_bits(q), _np_bits(k[:, :, :L])) / np.sqrt(D)
    P = np.exp(s - s.max(-1, keepdims=True))
    return P / P.sum(-1, keepdims=True)


def test_sparvar_units_partition_the_keys():
    d = 5                                             # decision scale 24
    unit_of, units, n_sink = oracle.sparvar_units(SV_SIDES, d, SV_SINK)
    L = cum(SV_SIDES, d)
    assert len(unit_of) == L and n_sink == 1
    sizes = np.bincount(unit_of, minlength=len(units))
    assert sizes[0] == 21                             # the sink range in one 64-token chunk
    for idx in range(n_sink, len(units)):
        sc, u, v = units[idx]
        s = SV_SIDES[sc]
        assert sizes[idx] == min(8, s - 8 * u) * min(8, s - 8 * v)
    assert len(units) == 1 + 1 + 4 + 9               # 8: one block, 16: 2x2, 24: 3x3
    # a block's keys are exactly its rows and columns of its scale
    off = cum(SV_SIDES, 4)                            # start of the 24 scale
    j = off + 9 * 24 + 17                             # row 9, column 17 -> block (1, 2)
    assert units[unit_of[j]] == (5, 1, 2)


def test_sparvar_unit_mass_matches_bruteforce():
    B, H, D, d = 2, 2, 16, 4                          # decision scale 16 (2 x 2 query blocks)
    L, N = cum(SV_SIDES, d), 16 * 16
    q = randn_bf16((B, H, N, D), 701)
    k = randn_bf16((B, H, L + 5, D), 702)             # a cache with spare capacity
    unit_of, units, n_sink = oracle.sparvar_units(SV_SIDES, d, SV_SINK)
    P = _np_probs(q, k, L)
    mass = np.zeros(P.shape[:3] + (len(units),))
    for u in range(len(units)):
        mass[..., u] = P[..., unit_of == u].sum(-1)
    A_ref = mass.reshape(B, H, 2, 8, 2, 8, len(units)).sum(axis=(0, 1, 3, 5)).reshape(4, -1) / (B * H * 64)
    A = oracle.sparvar_scores(q, k, SV_SIDES, d, SV_SINK)
    assert np.max(np.abs(A - A_ref)) < 1e-13
    assert np.allclose(A.sum(axis=1), 1.0, rtol=0, atol=1e-12)   # every query's mass is 1


def test_sparvar_block_score_sums_in_the_stated_order():
    """The block score adds the 2 x 2 x 64 per-query masses one at a time in the
    order (b, h, y, x), in fp64, then divides by B H 64: equal bit for bit to
    that sequence of additions done with Python floats."""
    B, H, D, d = 2, 2, 16, 4
    L, N = cum(SV_SIDES, d), 16 * 16
    q = randn_bf16((B, H, N, D), 711)
    k = randn_bf16((B, H, L, D), 712)
    unit_of, units, _ = oracle.sparvar_units(SV_SIDES, d, SV_SINK)
    U = len(units)
    mass = np.zeros((B, H, N, U))
    lib = oracle.lib()
    assert lib.oracle_unit_mass(B, H, N, L, L, D, 1.0 / np.sqrt(D), oracle._ptr(oracle._bits(q)),
                                oracle._ptr(oracle._bits(k)), oracle._ptr(unit_of), U, oracle._ptr(mass)) == 0
    A = oracle.sparvar_scores(q, k, SV_SIDES, d, SV_SINK)
    for qb in range(4):
        by, bx = divmod(qb, 2)
        for u in range(U):
            acc = 0.0
            for b in range(B):
                for h in range(H):
                    for y in range(8):
                        for x in range(8):
                            acc += float(mass[b, h, (8 * by + y) * 16 + 8 * bx + x, u])
            assert A[qb, u] == acc / (B * H * 64)


def test_sparvar_unit_mass_uniform_closed_form():
    # q = 0: every key gets 1/L, so a unit's mass is its size over L
    B, H, D, d = 1, 2, 8, 4
    L = cum(SV_SIDES, d)
    q = torch.zeros((B, H, 256, D), dtype=torch.bfloat16)
    k = randn_bf16((B, H, L, D), 703)
    unit_of, units, _ = oracle.sparvar_units(SV_SIDES, d, SV_SINK)
    A = oracle.sparvar_scores(q, k, SV_SIDES, d, SV_SINK)
    sizes = np.bincount(unit_of, minlength=len(units))
    assert np.allclose(A, np.tile(sizes / L, (4, 1)), rtol=0, atol=1e-14)


def test_sparvar_select_threshold_rule():
    A = np.array([[0.1, 0.3, 0.2, 0.3, 0.1],          # unit 0 is the sink
                  [0.5, 0.1, 0.1, 0.1, 0.2]])
    assert oracle.sparvar_select(A, 1, 0.0) == [[], []]
    assert oracle.sparvar_select(A, 1, 1.0) == [[1, 2, 3, 4], [1, 2, 3, 4]]
    # tau 0.5: row 0 takes unit 1 (tie with 3, lower index first): 0.1 + 0.3 = 0.4 < 0.5,
    # then unit 3: 0.7; row 1: the sink alone holds 0.5
    assert oracle.sparvar_select(A, 1, 0.5) == [[1, 3], []]
    assert oracle.sparvar_select(A, 1, 0.75) == [[1, 2, 3], [1, 4]]
    # monotone in tau
    prev = [set(), set()]
    for tau in np.linspace(0, 1, 21):
        cur = [set(x) for x in oracle.sparvar_select(A, 1, tau)]
        assert all(p <= c for p, c in zip(prev, cur))
        prev = cur


def test_sparvar_keep_mask_identity_at_the_decision_step():
    d = 5
    unit_of, units, n_sink = oracle.sparvar_units(SV_SIDES, d, SV_SINK)
    rng = np.random.default_rng(704)
    kept = [sorted(rng.choice(np.arange(n_sink, len(units)), size=3, replace=False).tolist()) for _ in range(9)]
    keep = oracle.sparvar_keep_mask(SV_SIDES, d, d, units, kept, SV_SINK)
    s = SV_SIDES[d]
    for i in range(s * s):
        qb = (i // s // 8) * 3 + (i % s) // 8
        want = np.isin(unit_of, list(range(n_sink)) + kept[qb]).astype(np.uint8)
        assert np.array_equal(keep[i], want)


def test_sparvar_keep_mask_maps_by_rescaling():
    # decision 16 (2 x 2 blocks) -> target 32 (4 x 4 blocks): target block (by, bx) reads
    # decision block (by // 2, bx // 2); a kept 16-scale block (u, v) covers the 24 scale
    # rows [floor(8u * 1.5), ceil((8u + 8) * 1.5)) and exactly block (u, v) of the 16
    # scale, and at the 32 scale the 2 x 2 blocks (2u.., 2v..)
    d, k_step = 4, 6
    unit_of, units, n_sink = oracle.sparvar_units(SV_SIDES, d, SV_SINK)
    idx = {units[i]: i for i in range(len(units))}
    kept = [[idx[(4, 0, 1)], idx[(3, 0, 0)]], [], [], [idx[(4, 1, 1)]]]
    keep = oracle.sparvar_keep_mask(SV_SIDES, d, k_step, units, kept, SV_SINK)
    offs = np.cumsum([0] + [s * s for s in SV_SIDES])
    L = offs[k_step + 1]
    assert keep.shape == (32 * 32, L)

    def grid(row, sc):
        s = SV_SIDES[sc]
        return row[offs[sc]:offs[sc] + s * s].reshape(s, s)

    # a query of target block (0, 1) -> decision block (0, 0): sinks, (3,0,0), (4,0,1) mapped
    r = keep[0 * 32 + 9]
    assert r[:21].all()
    assert grid(r, 3).all()                                   # the whole 8 scale
    g16 = grid(r, 4)
    assert g16[:8, 8:].all() and g16.sum() == 64
    g24 = grid(r, 5)                                          # rows [0, 12) -> blocks 0, 1; cols [12, 24) -> 1, 2
    want = np.zeros((24, 24), dtype=np.uint8)
    want[:16, 8:24] = 1
    assert np.array_equal(g24, want)
    g32 = grid(r, 6)
    want = np.zeros((32, 32), dtype=np.uint8)
    want[:16, 16:32] = 1
    assert np.array_equal(g32, want)
    # target block (1, 1) reads decision block (0, 0) too; block (2, 2) reads (1, 1)
    assert np.array_equal(keep[8 * 32 + 8], keep[0 * 32 + 9])
    r2 = keep[16 * 32 + 16]
    assert grid(r2, 3).sum() == 0 and grid(r2, 4)[8:, 8:].all() and grid(r2, 4).sum() == 64
    # nothing outside the sinks for blocks that kept nothing
    assert keep[0 * 32 + 20][21:].sum() == 0


def test_sparvar_keep_mask_covers_the_rescaled_block():
    # every key whose position, mapped back to the decision scale, falls inside a kept
    # decision-scale block is kept; every kept block of a later scale touches it
    d, k_step = 5, 6                                          # 24 -> 32
    unit_of, units, n_sink = oracle.sparvar_units(SV_SIDES, d, SV_SINK)
    kept = [[i for i in range(n_sink, len(units)) if units[i][0] == 5 and (units[i][1] + units[i][2]) % 3 == 0]] * 9
    keep = oracle.sparvar_keep_mask(SV_SIDES, d, k_step, units, kept, SV_SINK)
    offs = np.cumsum([0] + [s * s for s in SV_SIDES])
    row = keep[0]
    sel = {(units[i][1], units[i][2]) for i in kept[0]}
    s_d, s2 = 24, 32
    g = row[offs[6]:offs[6] + s2 * s2].reshape(s2, s2)
    for y in range(s2):
        for x in range(s2):
            # the decision-scale area of this key [y, y+1) x [x, x+1) scaled by 24/32
            ys = {int(np.floor(y * s_d / s2)), int(np.ceil((y + 1) * s_d / s2)) - 1}
            xs = {int(np.floor(x * s_d / s2)), int(np.ceil((x + 1) * s_d / s2)) - 1}
            inside = any((yy // 8, xx // 8) in sel for yy in ys for xx in xs)
            if inside:
                assert g[y, x] == 1
            if g[y, x]:
                # some decision block of the selection meets this key's whole 8 x 8 block
                by, bx = y // 8, x // 8
                ry = range(int(np.floor(8 * by * s_d / s2)), int(np.ceil((8 * by + 8) * s_d / s2)))
                rx = range(int(np.floor(8 * bx * s_d / s2)), int(np.ceil((8 * bx + 8) * s_d / s2)))
                assert any((yy // 8, xx // 8) in sel for yy in ry for xx in rx)


def test_attention_keep_matches_dense_masked_and_bruteforce():
    B, H, D = 1, 2, 8
    sides = (1, 2, 4, 8)
    L, N = cum(sides, 3), 64
    q = randn_bf16((B, H, N, D), 705)
    k = randn_bf16((B, H, L, D), 706)
    v = randn_bf16((B, H, L, D), 707)
    ones = np.ones((N, L), dtype=np.uint8)
    assert np.max(np.abs(oracle.attention_keep(q, k, v, L, ones) - oracle.attention(q, k, v, L))) < 1e-15
    rng = np.random.default_rng(708)
    keep = (rng.random((N, L)) < 0.3).astype(np.uint8)
    keep[5] = 0                                               # a row that keeps nothing: zeros
    got = oracle.attention_keep(q, k, v, L, keep)
    s = np.einsum("bhnd,bhld->bhnl", _np_bits(q), _np_bits(k)) / np.sqrt(D)
    s = np.where(keep[None, None] > 0, s, -np.inf)
    for i in range(N):
        if keep[i].sum() == 0:
            assert np.all(got[:, :, i] == 0)
            continue
        p = np.exp(s[:, :, i] - s[:, :, i].max(-1, keepdims=True))
        ref = np.einsum("bhl,bhld->bhd", p / p.sum(-1, keepdims=True), _np_bits(v))
        assert np.max(np.abs(got[:, :, i] - ref)) < 1e-12
