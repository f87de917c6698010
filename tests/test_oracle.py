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
