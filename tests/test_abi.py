"""Host-side checks of the C ABI (no GPU): the library loads, exports every
declared entry point, rejects bad arguments before touching the device, and
its host-built block mask equals the oracle's token-level rule exactly."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import SCHEDULE_1024, SCHEDULE_2K, SCHEDULE_256
from tests._util import csr_to_token_mask as _csr_to_token_mask


def test_library_exports_every_declared_symbol():
    names = V.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(V.lib(), n), n
    for n in ("var_attn_dense", "var_attn_pruned", "var_attn_blocksparse", "var_pivot_select",
              "var_restore_scatter"):
        assert n in names


def test_keep_count_and_status_strings():
    assert V.var_keep_count(4096, 1, 5) == 819
    assert V.var_keep_count(2304, 2, 5) == 921
    assert V.var_keep_count(4096, 1, 1) == 4096
    assert V.var_keep_count(7, 0, 3) == 0
    assert V.var_keep_count(7, 4, 3) == -1
    for s in range(7):
        assert V.var_status_string(s) != "unknown status"
    assert V.var_status_string(99) == "unknown status"


def _fake(n=1 << 20):
    # a host address never dereferenced: every call below must fail validation first
    return C.c_void_p(0x10000)


@pytest.mark.parametrize("head_dim,expect", [(96, V.VAR_ERR_UNSUPPORTED), (0, V.VAR_ERR_UNSUPPORTED)])
def test_dense_rejects_head_dim(head_dim, expect):
    p = V.problem(1, 2, head_dim, SCHEDULE_256)
    assert V.lib().var_attn_dense(C.byref(p), 9, _fake(), _fake(), _fake(), _fake(), None) == expect


def test_dense_rejects_bad_arguments():
    L = V.lib()
    p = V.problem(1, 2, 64, SCHEDULE_256)
    f = _fake()
    assert L.var_attn_dense(C.byref(p), 9, None, f, f, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_dense(C.byref(p), 10, f, f, f, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_dense(C.byref(p), -1, f, f, f, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_dense(None, 0, f, f, f, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_dense(C.byref(p), 9, C.c_void_p(0x10008), f, f, f, None) == V.VAR_ERR_UNSUPPORTED
    small = V.problem(1, 2, 64, SCHEDULE_256, kv_capacity=679)
    assert L.var_attn_dense(C.byref(small), 9, f, f, f, f, None) == V.VAR_ERR_INVALID_ARG
    neg = V.problem(1, 2, 64, SCHEDULE_256, softmax_scale=-1.0)
    assert L.var_attn_dense(C.byref(neg), 9, f, f, f, f, None) == V.VAR_ERR_INVALID_ARG


def test_pruned_restore_pivot_reject_bad_arguments():
    L = V.lib()
    p = V.problem(2, 16, 128, SCHEDULE_1024)
    f = _fake()
    assert L.var_attn_pruned(C.byref(p), 12, f, f, f, f, 4097, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_pruned(C.byref(p), 12, f, f, f, f, -1, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_pruned(C.byref(p), 12, f, f, f, None, 5, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_pruned(C.byref(p), 12, f, f, f, f, 0, f, None) == V.VAR_OK   # no-op
    assert L.var_restore_scatter(C.byref(p), 0, f, f, f, 4, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_restore_scatter(C.byref(p), 12, f, None, None, 3, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_restore_scatter(C.byref(p), 12, f, f, f, 4097, f, None) == V.VAR_ERR_INVALID_ARG
    ws = L.var_pivot_workspace_bytes(C.byref(p), 12, 2048)
    assert ws > 0
    assert L.var_pivot_workspace_bytes(C.byref(p), 12, 2047) == 0
    assert L.var_pivot_select(C.byref(p), 12, f, 2048, 819, f, None, None, 0, None) == V.VAR_ERR_WORKSPACE
    assert L.var_pivot_select(C.byref(p), 12, f, 2048, 819, f, None, f, ws - 1, None) == V.VAR_ERR_WORKSPACE
    assert L.var_pivot_select(C.byref(p), 12, f, 2040, 819, f, None, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_pivot_select(C.byref(p), 12, f, 2048, 4097, f, None, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_pruned_scatter(C.byref(p), 12, f, f, f, f, 4097, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_pruned_scatter(C.byref(p), 12, f, f, f, None, 5, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_pruned_scatter(C.byref(p), 12, f, f, f, f, 0, f, None) == V.VAR_OK   # no-op
    assert L.var_restore_fill(C.byref(p), 0, f, f, 4, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_restore_fill(C.byref(p), 12, f, None, 3, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_restore_fill(C.byref(p), 12, f, f, -1, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_pruned_in_place(C.byref(p), 0, f, f, f, f, f, 4, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_pruned_in_place(C.byref(p), 12, f, f, f, f, None, 3, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_pruned_in_place(C.byref(p), 12, None, f, f, f, f, 3, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_pruned_in_place(C.byref(p), 12, f, f, f, None, f, 3, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_pruned_in_place(C.byref(p), 12, f, f, f, f, f, -1, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_pruned_in_place(C.byref(p), 12, f, f, f, f, f, 4097, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_pruned_in_place(C.byref(p), 12, f, f, f, C.c_void_p(0x10008), f, 3, f, None) == \
        V.VAR_ERR_UNSUPPORTED
    step = L.var_pruned_step
    assert step(C.byref(p), 0, f, 2048, 819, f, f, f, f, f, f, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert step(C.byref(p), 12, None, 2048, 819, f, f, f, f, f, f, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert step(C.byref(p), 12, f, 2040, 819, f, f, f, f, f, f, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert step(C.byref(p), 12, f, 2048, 4097, f, f, f, f, f, f, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert step(C.byref(p), 12, f, 2048, 819, f, f, f, f, None, f, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert step(C.byref(p), 12, f, 2048, 819, None, f, f, f, f, f, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert step(C.byref(p), 12, f, 2048, 819, f, f, f, None, f, f, f, ws, None) == V.VAR_ERR_INVALID_ARG
    assert step(C.byref(p), 12, f, 2048, 819, f, f, f, f, f, f, None, 0, None) == V.VAR_ERR_WORKSPACE
    assert step(C.byref(p), 12, f, 2048, 819, f, f, f, f, f, f, f, ws - 1, None) == V.VAR_ERR_WORKSPACE
    assert step(C.byref(p), 12, f, 2048, 819, f, f, f, C.c_void_p(0x10008), f, f, f, ws, None) == \
        V.VAR_ERR_UNSUPPORTED
    odd = V.problem(3, 16, 128, SCHEDULE_1024)
    assert L.var_attn_dense_halved(C.byref(odd), 12, f, f, f, f, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_attn_dense_halved(C.byref(p), 12, f, None, f, f, None) == V.VAR_ERR_INVALID_ARG


@pytest.mark.parametrize("sides,qbs,radius,sink", [
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32), 8, 2, 16),
    ((1, 2, 4, 8, 12, 16, 24, 32), 8, 1, 8),
    ((1, 3, 5, 10, 15, 20), 5, 1, 5),
    ((1, 2, 4, 6, 8, 12, 16), 4, 0, 4),
])
def test_block_mask_csr_equals_oracle_token_mask(sides, qbs, radius, sink):
    step = len(sides) - 1
    p = V.problem(1, 1, 64, sides)
    row_ptr, entries, sink_len = V.var_block_mask_build(p, step, qbs, radius, sink)
    assert sink_len == sum(s * s for s in sides if s <= sink)
    got = _csr_to_token_mask(sides, step, qbs, row_ptr, entries, sink_len)
    ref = oracle.block_mask_rows(oracle.mask_spec(sides, step, qbs, radius, sink), 0, sides[step] ** 2)
    assert np.array_equal(got, ref.astype(bool))


def test_block_mask_2k_statistics_and_rows():
    p = V.problem(2, 16, 128, SCHEDULE_2K)
    row_ptr, entries, sink_len = V.var_block_mask_build(p, 15, 8, 2, 16)
    assert sink_len == 521 and row_ptr.shape == (257,) and len(entries) == 20164
    assert np.all(np.diff(row_ptr) > 0)
    for qb in range(256):
        e = entries[row_ptr[qb]:row_ptr[qb + 1]]
        assert np.all(np.diff(e) > 0)             # ascending, no duplicates
    # spot-check whole rows of blocks against the oracle rule
    sides = SCHEDULE_2K
    m = oracle.mask_spec(sides, 15, 8, 2, 16)
    offs = np.cumsum([0] + [s * s for s in sides])
    for qb in (0, 17, 136, 255):
        by, bx = divmod(qb, 16)
        qi = (by * 8) * 128 + bx * 8
        ref = oracle.block_mask_rows(m, qi, qi + 1)[0].astype(bool)
        keys = np.zeros(offs[-1], dtype=bool)
        keys[:sink_len] = True
        for e in entries[row_ptr[qb]:row_ptr[qb + 1]]:
            sc, u, w = e >> 24, (e >> 12) & 0xFFF, e & 0xFFF
            s = sides[sc]
            for r in range(u * 8, min(s, u * 8 + 8)):
                keys[offs[sc] + r * s + w * 8: offs[sc] + r * s + min(s, w * 8 + 8)] = True
        assert np.array_equal(keys, ref)


@pytest.mark.parametrize("sides,radius,sink", [
    (SCHEDULE_2K, 2, 16),
    ((1, 2, 4, 8, 16, 24, 40), 2, 4),          # 5x5 query blocks: squares at the edge are partial
])
def test_block_mask_plan_is_the_union_of_each_square(sides, radius, sink):
    step = len(sides) - 1
    p = V.problem(2, 16, 128, sides)
    rp, en, sink_len = V.var_block_mask_build(p, step, 8, radius, sink)
    sq_ptr, sq_units, sq_order = V.var_block_mask_plan(p, step, 8, rp, en, sink_len)
    nb = sides[step] // 8
    nsq = (nb + 1) // 2
    n_sink = (sink_len + 63) // 64
    assert len(sq_order) == nsq * nsq and sorted(sq_order.tolist()) == list(range(nsq * nsq))
    counts = np.diff(sq_ptr)
    assert all(counts[sq_order[i]] >= counts[sq_order[i + 1]] for i in range(len(sq_order) - 1))
    for sq in range(nsq * nsq):
        by0, bx0 = 2 * (sq // nsq), 2 * (sq % nsq)
        member = {}
        for t in range(4):
            by, bx = by0 + t // 2, bx0 + t % 2
            if by < nb and bx < nb:
                qb = by * nb + bx
                for e in en[rp[qb]:rp[qb + 1]]:
                    member[int(e)] = member.get(int(e), 0) | (1 << t)
        units = sq_units[2 * sq_ptr[sq]: 2 * sq_ptr[sq + 1]].reshape(-1, 2)
        assert len(units) == n_sink + len(member)
        assert [int(u) for u in units[:n_sink, 0]] == [-1 - c for c in range(n_sink)]
        assert [int(u) for u in units[n_sink:, 0]] == sorted(member)
        for e, meta in units[n_sink:]:
            s = sides[int(e) >> 24]
            u, v = (int(e) >> 12) & 0xFFF, int(e) & 0xFFF
            rows, cols = min(8, s - 8 * u), min(8, s - 8 * v)
            assert int(meta) & 0xF == member[int(e)]
            assert (int(meta) >> 8) & 15 == rows and (int(meta) >> 12) & 15 == cols


def test_block_mask_rejects_bad_shapes():
    p = V.problem(1, 1, 64, (1, 2, 4, 6, 8, 12, 16, 20))
    with pytest.raises(V.VarError):
        V.var_block_mask_build(p, 7, 8, 2, 16)      # 20 is not a multiple of 8
    q = V.problem(1, 1, 64, (1, 32, 4, 64))
    with pytest.raises(V.VarError):
        V.var_block_mask_build(q, 3, 8, 1, 4)       # a sink scale after a non-sink one


# ---------------------------------------------------------------- dynamic pattern (SparVAR)

@pytest.mark.parametrize("sides,d,k_step,sink", [
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32, 40, 48, 64), 9, 12, 16),     # 1024px: 32x32 decides 64x64
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32, 40, 48, 64), 11, 12, 16),    # 48 -> 64 (non-integer ratio)
    ((1, 2, 4, 6, 8, 12, 16, 20, 24, 32, 40, 48, 64), 9, 9, 16),      # the decision step itself
    ((1, 2, 4, 8, 16, 24, 32), 4, 6, 4),
])
def test_sparvar_mask_equals_oracle(sides, d, k_step, sink):
    p = V.problem(1, 1, 64, sides)
    U, n_sink = V.var_sparvar_units(p, d, sink)
    unit_of, units, ns = oracle.sparvar_units(sides, d, sink)
    assert (U, n_sink) == (len(units), ns)
    nqb = (sides[d] // 8) ** 2
    rng = np.random.default_rng(901 + d)
    A = rng.random((nqb, U)) ** 3
    A[:, n_sink + 2] = A[:, n_sink + 1]                 # equal scores: the lower unit goes first
    A /= A.sum(axis=1, keepdims=True)
    for tau in (0.0, 0.3, 0.8, 1.0):
        rp, en, sink_len = V.var_sparvar_mask_build(p, d, k_step, sink, A, tau)
        got = _csr_to_token_mask(sides, k_step, 8, rp, en, sink_len)
        kept = oracle.sparvar_select(A, ns, tau)
        ref = oracle.sparvar_keep_mask(sides, d, k_step, units, kept, sink)
        assert np.array_equal(got, ref.astype(bool)), tau
        for qb in range(len(rp) - 1):                   # sorted, unique rows
            row = en[rp[qb]:rp[qb + 1]]
            assert np.all(np.diff(row) > 0)


def test_sparvar_rejects_bad_arguments():
    sides = (1, 2, 4, 6, 8, 12, 16, 20, 24, 32, 40, 48, 64)
    p = V.problem(2, 16, 128, sides)
    A = np.full((16, 43), 1.0 / 43)
    with pytest.raises(V.VarError):
        V.var_sparvar_units(p, 7, 16)                   # side 20 is not a multiple of 8
    with pytest.raises(V.VarError):
        V.var_sparvar_units(p, 6, 16)                   # side 16 is a sink scale
    with pytest.raises(V.VarError):
        V.var_sparvar_mask_build(p, 9, 8, 16, A, 0.5)   # target before the decision step
    with pytest.raises(V.VarError):
        V.var_sparvar_mask_build(p, 9, 12, 16, A, 1.5)  # tau outside [0, 1]
    q = V.problem(2, 16, 128, (1, 2, 4, 8, 16, 24, 36))
    with pytest.raises(V.VarError):
        V.var_sparvar_mask_build(q, 5, 6, 4, np.full((9, 15), 1 / 15), 0.5)   # target side 36
    L = V.lib()
    f = _fake()
    assert L.var_sparvar_workspace_bytes(None, 9, 16) == 0
    assert L.var_sparvar_workspace_bytes(C.byref(p), 7, 16) == 0              # side 20
    ws = L.var_sparvar_workspace_bytes(C.byref(p), 9, 16)
    assert ws > 0
    sc = V.lib().var_sparvar_scores
    assert sc(C.byref(p), 9, 16, 0.5, 0, None, None, None, 0, None, None, None) == V.VAR_ERR_INVALID_ARG
    assert sc(C.byref(p), 9, 16, 1.5, 0, f, f, f, ws, f, None, None) == V.VAR_ERR_INVALID_ARG     # tau
    assert sc(C.byref(p), 9, 16, -0.1, 0, f, f, f, ws, f, None, None) == V.VAR_ERR_INVALID_ARG
    assert sc(C.byref(p), 9, 16, 0.5, 2, f, f, f, ws, f, None, None) == V.VAR_ERR_INVALID_ARG     # flags
    assert sc(C.byref(p), 9, 16, 0.5, 0, f, f, f, ws - 1, f, None, None) == V.VAR_ERR_WORKSPACE
    assert sc(C.byref(p), 9, 16, 0.5, 0, f, f, C.c_void_p(0x10010), ws, f, None, None) == V.VAR_ERR_UNSUPPORTED
    big = V.problem(2, 16, 128, (1, 2, 4, 8, 16, 32, 64, 96, 128, 160))     # 6 + 16 + 64 + 144 + 256 + 400 units
    assert sc(C.byref(big), 9, 16, 0.5, 0, f, f, f, 1 << 40, f, None, None) == V.VAR_ERR_UNSUPPORTED
    fast = V.lib().var_sparvar_scores_fast
    assert fast(C.byref(p), 9, 16, f, f, None, f, ws, f, None) == V.VAR_ERR_INVALID_ARG          # no lse
    assert fast(C.byref(p), 9, 16, f, f, f, f, ws - 1, f, None) == V.VAR_ERR_WORKSPACE
    assert fast(C.byref(p), 9, 16, f, f, C.c_void_p(0x10002), f, ws, f, None) == V.VAR_ERR_UNSUPPORTED
    assert fast(C.byref(p), 7, 16, f, f, f, f, 1 << 40, f, None) == V.VAR_ERR_UNSUPPORTED       # side 20
    wide = V.problem(2, 16, 128, (1, 2, 4, 8, 16, 32, 64, 72))                # 81 query blocks at side 72
    assert fast(C.byref(wide), 7, 16, f, f, f, f, 1 << 40, f, None) == V.VAR_ERR_UNSUPPORTED


def test_selftest_wait_timeout_rejects_bad_limits():
    L = V.lib()
    assert L.var_selftest_wait_timeout(0, None, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_selftest_wait_timeout(10000001, None, None) == V.VAR_ERR_INVALID_ARG


def test_workspace_bytes_is_the_pivot_scratch():
    p = V.problem(2, 16, 128, SCHEDULE_1024)
    assert V.var_workspace_bytes(p, 12, 2048, 819) == V.var_pivot_workspace_bytes(p, 12, 2048) > 0
    assert V.var_workspace_bytes(p, 12, 2048, 4097) == 0       # keep_k above N
    assert V.var_workspace_bytes(p, 12, 2048, -1) == 0


def test_noalloc_pivot_rejects_what_the_workspace_version_rejects():
    """var_pivot_select_noalloc runs the same argument checks, in the same order,
    as var_pivot_select; only then come the limits of its static scratch."""
    L = V.lib()
    f = _fake()
    good = dict(b=2, h=16, d=128, sides=SCHEDULE_1024, cap=0, scale=0.0)
    cases = [
        (dict(), 12, f, 2048, 819, f),                      # valid: both fail only later (workspace / device)
        (dict(d=96), 12, f, 2048, 819, f),                  # head_dim
        (dict(h=0), 12, f, 2048, 819, f),                   # heads
        (dict(), 13, f, 2048, 819, f),                      # step past the schedule
        (dict(), -1, f, 2048, 819, f),
        (dict(cap=100), 12, f, 2048, 819, f),               # kv_capacity < L
        (dict(scale=-1.0), 12, f, 2048, 819, f),            # softmax scale
        (dict(), 12, None, 2048, 819, f),                   # null x
        (dict(), 12, f, 2040, 819, f),                      # channels not a multiple of 32
        (dict(), 12, f, 0, 819, f),
        (dict(), 12, f, 2048, 4097, f),                     # keep_k > N
        (dict(), 12, f, 2048, -1, f),
        (dict(), 12, f, 2048, 819, None),                   # idx null with keep_k > 0
        (dict(), 12, C.c_void_p(0x10008), 2048, 819, f),    # misaligned x
    ]
    for over, step, x, ch, k, idx in cases[1:]:
        a = dict(good, **over)
        p = V.problem(a["b"], a["h"], a["d"], a["sides"], kv_capacity=a["cap"], softmax_scale=a["scale"])
        ws = L.var_pivot_workspace_bytes(C.byref(V.problem(2, 16, 128, SCHEDULE_1024)), 12, 2048)
        want = L.var_pivot_select(C.byref(p), step, x, ch, k, idx, None, f, ws, None)
        got = L.var_pivot_select_noalloc(C.byref(p), step, x, ch, k, idx, None, None)
        assert want not in (V.VAR_OK, V.VAR_ERR_WORKSPACE, V.VAR_ERR_CUDA), (over, step, ch, k, want)
        assert got == want, (over, step, ch, k, got, want)
    # beyond the static scratch: batch 8, channels 8192 -- after the common checks pass
    p8 = V.problem(8, 1, 128, (1, 16))
    assert L.var_pivot_select_noalloc(C.byref(p8), 1, f, 64, 4, f, None, None) == V.VAR_ERR_WORKSPACE
    p1 = V.problem(1, 1, 128, (1, 16))
    assert L.var_pivot_select_noalloc(C.byref(p1), 1, f, 8192, 4, f, None, None) == V.VAR_ERR_WORKSPACE
    assert L.var_pivot_select_noalloc(C.byref(p1), 1, f, 8192, 4, None, None, None) == V.VAR_ERR_INVALID_ARG


def test_status_word_must_be_aligned():
    L = V.lib()
    f = _fake()
    p = V.problem(1, 2, 64, SCHEDULE_256)
    p.status = 0x10002
    assert L.var_attn_dense(C.byref(p), 9, f, f, f, f, None) == V.VAR_ERR_INVALID_ARG
    out = C.c_int32()
    assert L.var_check_status(C.c_void_p(0x10002), C.byref(out), 0, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_check_status(f, None, 0, None) == V.VAR_ERR_INVALID_ARG
    assert L.var_selftest_wait_timeout(100, C.c_void_p(0x10002), None) == V.VAR_ERR_INVALID_ARG
