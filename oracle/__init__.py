"""CPU oracle for the next-scale VAR attention hot path (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  It wraps the plain fp64 C loops of
``varattn_oracle.c`` (see that file's header for the passages each function
follows and the readings taken where the pages are silent) and shares no code
with the CUDA library.

Every function takes the exact bf16 tensors the GPU reads and returns fp64
results (indices as int32).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

MAX_SCALES = 32


class MaskSpec(C.Structure):
    _fields_ = [("n_scales", C.c_int32), ("side", C.c_int32 * MAX_SCALES), ("step", C.c_int32),
                ("qblock_side", C.c_int32), ("radius", C.c_int32), ("sink_max_side", C.c_int32)]


def mask_spec(sides: Sequence[int], step: int, qblock_side: int, radius: int,
              sink_max_side: int) -> MaskSpec:
    m = MaskSpec()
    m.n_scales = len(sides)
    for i, s in enumerate(sides):
        m.side[i] = s
    m.step, m.qblock_side, m.radius, m.sink_max_side = step, qblock_side, radius, sink_max_side
    return m


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        L.oracle_attention.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                       C.c_double, P, P, P, C.c_long, P, P, P]
        L.oracle_block_mask_rows.argtypes = [P, C.c_int, C.c_int, P]
        L.oracle_pivot_mean.argtypes = [C.c_int, C.c_int, C.c_int, P, P]
        L.oracle_pivot_scores.argtypes = [C.c_int, C.c_int, C.c_int, P, P, P]
        L.oracle_pivot_select.argtypes = [C.c_int, C.c_int, C.c_int, P, C.c_int, P, P]
        L.oracle_restore_scatter.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, P, P,
                                             P, C.c_int, P]
        L.oracle_attention_lse.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                           C.c_double, P, P, P]
        L.oracle_saliency.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                      C.c_double, P, P, P]
        L.oracle_unit_mass.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                        C.c_double, P, P, P, C.c_int, P]
        L.oracle_attention_keep.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                            C.c_double, P, P, P, P, P]
        L.oracle_num_threads.restype = C.c_int
        L.oracle_num_threads.argtypes = []
        for f in ("oracle_attention", "oracle_block_mask_rows", "oracle_pivot_mean",
                  "oracle_pivot_scores", "oracle_pivot_select", "oracle_restore_scatter",
                  "oracle_attention_lse", "oracle_saliency", "oracle_unit_mass", "oracle_attention_keep"):
            getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def num_threads() -> int:
    """Threads the oracle's parallel loops use."""
    return int(lib().oracle_num_threads())


def _bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> contiguous uint16 bit array (CPU)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, L: int,
              scale: Optional[float] = None, rows: Optional[np.ndarray] = None,
              mask: Optional[MaskSpec] = None) -> np.ndarray:
    """Softmax attention of q [B,H,N,D] over the first L rows of k, v [B,H,cap,D].

    rows: optional flat query ids ((b*H + h)*N + i); returns [len(rows), D] then,
    else [B, H, N, D].  mask: optional block-sparse rule.
    """
    B, H, N, D = q.shape
    cap = k.shape[2]
    assert k.shape == (B, H, cap, D) and v.shape == k.shape and cap >= L
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((len(rows), D), dtype=np.float64)
        n = len(rows)
    else:
        out = np.zeros((B, H, N, D), dtype=np.float64)
        n = 0
    rc = lib().oracle_attention(B, H, N, L, cap, D, scale, _ptr(qb), _ptr(kb), _ptr(vb), n,
                                _ptr(rows), None if mask is None else C.byref(mask), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_attention failed ({rc})")
    return out


def attention_lse(q: torch.Tensor, k: torch.Tensor, L: int, scale: Optional[float] = None) -> np.ndarray:
    """Row log2-sum-exp of the scaled scores over the first L keys: [B, H, N] fp64,
    so that the attention probability is 2^(s_ij log2(e) - lse_i)."""
    B, H, N, D = q.shape
    cap = k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.zeros((B, H, N), dtype=np.float64)
    if lib().oracle_attention_lse(B, H, N, L, cap, D, scale, _ptr(_bits(q)), _ptr(_bits(k)), _ptr(out)) != 0:
        raise ValueError("oracle_attention_lse failed")
    return out


def saliency(q_src: torch.Tensor, k: torch.Tensor, L_src: int, scale: Optional[float] = None) -> np.ndarray:
    """ARVAR attention retrospect: for each (b, h) and token j of the source grid
    (key L_src - N' + j, the source step's own scale), the attention probability
    it receives summed over the N' source queries: [B, H, N'] fp64."""
    B, H, N, D = q_src.shape
    cap = k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.zeros((B, H, N), dtype=np.float64)
    if lib().oracle_saliency(B, H, N, L_src, cap, D, scale, _ptr(_bits(q_src)), _ptr(_bits(k)), _ptr(out)) != 0:
        raise ValueError("oracle_saliency failed")
    return out


def bilinear_map(m: np.ndarray, side: int) -> np.ndarray:
    """Bilinear upsampling of [..., sp*sp] maps to [..., side*side] in fp64: half-pixel
    centres, edge clamp, no antialias (the restore's convention)."""
    sp = int(round(m.shape[-1] ** 0.5))
    assert sp * sp == m.shape[-1]

    def axis(n_out):
        dst = np.arange(n_out, dtype=np.float64)
        src = np.maximum((dst + 0.5) * sp / n_out - 0.5, 0.0)
        i0 = np.minimum(np.floor(src).astype(np.int64), sp - 1)
        i1 = np.minimum(i0 + 1, sp - 1)
        return i0, i1, src - i0

    y0, y1, ly = axis(side)
    x0, x1, lx = axis(side)
    g = m.reshape(m.shape[:-1] + (sp, sp))
    ly = ly[:, None]
    lx = lx[None, :]
    top = g[..., y0[:, None], x0[None, :]] * (1 - lx) + g[..., y0[:, None], x1[None, :]] * lx
    bot = g[..., y1[:, None], x0[None, :]] * (1 - lx) + g[..., y1[:, None], x1[None, :]] * lx
    return (top * (1 - ly) + bot * ly).reshape(m.shape[:-1] + (side * side,))


def top_k_ascending(values: np.ndarray, keep_k: int) -> np.ndarray:
    """Per row of [B, N]: the keep_k largest (equal values: lower index first), ascending."""
    B, N = values.shape
    out = np.zeros((B, keep_k), dtype=np.int32)
    for b in range(B):
        order = sorted(range(N), key=lambda i: (-values[b, i], i))
        out[b] = np.sort(np.array(order[:keep_k], dtype=np.int32))
    return out


def guided_pivot(sal: np.ndarray, side: int, keep_k: int):
    """ARVAR attention-guided pivots: the head and query mean of the per-head
    saliency sums [B, H, N'], bilinearly upsampled to side x side, Top-K.
    The heads are added one at a time in order, in fp64 (a fixed order, so the
    rounding is defined), then divided by H N'.
    Returns (idx [B, K] ascending, values [B, side*side])."""
    B, H, Np = sal.shape
    acc = np.zeros((B, Np), dtype=np.float64)
    for h in range(H):
        acc += sal[:, h, :]
    v = bilinear_map(acc / (H * Np), side)
    return top_k_ascending(v, keep_k), v


def branch_halved_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, L: int,
                            scale: Optional[float] = None) -> np.ndarray:
    """Branch Halving ("ARVAR" Key Design 1): only the conditional branch -- the
    first half of the batch, the classifier-free-guidance pair concatenated along
    the batch -- is computed; its output is repeated into the second half.
    Returns [B, H, N, D] fp64."""
    B = q.shape[0]
    assert B % 2 == 0
    h = B // 2
    cond = attention(q[:h].contiguous(), k[:h].contiguous(), v[:h].contiguous(), L, scale=scale)
    return np.concatenate([cond, cond], axis=0)


# ----------------------------------------------------------------------------- dynamic pattern
# SparVAR (abstract): the sparse attention pattern of later high-resolution
# scales is predicted from a sparse decision scale and carried to them by index
# mapping, giving scale self-similar sparse attention.  The pages fix no score,
# threshold or mapping formula; the reading implemented here:
#   units     the decision step's keys in 64-key units: the sink range (leading
#             scales with side <= sink_max_side) in 64-token chunks, then every
#             8x8 key block of each later scale up to the decision scale;
#   score     A[qb, u]: the attention mass unit u receives, averaged over the 64
#             queries of the decision step's 8x8 query block qb, its heads and
#             batch elements (one pattern, as the block mask is one for all);
#   select    per qb the sinks, then the other units by score (equal scores:
#             lower unit first) until the kept mass reaches tau of the total;
#   map       a target step's query block takes the decision block under its
#             centre; kept blocks of scales below the decision scale are kept
#             as they are, kept blocks of the decision scale are kept and also
#             mapped into every later scale up to the target, to the blocks
#             that meet the rescaled block (rounded outward).


def sparvar_units(sides: Sequence[int], d: int, sink_max_side: int):
    """The decision step's key units: (unit_of_key int32[L_d], units, n_sink).
    units[u] = ("sink", c) for tokens [64c, 64c + 64) of the sink range, or
    (scale, u, v) for key block (u, v) of that scale (rows 8u.., cols 8v..)."""
    sink_len = 0
    sc = 0
    while sc <= d and sides[sc] <= sink_max_side:
        sink_len += sides[sc] ** 2
        sc += 1
    L = sum(sides[i] ** 2 for i in range(d + 1))
    unit_of = np.zeros(L, dtype=np.int32)
    units = []
    for c in range((sink_len + 63) // 64):
        unit_of[64 * c:min(64 * c + 64, sink_len)] = len(units)
        units.append(("sink", c))
    n_sink = len(units)
    off = sink_len
    for scale in range(sc, d + 1):
        s = sides[scale]
        nbs = (s + 7) // 8
        for u in range(nbs):
            for v in range(nbs):
                for r in range(8 * u, min(8 * u + 8, s)):
                    unit_of[off + r * s + 8 * v:off + r * s + min(8 * v + 8, s)] = len(units)
                units.append((scale, u, v))
        off += s * s
    return unit_of, units, n_sink


def sparvar_scores(q_d: torch.Tensor, k: torch.Tensor, sides: Sequence[int], d: int, sink_max_side: int,
                   scale: Optional[float] = None) -> np.ndarray:
    """A[qb, u] fp64: unit u's attention mass averaged over the 64 queries of the
    decision step's 8x8 query block qb (row-major blocks), heads and batch: the
    sum over (b, h, y, x) in that order, divided by B * H * 64."""
    B, H, N, D = q_d.shape
    s_d = sides[d]
    assert N == s_d * s_d and s_d % 8 == 0
    unit_of, units, _ = sparvar_units(sides, d, sink_max_side)
    L = len(unit_of)
    U = len(units)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    mass = np.zeros((B, H, N, U), dtype=np.float64)
    if lib().oracle_unit_mass(B, H, N, L, k.shape[2], D, scale, _ptr(_bits(q_d)), _ptr(_bits(k)),
                              _ptr(unit_of), U, _ptr(mass)) != 0:
        raise ValueError("oracle_unit_mass failed")
    nb = s_d // 8
    g = mass.reshape(B, H, nb, 8, nb, 8, U)            # [b, h, by, y, bx, x, u]
    # The per-query masses of a block are added one at a time in the order
    # (b, h, y, x), starting from 0, in fp64: a fixed order, so the rounding
    # of the sum is defined (the pages fix none).
    acc = np.zeros((nb, nb, U), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for y in range(8):
                for x in range(8):
                    acc += g[b, h, :, y, :, x, :]
    return acc.reshape(nb * nb, U) / (B * H * 64)


def sparvar_select(A: np.ndarray, n_sink: int, tau: float):
    """Per decision query block: the kept non-sink unit indices (ascending).  The
    sinks are always kept; the other units are taken by decreasing score (equal
    scores: lower unit first) until the kept mass reaches tau of the row total.
    Masses are added in fp64 in that order."""
    kept = []
    for row in A:
        total = 0.0
        for x in row:
            total += float(x)
        have = 0.0
        for u in range(n_sink):
            have += float(row[u])
        order = sorted(range(n_sink, len(row)), key=lambda u: (-float(row[u]), u))
        take = []
        for u in order:
            if have >= tau * total:
                break
            take.append(u)
            have += float(row[u])
        kept.append(sorted(take))
    return kept


def sparvar_keep_mask(sides: Sequence[int], d: int, k_step: int, units, kept, sink_max_side: int) -> np.ndarray:
    """Token-level keep mask [N_k, L_k] (uint8) of the target step k >= d, built
    from the definition: per target query token, its 8x8 block, the decision
    block under that block's centre, and the keys its kept units cover there."""
    s_d, s_k = sides[d], sides[k_step]
    nb_d, nb_k = s_d // 8, s_k // 8
    offs = np.cumsum([0] + [s * s for s in sides[:k_step + 1]])
    L = int(offs[-1])
    sink_len = 0
    sc = 0
    while sc <= k_step and sides[sc] <= sink_max_side:
        sink_len += sides[sc] ** 2
        sc += 1
    block_keys = np.zeros((nb_d * nb_d, L), dtype=np.uint8)   # keys kept by each decision block
    for qb, lst in enumerate(kept):
        row = block_keys[qb]
        row[:sink_len] = 1
        for u_idx in lst:
            scale, u, v = units[u_idx]
            targets = [(scale, u, v)] if scale < d else []
            if scale == d:
                for sc2 in range(d, k_step + 1):
                    s2 = sides[sc2]
                    # rows of the decision block [8u, 8u+8) clipped, rescaled to s2, outward
                    r0, r1 = 8 * u, min(8 * u + 8, s_d)
                    c0, c1 = 8 * v, min(8 * v + 8, s_d)
                    lo_r, hi_r = (r0 * s2) // s_d, -((-r1 * s2) // s_d)
                    lo_c, hi_c = (c0 * s2) // s_d, -((-c1 * s2) // s_d)
                    for uu in range((s2 + 7) // 8):
                        if not (8 * uu < hi_r and lo_r < min(8 * uu + 8, s2)):
                            continue
                        for vv in range((s2 + 7) // 8):
                            if 8 * vv < hi_c and lo_c < min(8 * vv + 8, s2):
                                targets.append((sc2, uu, vv))
            for (sc2, uu, vv) in targets:
                s2 = sides[sc2]
                for r in range(8 * uu, min(8 * uu + 8, s2)):
                    a = offs[sc2] + r * s2
                    row[a + 8 * vv:a + min(8 * vv + 8, s2)] = 1
    keep = np.zeros((s_k * s_k, L), dtype=np.uint8)
    for y in range(s_k):
        for x in range(s_k):
            by, bx = y // 8, x // 8
            dy = ((2 * by + 1) * nb_d) // (2 * nb_k)
            dx = ((2 * bx + 1) * nb_d) // (2 * nb_k)
            keep[y * s_k + x] = block_keys[dy * nb_d + dx]
    return keep


def attention_keep(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, L: int, keep: np.ndarray,
                   scale: Optional[float] = None) -> np.ndarray:
    """Attention of q [B,H,N,D] over the first L keys, query i keeping key j iff
    keep[i, j] (one mask for every (b, h)); [B, H, N, D] fp64."""
    B, H, N, D = q.shape
    keep = np.ascontiguousarray(keep, dtype=np.uint8)
    assert keep.shape == (N, L)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.zeros((B, H, N, D), dtype=np.float64)
    if lib().oracle_attention_keep(B, H, N, L, k.shape[2], D, scale, _ptr(_bits(q)), _ptr(_bits(k)),
                                   _ptr(_bits(v)), _ptr(keep), _ptr(out)) != 0:
        raise ValueError("oracle_attention_keep failed")
    return out


def block_mask_rows(m: MaskSpec, q0: int, q1: int) -> np.ndarray:
    """Token-level keep mask [q1-q0, L] (uint8) of the block-sparse rule."""
    L = sum(m.side[i] ** 2 for i in range(m.step + 1))
    out = np.zeros((q1 - q0, L), dtype=np.uint8)
    if lib().oracle_block_mask_rows(C.byref(m), q0, q1, _ptr(out)) != 0:
        raise ValueError("oracle_block_mask_rows failed")
    return out


def pivot_mean(x: torch.Tensor) -> np.ndarray:
    B, N, Ch = x.shape
    out = np.zeros((B, Ch), dtype=np.float64)
    if lib().oracle_pivot_mean(B, N, Ch, _ptr(_bits(x)), _ptr(out)) != 0:
        raise ValueError("oracle_pivot_mean failed")
    return out


def pivot_scores(x: torch.Tensor) -> np.ndarray:
    B, N, Ch = x.shape
    mean = pivot_mean(x)
    out = np.zeros((B, N), dtype=np.float64)
    if lib().oracle_pivot_scores(B, N, Ch, _ptr(_bits(x)), _ptr(mean), _ptr(out)) != 0:
        raise ValueError("oracle_pivot_scores failed")
    return out


def pivot_select(x: torch.Tensor, keep_k: int):
    """Return (idx [B, K] int32 ascending, scores [B, N] fp64)."""
    B, N, Ch = x.shape
    idx = np.zeros((B, keep_k), dtype=np.int32)
    sc = np.zeros((B, N), dtype=np.float64)
    if lib().oracle_pivot_select(B, N, Ch, _ptr(_bits(x)), keep_k, _ptr(idx), _ptr(sc)) != 0:
        raise ValueError("oracle_pivot_select failed")
    return idx, sc


def restore_scatter(prev: torch.Tensor, oc: torch.Tensor, idx: np.ndarray, side: int) -> np.ndarray:
    """Bilinear Up(prev) to side x side, then overwrite rows idx with oc.

    prev [B,H,sp*sp,D], oc [B,H,K,D] bf16; idx [B,K] int32 ascending.
    Returns [B,H,side*side,D] fp64.
    """
    B, H, Np, D = prev.shape
    sp = int(round(Np ** 0.5))
    assert sp * sp == Np
    K = oc.shape[2]
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(B, K)
    out = np.zeros((B, H, side * side, D), dtype=np.float64)
    rc = lib().oracle_restore_scatter(B, H, sp, side, D, _ptr(_bits(prev)), _ptr(_bits(oc)),
                                      _ptr(idx), K, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_restore_scatter failed ({rc})")
    return out
