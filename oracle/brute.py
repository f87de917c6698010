"""Brute-force NumPy checks of the C oracle on tiny inputs (TEST INFRASTRUCTURE).

A second, independent formulation of each function: attention with the whole
probability matrix materialised; the block mask built from sets of covered key
rows instead of interval tests; pivot ranking with exact rational arithmetic;
bilinear upsampling written as a separable interpolation matrix.  Used only to
pin the C oracle (``varattn_oracle.c``) in the CPU test-suite.
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Sequence

import numpy as np


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
              keep: np.ndarray = None) -> np.ndarray:
    """q [N,D], k/v [L,D] (fp64); keep [N,L] bool or None -> [N,D]."""
    s = (q @ k.T) * scale
    if keep is not None:
        s = np.where(keep, s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ v


def block_mask(sides: Sequence[int], step: int, qbs: int, radius: int, sink_max_side: int) -> np.ndarray:
    """Token mask [N, L] from covered-row sets: for each query block and key scale,
    collect the key rows (and columns) the rescaled window touches, widen them to
    whole key blocks, and keep the cross product."""
    sq = sides[step]
    L = sum(s * s for s in sides[: step + 1])
    N = sq * sq
    out = np.zeros((N, L), dtype=bool)
    nb = (sq + qbs - 1) // qbs

    def covered(qb: int, s: int) -> set:
        lo = max(0, qbs * (qb - radius))
        hi = min(sq, qbs * (qb + radius + 1))
        rows = set()
        # key row t of scale s spans [t*sq/s, (t+1)*sq/s) in query coordinates;
        # the window touches it when that span meets [lo, hi)
        for t in range(s):
            a = Fraction(t * sq, s)
            b = Fraction((t + 1) * sq, s)
            if a < hi and lo < b:
                rows.add(t)
        blocks = {t // qbs for t in rows}
        return {t for t in range(s) if t // qbs in blocks}

    for by in range(nb):
        for bx in range(nb):
            qrows = [y * sq + x for y in range(by * qbs, min(sq, by * qbs + qbs))
                     for x in range(bx * qbs, min(sq, bx * qbs + qbs))]
            off = 0
            keys: List[int] = []
            for s in sides[: step + 1]:
                if s <= sink_max_side:
                    keys.extend(range(off, off + s * s))
                else:
                    ry = covered(by, s)
                    rx = covered(bx, s)
                    keys.extend(off + r * s + c for r in sorted(ry) for c in sorted(rx))
                off += s * s
            for qi in qrows:
                out[qi, keys] = True
    return out


def pivot_ranking_exact(x: np.ndarray, keep_k: int) -> List[int]:
    """x [N,C] of exactly representable values (fp64 holding bf16 values).
    Exact rational scores; K largest, ties to the lower index; ascending."""
    N, Cc = x.shape
    xs = [[Fraction(float(x[i, c])) for c in range(Cc)] for i in range(N)]
    mean = [sum(xs[i][c] for i in range(N)) / N for c in range(Cc)]
    score = [sum((xs[i][c] - mean[c]) ** 2 for c in range(Cc)) for i in range(N)]
    order = sorted(range(N), key=lambda i: (-score[i], i))
    return sorted(order[:keep_k])


def upsample_matrix(sp: int, s: int) -> np.ndarray:
    """[s, sp] linear interpolation matrix, half-pixel centres, edge clamp."""
    M = np.zeros((s, sp))
    for d in range(s):
        src = max((d + 0.5) * sp / s - 0.5, 0.0)
        i0 = min(int(np.floor(src)), sp - 1)
        i1 = min(i0 + 1, sp - 1)
        lam = src - i0
        M[d, i0] += 1 - lam
        M[d, i1] += lam
    return M


def restore_scatter(prev: np.ndarray, oc: np.ndarray, idx: np.ndarray, s: int) -> np.ndarray:
    """prev [Np, D] (sp x sp grid), oc [K, D], idx [K] -> [s*s, D]."""
    Np, D = prev.shape
    sp = int(round(Np ** 0.5))
    M = upsample_matrix(sp, s)
    g = prev.reshape(sp, sp, D)
    up = np.einsum("ya,xb,abd->yxd", M, M, g).reshape(s * s, D)
    up[idx] = oc
    return up
