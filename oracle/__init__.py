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
        L.oracle_num_threads.restype = C.c_int
        L.oracle_num_threads.argtypes = []
        for f in ("oracle_attention", "oracle_block_mask_rows", "oracle_pivot_mean",
                  "oracle_pivot_scores", "oracle_pivot_select", "oracle_restore_scatter",
                  "oracle_attention_lse", "oracle_saliency"):
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
    Returns (idx [B, K] ascending, values [B, side*side])."""
    B, H, Np = sal.shape
    v = bilinear_map(sal.sum(axis=1) / (H * Np), side)
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
