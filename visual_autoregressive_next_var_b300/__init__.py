"""Python binding of libvarattn (include/varattn.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: tensors are passed as device pointers, the stream is
torch's current CUDA stream unless one is given, and a non-zero status raises
``VarError``.  PyTorch is used only to own device memory and streams.

Importing this module loads the shared library and fails loudly if it is
missing; run ``python visual_autoregressive_next_var_b300/build.py`` (or
``__graft_entry__.build()``) first.
"""
from __future__ import annotations

import ctypes as C
import os
import re
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# VARATTN_DEBUG=1 loads the debug build (device-side input checks, see build.py --debug)
LIB_PATH = os.path.join(_HERE, "libvarattn_debug.so" if os.environ.get("VARATTN_DEBUG") == "1" else "libvarattn.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "varattn.h")
TEST_HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "varattn_test.h")
MAX_SCALES = 32

VAR_OK = 0
VAR_ERR_INVALID_ARG = 1
VAR_ERR_UNSUPPORTED = 2
VAR_ERR_CUDA = 3
VAR_ERR_TIMEOUT = 4
VAR_ERR_NUMERIC = 5
VAR_ERR_WORKSPACE = 6


class VarError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({var_status_string(status)})")
        self.status = status


class var_problem(C.Structure):
    _fields_ = [("batch", C.c_int32), ("heads", C.c_int32), ("head_dim", C.c_int32),
                ("n_scales", C.c_int32), ("side", C.c_int32 * MAX_SCALES),
                ("kv_capacity", C.c_int32), ("softmax_scale", C.c_float), ("status", C.c_void_p)]


class var_block_mask(C.Structure):
    _fields_ = [("qblock_side", C.c_int32), ("n_qblocks", C.c_int32), ("sink_len", C.c_int32),
                ("nnz", C.c_int32), ("row_ptr", C.c_void_p), ("entries", C.c_void_p),
                ("n_squares", C.c_int32), ("plan_units", C.c_int32), ("sq_ptr", C.c_void_p),
                ("sq_units", C.c_void_p), ("sq_order", C.c_void_p)]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                      "(python visual_autoregressive_next_var_b300/build.py [--debug])")
_lib = C.CDLL(LIB_PATH)

_P = C.c_void_p
_PROB = C.POINTER(var_problem)
_SIGS = {
    "var_attn_dense": (C.c_int, [_PROB, C.c_int32, _P, _P, _P, _P, _P]),
    "var_pivot_workspace_bytes": (C.c_size_t, [_PROB, C.c_int32, C.c_int32]),
    "var_pivot_select": (C.c_int, [_PROB, C.c_int32, _P, C.c_int32, C.c_int32, _P, _P, _P,
                                   C.c_size_t, _P]),
    "var_pivot_select_noalloc": (C.c_int, [_PROB, C.c_int32, _P, C.c_int32, C.c_int32, _P, _P, _P]),
    "var_attn_pruned": (C.c_int, [_PROB, C.c_int32, _P, _P, _P, _P, C.c_int32, _P, _P]),
    "var_restore_scatter": (C.c_int, [_PROB, C.c_int32, _P, _P, _P, C.c_int32, _P, _P]),
    "var_attn_pruned_scatter": (C.c_int, [_PROB, C.c_int32, _P, _P, _P, _P, C.c_int32, _P, _P]),
    "var_restore_fill": (C.c_int, [_PROB, C.c_int32, _P, _P, C.c_int32, _P, _P]),
    "var_pruned_in_place": (C.c_int, [_PROB, C.c_int32, _P, _P, _P, _P, _P, C.c_int32, _P, _P]),
    "var_pruned_step": (C.c_int, [_PROB, C.c_int32, _P, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P, _P,
                                  C.c_size_t, _P]),
    "var_attn_dense_halved": (C.c_int, [_PROB, C.c_int32, _P, _P, _P, _P, _P]),
    "var_guided_pivot_exact_workspace_bytes": (C.c_size_t, [_PROB, C.c_int32, C.c_int32]),
    "var_guided_pivot_select_exact": (C.c_int, [_PROB, C.c_int32, C.c_int32, _P, _P, C.c_int32, _P, _P, _P,
                                                C.c_size_t, _P]),
    "var_attn_dense_lse": (C.c_int, [_PROB, C.c_int32, _P, _P, _P, _P, _P, _P]),
    "var_attn_saliency": (C.c_int, [_PROB, C.c_int32, _P, _P, _P, _P, _P]),
    "var_guided_pivot_workspace_bytes": (C.c_size_t, [_PROB, C.c_int32]),
    "var_guided_pivot_select": (C.c_int, [_PROB, C.c_int32, C.c_int32, _P, C.c_int32, _P, _P, _P, C.c_size_t,
                                          _P]),
    "var_block_mask_build": (C.c_int, [_PROB, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _P, _P,
                                       C.c_int32, _P, _P, _P]),
    "var_block_mask_plan": (C.c_int, [_PROB, C.c_int32, C.c_int32, _P, _P, C.c_int32, _P, _P, C.c_int32, _P,
                                      _P, _P]),
    "var_attn_blocksparse": (C.c_int, [_PROB, C.c_int32, _P, _P, _P,
                                       C.POINTER(var_block_mask), _P, _P]),
    "var_sparvar_units": (C.c_int, [_PROB, C.c_int32, C.c_int32, _P, _P]),
    "var_sparvar_workspace_bytes": (C.c_size_t, [_PROB, C.c_int32, C.c_int32]),
    "var_sparvar_scores": (C.c_int, [_PROB, C.c_int32, C.c_int32, C.c_double, C.c_int32, _P, _P, _P, C.c_size_t,
                                     _P, _P, _P]),
    "var_sparvar_scores_fast": (C.c_int, [_PROB, C.c_int32, C.c_int32, _P, _P, _P, _P, C.c_size_t, _P, _P]),
    "var_sparvar_mask_build": (C.c_int, [_PROB, C.c_int32, C.c_int32, C.c_int32, _P, C.c_double, _P, _P,
                                         C.c_int32, _P, _P, _P]),
    "var_selftest_wait_timeout": (C.c_int, [C.c_int32, _P, _P]),
    "var_check_status": (C.c_int, [_P, _P, C.c_int32, _P]),
    "var_test_mock_cuda": (C.c_int, [C.c_int32, C.c_int64]),
    "var_test_mock_calls": (C.c_int64, []),
    "var_workspace_bytes": (C.c_size_t, [_PROB, C.c_int32, C.c_int32, C.c_int32]),
    "var_keep_count": (C.c_int32, [C.c_int32, C.c_int32, C.c_int32]),
    "var_status_string": (C.c_char_p, [C.c_int]),
    "var_device_status": (C.c_int, [_P, C.c_int32]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def header_functions() -> Sequence[str]:
    """Names of the functions include/varattn.h and include/varattn_test.h declare."""
    names = []
    for path in (HEADER_PATH, TEST_HEADER_PATH):
        text = open(path).read()
        names += re.findall(r"^\s*VAR_API\s+(?:int|int32_t|int64_t|size_t|const char\*)\s+(var_\w+)\s*\(",
                            text, re.M)
    return names


def lib() -> C.CDLL:
    return _lib


def problem(batch: int, heads: int, head_dim: int, sides: Sequence[int], kv_capacity: int = 0,
            softmax_scale: float = 0.0, status: Optional[torch.Tensor] = None) -> var_problem:
    """The problem statement; `status`: an optional int32 device tensor whose first
    element is the calls' own status word (var_problem.status)."""
    p = var_problem()
    p.batch, p.heads, p.head_dim = batch, heads, head_dim
    p.n_scales = len(sides)
    for i, s in enumerate(sides):
        p.side[i] = s
    p.kv_capacity = kv_capacity
    p.softmax_scale = softmax_scale
    p.status = None if status is None else status.data_ptr()
    return p


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(name: str, rc: int) -> None:
    if rc != VAR_OK:
        raise VarError(name, rc)


def var_status_string(status: int) -> str:
    return _lib.var_status_string(status).decode()


def var_keep_count(n: int, num: int, den: int) -> int:
    return _lib.var_keep_count(n, num, den)


def var_device_status(clear: bool = True) -> int:
    out = C.c_int32(0)
    _check("var_device_status", _lib.var_device_status(C.byref(out), 1 if clear else 0))
    return out.value


def var_check_status(status: Optional[torch.Tensor], clear: bool = True, stream=None) -> int:
    """Read (and clear) a caller-owned status word (int32 device tensor; None = the
    per-device word) in the order of `stream`."""
    out = C.c_int32(0)
    _check("var_check_status", _lib.var_check_status(_ptr(status), C.byref(out), 1 if clear else 0,
                                                     _stream(stream)))
    return out.value


def var_attn_dense(p: var_problem, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                   o: torch.Tensor, stream=None) -> None:
    _check("var_attn_dense", _lib.var_attn_dense(C.byref(p), step, _ptr(q), _ptr(k), _ptr(v),
                                                 _ptr(o), _stream(stream)))


def var_pivot_workspace_bytes(p: var_problem, step: int, channels: int) -> int:
    return _lib.var_pivot_workspace_bytes(C.byref(p), step, channels)


def var_pivot_select(p: var_problem, step: int, x: torch.Tensor, keep_k: int, idx: torch.Tensor,
                     workspace: torch.Tensor, scores: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    channels = x.shape[-1]
    _check("var_pivot_select",
           _lib.var_pivot_select(C.byref(p), step, _ptr(x), channels, keep_k, _ptr(idx),
                                 _ptr(scores), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)))


def var_pivot_select_noalloc(p: var_problem, step: int, x: torch.Tensor, keep_k: int, idx: torch.Tensor,
                             scores: Optional[torch.Tensor] = None, stream=None) -> None:
    """var_pivot_select with the library's own static scratch (no workspace argument)."""
    channels = x.shape[-1]
    _check("var_pivot_select_noalloc",
           _lib.var_pivot_select_noalloc(C.byref(p), step, _ptr(x), channels, keep_k, _ptr(idx),
                                         _ptr(scores), _stream(stream)))


def var_attn_pruned(p: var_problem, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    idx: torch.Tensor, keep_k: int, o_compact: torch.Tensor, stream=None) -> None:
    _check("var_attn_pruned", _lib.var_attn_pruned(C.byref(p), step, _ptr(q), _ptr(k), _ptr(v),
                                                   _ptr(idx), keep_k, _ptr(o_compact),
                                                   _stream(stream)))


def var_attn_pruned_scatter(p: var_problem, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            idx: torch.Tensor, keep_k: int, out: torch.Tensor, stream=None) -> None:
    _check("var_attn_pruned_scatter",
           _lib.var_attn_pruned_scatter(C.byref(p), step, _ptr(q), _ptr(k), _ptr(v), _ptr(idx), keep_k,
                                        _ptr(out), _stream(stream)))


def var_restore_fill(p: var_problem, step: int, prev: torch.Tensor, idx: Optional[torch.Tensor], keep_k: int,
                     out: torch.Tensor, stream=None) -> None:
    _check("var_restore_fill",
           _lib.var_restore_fill(C.byref(p), step, _ptr(prev), _ptr(idx), keep_k, _ptr(out), _stream(stream)))


def var_pruned_in_place(p: var_problem, step: int, q: Optional[torch.Tensor], k: Optional[torch.Tensor],
                        v: Optional[torch.Tensor], prev: torch.Tensor, idx: Optional[torch.Tensor], keep_k: int,
                        out: torch.Tensor, stream=None) -> None:
    _check("var_pruned_in_place",
           _lib.var_pruned_in_place(C.byref(p), step, _ptr(q), _ptr(k), _ptr(v), _ptr(prev), _ptr(idx), keep_k,
                                    _ptr(out), _stream(stream)))


def var_pruned_step(p: var_problem, step: int, x: torch.Tensor, keep_k: int, q: Optional[torch.Tensor],
                    k: Optional[torch.Tensor], v: Optional[torch.Tensor], prev: torch.Tensor,
                    idx: Optional[torch.Tensor], out: torch.Tensor, workspace: Optional[torch.Tensor],
                    stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("var_pruned_step",
           _lib.var_pruned_step(C.byref(p), step, _ptr(x), x.shape[-1], keep_k, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(prev), _ptr(idx), _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)))


def var_attn_dense_halved(p: var_problem, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                          o: torch.Tensor, stream=None) -> None:
    _check("var_attn_dense_halved", _lib.var_attn_dense_halved(C.byref(p), step, _ptr(q), _ptr(k), _ptr(v),
                                                               _ptr(o), _stream(stream)))


def var_attn_dense_lse(p: var_problem, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       o: torch.Tensor, lse: torch.Tensor, stream=None) -> None:
    _check("var_attn_dense_lse", _lib.var_attn_dense_lse(C.byref(p), step, _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                         _ptr(lse), _stream(stream)))


def var_attn_saliency(p: var_problem, src_step: int, q_src: torch.Tensor, k: torch.Tensor, lse: torch.Tensor,
                      sal: torch.Tensor, stream=None) -> None:
    _check("var_attn_saliency", _lib.var_attn_saliency(C.byref(p), src_step, _ptr(q_src), _ptr(k), _ptr(lse),
                                                       _ptr(sal), _stream(stream)))


def var_guided_pivot_workspace_bytes(p: var_problem, step: int) -> int:
    return _lib.var_guided_pivot_workspace_bytes(C.byref(p), step)


def var_guided_pivot_select(p: var_problem, step: int, src_step: int, sal: torch.Tensor, keep_k: int,
                            idx: Optional[torch.Tensor], workspace: torch.Tensor,
                            scores: Optional[torch.Tensor] = None, stream=None) -> None:
    _check("var_guided_pivot_select",
           _lib.var_guided_pivot_select(C.byref(p), step, src_step, _ptr(sal), keep_k, _ptr(idx), _ptr(scores),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)))


def var_guided_pivot_exact_workspace_bytes(p: var_problem, step: int, src_step: int) -> int:
    return _lib.var_guided_pivot_exact_workspace_bytes(C.byref(p), step, src_step)


def var_guided_pivot_select_exact(p: var_problem, step: int, src_step: int, q_src: torch.Tensor, k: torch.Tensor,
                                  keep_k: int, idx: Optional[torch.Tensor], workspace: torch.Tensor,
                                  values: Optional[torch.Tensor] = None, stream=None) -> None:
    """Attention-guided pivots ranked on fp64 values evaluated in the definition's order."""
    _check("var_guided_pivot_select_exact",
           _lib.var_guided_pivot_select_exact(C.byref(p), step, src_step, _ptr(q_src), _ptr(k), keep_k, _ptr(idx),
                                              _ptr(values), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _stream(stream)))


def var_workspace_bytes(p: var_problem, step: int, channels: int, keep_k: int) -> int:
    """Device workspace bytes the path's calls need at `step` (pivot selection's scratch)."""
    return _lib.var_workspace_bytes(C.byref(p), step, channels, keep_k)


def var_selftest_wait_timeout(limit_us: int, status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Diagnostics: a kernel whose bounded wait gives up and records VAR_ERR_TIMEOUT
    in `status` (None = the per-device word)."""
    _check("var_selftest_wait_timeout", _lib.var_selftest_wait_timeout(limit_us, _ptr(status), _stream(stream)))


def var_sparvar_units(p: var_problem, decision_step: int, sink_max_side: int) -> Tuple[int, int]:
    """Host call: (U, n_sink) -- the decision step's 64-key units and how many are sink chunks."""
    u, ns = C.c_int32(), C.c_int32()
    _check("var_sparvar_units", _lib.var_sparvar_units(C.byref(p), decision_step, sink_max_side, C.byref(u),
                                                       C.byref(ns)))
    return u.value, ns.value


VAR_SPARVAR_RESCORE_ALL = 1


def var_sparvar_workspace_bytes(p: var_problem, decision_step: int, sink_max_side: int) -> int:
    return _lib.var_sparvar_workspace_bytes(C.byref(p), decision_step, sink_max_side)


def var_sparvar_scores(p: var_problem, decision_step: int, sink_max_side: int, tau: float, q: torch.Tensor,
                       k: torch.Tensor, workspace: torch.Tensor, scores: torch.Tensor,
                       rescored: Optional[torch.Tensor] = None, flags: int = 0, stream=None) -> None:
    """scores: device float64 [(side/8)^2, U], exact enough to decide the selection at tau;
    rescored: optional device int32 [(side/8)^2], 1 where a block was re-scored in fp64."""
    _check("var_sparvar_scores",
           _lib.var_sparvar_scores(C.byref(p), decision_step, sink_max_side, tau, flags, _ptr(q), _ptr(k),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(scores),
                                   _ptr(rescored), _stream(stream)))


def var_sparvar_scores_fast(p: var_problem, decision_step: int, sink_max_side: int, q: torch.Tensor,
                            k: torch.Tensor, lse: torch.Tensor, workspace: torch.Tensor, scores: torch.Tensor,
                            stream=None) -> None:
    """scores: device float64 [(side/8)^2, U] on the tensor cores from the decision step's
    row log2-sum-exp lse (device float32 [B, H, side^2], as var_attn_dense_lse writes it);
    deterministic fp32 masses with no error bound."""
    _check("var_sparvar_scores_fast",
           _lib.var_sparvar_scores_fast(C.byref(p), decision_step, sink_max_side, _ptr(q), _ptr(k), _ptr(lse),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(scores),
                                        _stream(stream)))


def var_sparvar_mask_build(p: var_problem, decision_step: int, step: int, sink_max_side: int,
                           scores: np.ndarray, tau: float) -> Tuple[np.ndarray, np.ndarray, int]:
    """Host call: the target step's block mask (row_ptr, entries, sink_len) from the
    decision step's scores (host float64 [(side_d/8)^2, U])."""
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    nnz, nqb, sink = C.c_int32(), C.c_int32(), C.c_int32()
    _check("var_sparvar_mask_build",
           _lib.var_sparvar_mask_build(C.byref(p), decision_step, step, sink_max_side, sc.ctypes.data, tau, None,
                                       None, 0, C.byref(nnz), C.byref(nqb), C.byref(sink)))
    row_ptr = np.zeros(nqb.value + 1, dtype=np.int32)
    entries = np.zeros(max(1, nnz.value), dtype=np.int32)
    _check("var_sparvar_mask_build",
           _lib.var_sparvar_mask_build(C.byref(p), decision_step, step, sink_max_side, sc.ctypes.data, tau,
                                       row_ptr.ctypes.data, entries.ctypes.data, entries.size, C.byref(nnz),
                                       C.byref(nqb), C.byref(sink)))
    return row_ptr, entries[: nnz.value], sink.value


def var_restore_scatter(p: var_problem, step: int, prev: torch.Tensor, o_compact: Optional[torch.Tensor],
                        idx: Optional[torch.Tensor], keep_k: int, out: torch.Tensor,
                        stream=None) -> None:
    _check("var_restore_scatter",
           _lib.var_restore_scatter(C.byref(p), step, _ptr(prev), _ptr(o_compact), _ptr(idx), keep_k,
                                    _ptr(out), _stream(stream)))


def var_block_mask_build(p: var_problem, step: int, qblock_side: int, radius: int,
                         sink_max_side: int) -> Tuple[np.ndarray, np.ndarray, int]:
    """Host call: returns (row_ptr int32 [n_qblocks+1], entries int32 [nnz], sink_len)."""
    nnz, nqb, sink = C.c_int32(), C.c_int32(), C.c_int32()
    _check("var_block_mask_build",
           _lib.var_block_mask_build(C.byref(p), step, qblock_side, radius, sink_max_side, None, None,
                                     0, C.byref(nnz), C.byref(nqb), C.byref(sink)))
    row_ptr = np.zeros(nqb.value + 1, dtype=np.int32)
    entries = np.zeros(max(1, nnz.value), dtype=np.int32)
    _check("var_block_mask_build",
           _lib.var_block_mask_build(C.byref(p), step, qblock_side, radius, sink_max_side,
                                     row_ptr.ctypes.data_as(C.c_void_p),
                                     entries.ctypes.data_as(C.c_void_p), entries.size,
                                     C.byref(nnz), C.byref(nqb), C.byref(sink)))
    return row_ptr, entries[: nnz.value], sink.value


def var_block_mask_plan(p: var_problem, step: int, qblock_side: int, row_ptr: np.ndarray, entries: np.ndarray,
                        sink_len: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Host call: the block-sparse kernel's plan, (sq_ptr, sq_units, sq_order) int32 arrays."""
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    en = np.ascontiguousarray(entries, dtype=np.int32)
    n_sq, n_u = C.c_int32(), C.c_int32()
    _check("var_block_mask_plan",
           _lib.var_block_mask_plan(C.byref(p), step, qblock_side, rp.ctypes.data, en.ctypes.data, sink_len, None,
                                    None, 0, None, C.byref(n_sq), C.byref(n_u)))
    sq_ptr = np.zeros(n_sq.value + 1, dtype=np.int32)
    sq_units = np.zeros(2 * max(n_u.value, 1), dtype=np.int32)
    sq_order = np.zeros(n_sq.value, dtype=np.int32)
    _check("var_block_mask_plan",
           _lib.var_block_mask_plan(C.byref(p), step, qblock_side, rp.ctypes.data, en.ctypes.data, sink_len,
                                    sq_ptr.ctypes.data, sq_units.ctypes.data, n_u.value, sq_order.ctypes.data,
                                    C.byref(n_sq), C.byref(n_u)))
    return sq_ptr, sq_units[: 2 * n_u.value], sq_order


def block_mask_struct(qblock_side: int, row_ptr: torch.Tensor, entries: torch.Tensor,
                      sink_len: int, plan: Optional[Tuple[torch.Tensor, torch.Tensor, torch.Tensor]] = None
                      ) -> var_block_mask:
    """var_block_mask over device copies of var_block_mask_build's arrays and,
    optionally, of var_block_mask_plan's (sq_ptr, sq_units, sq_order)."""
    m = var_block_mask()
    m.qblock_side = qblock_side
    m.n_qblocks = row_ptr.numel() - 1
    m.sink_len = sink_len
    m.nnz = entries.numel()
    m.row_ptr = row_ptr.data_ptr()
    m.entries = entries.data_ptr()
    if plan is not None:
        sq_ptr, sq_units, sq_order = plan
        m.n_squares = sq_order.numel()
        m.plan_units = sq_units.numel() // 2
        m.sq_ptr = sq_ptr.data_ptr()
        m.sq_units = sq_units.data_ptr()
        m.sq_order = sq_order.data_ptr()
    return m


def var_attn_blocksparse(p: var_problem, step: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         mask: var_block_mask, o: torch.Tensor, stream=None) -> None:
    _check("var_attn_blocksparse",
           _lib.var_attn_blocksparse(C.byref(p), step, _ptr(q), _ptr(k), _ptr(v), C.byref(mask),
                                     _ptr(o), _stream(stream)))
