"""Seeded synthetic inputs for the VAR attention hot path.

This module only draws random numbers and lays them out in the shapes of the
workloads; it holds none of the method's arithmetic (no attention, no scoring,
no interpolation, no masks).  Both the CPU oracle tests and the CUDA path read
tensors made here, so parity never depends on the random stream.

Workloads (scale schedules of next-scale prediction, one token grid per scale,
tokens of a scale in row-major order, scales concatenated in order):

* ``dense_tiny``      -- 256px schedule, batch 1, 16 heads, head_dim 64, the
                         last step only (256 queries vs a 680-token cache).
* ``dense_256px``     -- 256px schedule, every step, batch 2 (classifier-free
                         guidance cond + uncond pair), 16 heads, head_dim 64,
                         scale-1 key scaled x4 to act as an attention sink.
* ``dense_1024px``    -- 1024px schedule, the final 64x64 step (4096 queries vs a
                         10,521-token cache), batch 2 CFG pair, head_dim 128, sink.
* ``pruned_1024px``   -- the 1024px tensors plus hidden-state grids (2048
                         channels) for the 48x48 and 64x64 steps, keep ratios
                         0.4 and 0.2.
* ``blocksparse_2k``  -- 2K schedule, the final 128x128 step (16,384 queries vs a
                         42,521-token cache) in 8x8 query blocks, batch 2,
                         head_dim 128, plain i.i.d. N(0,1).

Recipe: ``torch.Generator().manual_seed(seed)``, ``torch.randn`` in fp32 on the
CPU, rounded to bf16 (round-to-nearest-even, torch's ``.to(torch.bfloat16)``).
Draw order: K, V (whole cache), then Q of each step in schedule order, then the
unconditional-branch noise for K, V and each Q in the same order, then the
hidden states.  The unconditional branch is ``cond + 0.1 * noise`` computed in
fp32 and rounded once.  The sink multiplies key row 0 (the single token of the
1x1 scale) by 4 in both batch elements; x4 is exact in bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import torch

SCHEDULE_256 = (1, 2, 3, 4, 5, 6, 8, 10, 13, 16)
SCHEDULE_1024 = (1, 2, 4, 6, 8, 12, 16, 20, 24, 32, 40, 48, 64)
SCHEDULE_2K = SCHEDULE_1024 + (80, 96, 128)


@dataclass(frozen=True)
class Workload:
    name: str
    sides: Tuple[int, ...]
    batch: int
    heads: int
    head_dim: int
    steps: Tuple[int, ...]          # 0-based indices into ``sides`` that are run
    cfg_pair: bool = False          # batch 1 = batch 0 + 0.1 * noise
    sink: bool = False              # key row 0 multiplied by 4
    seed: int = 0
    channels: int = 0               # hidden-state width for pivot scoring
    keep: Tuple[Tuple[int, int, int], ...] = ()   # (step, ratio_num, ratio_den)
    qblock_side: int = 0            # block-sparse query block side
    radius: int = 0                 # block-sparse local window radius (blocks)
    sink_max_side: int = 0          # scales with side <= this are always kept

    @property
    def n_tokens(self) -> int:
        return sum(s * s for s in self.sides)


WORKLOADS: Dict[str, Workload] = {
    "dense_tiny": Workload("dense_tiny", SCHEDULE_256, 1, 16, 64, (9,), seed=0),
    "dense_256px": Workload("dense_256px", SCHEDULE_256, 2, 16, 64, tuple(range(10)),
                            cfg_pair=True, sink=True, seed=1),
    "dense_1024px": Workload("dense_1024px", SCHEDULE_1024, 2, 16, 128, (12,),
                             cfg_pair=True, sink=True, seed=2),
    "pruned_1024px": Workload("pruned_1024px", SCHEDULE_1024, 2, 16, 128, (10, 11, 12),
                              cfg_pair=True, sink=True, seed=3, channels=2048,
                              keep=((11, 2, 5), (12, 1, 5))),
    "blocksparse_2k": Workload("blocksparse_2k", SCHEDULE_2K, 2, 16, 128, (15,),
                               seed=4, qblock_side=8, radius=2, sink_max_side=16),
}


def _randn(gen: torch.Generator, shape: Sequence[int]) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def _pair(gen: torch.Generator, cond: torch.Tensor, n_extra: int = 0) -> torch.Tensor:
    """Stack cond (batch 0) with cond + 0.1*noise (batch 1), fp32."""
    noise = _randn(gen, cond.shape)
    return torch.stack([cond, cond + 0.1 * noise], dim=0)


@dataclass
class Inputs:
    workload: Workload
    k: torch.Tensor                       # [B, H, L_total, D] bf16
    v: torch.Tensor                       # [B, H, L_total, D] bf16
    q: Dict[int, torch.Tensor]            # step -> [B, H, side^2, D] bf16
    x: Dict[int, torch.Tensor] = field(default_factory=dict)  # step -> [B, side^2, C] bf16


def make_inputs(w: Workload, seed: Optional[int] = None,
                steps: Optional[Sequence[int]] = None) -> Inputs:
    """Draw the tensors of workload ``w`` (CPU, bf16)."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    steps = tuple(w.steps if steps is None else steps)
    L = w.n_tokens
    H, D = w.heads, w.head_dim
    b_draw = 1 if w.cfg_pair else w.batch
    k = _randn(gen, (b_draw, H, L, D))
    v = _randn(gen, (b_draw, H, L, D))
    qs = {s: _randn(gen, (b_draw, H, w.sides[s] ** 2, D)) for s in steps}
    if w.cfg_pair:
        k = _pair(gen, k[0])
        v = _pair(gen, v[0])
        qs = {s: _pair(gen, qs[s][0]) for s in steps}
    k = k.to(torch.bfloat16)
    v = v.to(torch.bfloat16)
    qs = {s: t.to(torch.bfloat16).contiguous() for s, t in qs.items()}
    if w.sink:
        k[:, :, 0, :] = k[:, :, 0, :] * 4
    xs = {}
    for (s, _num, _den) in w.keep:
        xs[s] = _randn(gen, (w.batch, w.sides[s] ** 2, w.channels)).to(torch.bfloat16)
    return Inputs(w, k.contiguous(), v.contiguous(), qs, xs)


def randn_bf16(shape: Sequence[int], seed: int) -> torch.Tensor:
    """Plain i.i.d. N(0,1) bf16 tensor of ``shape`` (CPU)."""
    gen = torch.Generator().manual_seed(seed)
    return _randn(gen, shape).to(torch.bfloat16)


def cache_len(sides: Sequence[int], step: int) -> int:
    """Number of cached tokens visible at ``step``: all tokens of scales 0..step."""
    return sum(s * s for s in sides[: step + 1])
