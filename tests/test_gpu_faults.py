"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up, the status word reports VAR_ERR_TIMEOUT, and the device
keeps working."""
import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import cache_len, randn_bf16
from tests._util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_that_runs_out_is_reported_and_the_device_stays_usable():
    V.var_device_status(clear=True)
    V.var_selftest_wait_timeout(20000)                # 20 ms, the per-device word
    torch.cuda.synchronize()
    assert V.var_device_status(clear=True) == V.VAR_ERR_TIMEOUT
    assert V.var_device_status(clear=False) == 0      # cleared
    sides, B, H, D = (1, 2, 4, 8), 1, 2, 64
    L, N = cache_len(sides, 3), 64
    q, k, v = randn_bf16((B, H, N, D), 51), randn_bf16((B, H, L, D), 52), randn_bf16((B, H, L, D), 53)
    o = torch.empty_like(q, device=DEV)
    V.var_attn_dense(V.problem(B, H, D, sides), 3, q.to(DEV), k.to(DEV), v.to(DEV), o)
    torch.cuda.synchronize()
    assert_close(o, oracle.attention(q, k, v, L), "dense after a timeout")
    assert V.var_device_status(clear=True) == 0
