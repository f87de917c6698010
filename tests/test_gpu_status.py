"""Per-call status words: a fault a kernel detects is recorded in the status
word of the call that raised it (var_problem.status), read in stream order by
var_check_status, and nowhere else."""
import numpy as np
import pytest
import torch

import oracle
import visual_autoregressive_next_var_b300 as V
from var_synth import cache_len, randn_bf16
from tests._util import assert_close, check_device_status

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_two_streams_only_the_faulting_call_reports():
    sides, D, B, H = (1, 2, 4, 8, 16, 32), 128, 1, 2
    step, L, N = 5, cache_len(sides, 5), 1024
    q = randn_bf16((B, H, N, D), 31)
    k = randn_bf16((B, H, L, D), 32)
    v = randn_bf16((B, H, L, D), 33)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    check_device_status()
    words = torch.zeros(2, dtype=torch.int32, device=DEV)
    p_bad = V.problem(B, H, D, sides, status=words[0:1])
    p_good = V.problem(B, H, D, sides, status=words[1:2])
    rp, ent, sink = V.var_block_mask_build(p_bad, step, 8, 1, 4)
    ent = ent.copy()
    ent[rp[1] - 1] = 31 << 24                     # last entry of block 0: a scale with no tensor map
    m = V.block_mask_struct(8, torch.as_tensor(rp, device=DEV), torch.as_tensor(ent, device=DEV), sink)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    o_bad = torch.empty_like(qd)
    o_good = torch.empty_like(qd)
    V.var_attn_blocksparse(p_bad, step, qd, kd, vd, m, o_bad, stream=s1)
    V.var_attn_dense(p_good, step, qd, kd, vd, o_good, stream=s2)
    assert V.var_check_status(words[0:1], clear=False, stream=s1) == V.VAR_ERR_INVALID_ARG
    assert V.var_check_status(words[1:2], stream=s2) == 0
    assert V.var_device_status(clear=False) == 0           # the per-device word saw nothing
    assert V.var_check_status(words[0:1], clear=True, stream=s1) == V.VAR_ERR_INVALID_ARG
    assert V.var_check_status(words[0:1], stream=s1) == 0   # cleared
    torch.cuda.synchronize()
    assert_close(o_good, oracle.attention(q, k, v, L), "dense beside a faulting call")
    check_device_status()


def test_timeout_lands_in_the_given_word():
    word = torch.zeros(1, dtype=torch.int32, device=DEV)
    check_device_status()
    V.var_selftest_wait_timeout(10000, status=word)          # 10 ms
    assert V.var_check_status(word) == V.VAR_ERR_TIMEOUT
    assert V.var_check_status(word) == 0
    assert V.var_device_status(clear=False) == 0
