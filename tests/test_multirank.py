"""The multi-GPU host logic of bench.py on CPU: two gloo ranks.  Each rank runs
the whole workload (weak scaling, no collective on the data path); the only
exchange is the barrier around the timed region and the max over ranks of the
measured time, from which `value` counts the work of every rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_info()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    my_ms = 1.5 + rank                                  # rank 1 is the slow one
    worst = bench.reduce_max(my_ms, ws, torch.device("cpu"))
    flops = 706.05e9
    value = ws * flops / worst / 1e9                    # whole-job TFLOP/s, as run_gpu computes it
    out[rank] = (worst, value)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time_and_count_all_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    assert out[0] == out[1]
    worst, value = out[0]
    assert worst == pytest.approx(2.5)
    assert value == pytest.approx(2 * 706.05e9 / 2.5 / 1e9)
