"""The N > 1 path of bench.py on CPU: two gloo ranks, each with its own
batch; the job time is the slowest rank's and the value counts every rank's
tokens (weak scaling, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_setup() == (world, rank, rank)
    local_ms = [0.5, 2.0][rank]                      # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, world)
    out[rank] = (ms, bench.weak_scaling_value(64, world, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_and_count_all_tokens():
    world, port = 2, _free_port()
    with tmp.Manager() as mgr:
        out = mgr.dict()
        tmp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0
    assert res[0][1] == pytest.approx(64 * 2 / 2e-3)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.weak_scaling_value(64, 1, 0.5) == pytest.approx(128000.0)
