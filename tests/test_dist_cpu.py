"""Multi-process path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The forward shards by work item with no data-path collective; the only
cross-rank steps are the barriers around the timed region and the max of
the per-rank times, which these tests exercise with world_size 2.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup()
    bench.barrier(w)
    m = bench.max_over_ranks(times[rank], w, torch.device("cpu"))
    bench.barrier(w)
    out_q.put((r, w, local, m))
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo path is the no-GPU configuration")
def test_two_ranks_max_time():
    world, port = 2, _free_port()
    times = [1.25, 3.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == world for r in res)
    assert all(r[3] == max(times) for r in res)  # every rank sees the slowest rank's time


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, torch.device("cpu")) == 2.5
    bench.barrier(1)  # no process group: a no-op
