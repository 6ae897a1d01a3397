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


def _shard_rank_main(rank, world, port, out_q):
    """One gloo rank: compute this rank's (b, n) slabs with the oracle, gather every rank's pieces."""
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    import synth
    from masked_attention_tri_gb300.shard import per_batch_pieces, slab_range
    dist.init_process_group("gloo")
    c = synth.make_triangle("shard", 2, 5, 2, 20, 24, 8, "bf16", "bf16", seed=71, mask="kvlen", kv_range=(0, 24))
    u0, u1 = slab_range(c.B * c.N, world, rank)
    mine = []
    for b, n0, n1 in per_batch_pieces(u0, u1, c.N):
        O, L, M = oracle.tri_fwd(c.q[b:b + 1, n0:n1], c.k[b:b + 1, n0:n1], c.v[b:b + 1, n0:n1], c.bias[b:b + 1],
                                 kv_lengths=c.kv_lengths[b:b + 1, n0:n1], scale=c.scale)
        mine.append((b, n0, n1, O, L, M))
    pieces = [None] * world
    dist.all_gather_object(pieces, mine)
    out_q.put((rank, u0, u1, pieces))
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo path is the no-GPU configuration")
def test_n_slab_split_covers_each_slab_once_and_matches_whole_problem():
    """World size 2: the ranks' slab ranges partition B*N, and their per-slab results, put side by
    side, equal the whole problem computed at once (the bias is replicated, nothing is exchanged)."""
    import numpy as np
    import oracle
    import synth
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    c = synth.make_triangle("shard", 2, 5, 2, 20, 24, 8, "bf16", "bf16", seed=71, mask="kvlen", kv_range=(0, 24))
    assert [(r[1], r[2]) for r in res] == [(0, 5), (5, 10)]
    rO, rL, rM = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale)
    seen = np.zeros((c.B, c.N), int)
    for b, n0, n1, O, L, M in (p for rank_pieces in res[0][3] for p in rank_pieces):
        seen[b, n0:n1] += 1
        np.testing.assert_array_equal(O[0], rO[b, n0:n1])
        np.testing.assert_array_equal(L[0], rL[b, n0:n1])
        np.testing.assert_array_equal(M[0], rM[b, n0:n1])
    assert (seen == 1).all()


def test_slab_ranges_partition_for_any_world():
    sys.path.insert(0, ROOT)
    from masked_attention_tri_gb300.shard import per_batch_pieces, slab_range
    for units in (1, 7, 768, 1000):
        for world in (1, 2, 3, 8):
            ranges = [slab_range(units, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == units
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [r[1] - r[0] for r in ranges]
            assert max(sizes) - min(sizes) <= 1
    assert list(per_batch_pieces(3, 12, 5)) == [(0, 3, 5), (1, 0, 5), (2, 0, 2)]
    with pytest.raises(ValueError):
        slab_range(10, 2, 2)
