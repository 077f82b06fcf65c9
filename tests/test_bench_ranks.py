"""bench.py's multi-rank helpers on CPU: two gloo ranks agree on the
maximum of their timings (the whole-job time is the slowest rank's)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    m = bench.max_over_ranks(10.0 + 5.0 * rank, ws)
    out[rank] = m
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0


def test_region_split_and_median():
    import bench
    assert bench.region_sizes(20) == [4, 4, 4, 4, 4]
    assert bench.region_sizes(7) == [2, 2, 1, 1, 1]
    assert bench.region_sizes(3) == [1, 1, 1]
    assert sum(bench.region_sizes(1307)) == 1307
    # rates 1, 4, 2, 5, 3 steps/ms: the median region is the one at 3
    sizes, ms = [2, 4, 2, 5, 3], [2.0, 1.0, 1.0, 1.0, 1.0]
    assert bench.median_region(sizes, ms) == 4
