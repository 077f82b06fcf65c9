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


def test_oracle_sample_share_is_the_pieces_flops(monkeypatch):
    # the bounded oracle baseline: above the threshold a block is sampled as
    # 1/H of it and counted by the piece's share of the block's FLOPs
    import numpy as np
    import bench
    from layerwise_weight_offload_gb300 import workloads as W
    w = W.custom("samp", n_blocks=1, hidden=128, heads=2, mlp=512, tokens=64, shards=1)
    monkeypatch.setattr(bench, "FULL_ORACLE_FLOPS", 0)
    run, share, text, threads = bench.oracle_sample(w)
    d, f, T, hd, r = 128, 512, 64, 64, 32
    flops = 2 * T * d * 3 * hd + 4 * T * T * hd + 2 * r * (d * d + 2 * d * f)
    assert abs(share - flops / w.flops_per_block()) < 1e-12
    out = run()
    assert out.shape == (r, d) and np.isfinite(out).all()
    assert "1/2 of an fp64 oracle block forward" in text
    monkeypatch.setattr(bench, "FULL_ORACLE_FLOPS", 1e30)
    run, share, text, _ = bench.oracle_sample(w)
    assert share == 1.0 and text.startswith("one fp64 oracle block forward")
    run()
