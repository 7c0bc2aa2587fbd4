"""The N > 1 host logic of bench.py on CPU: two gloo ranks on 127.0.0.1 run
the same set-up, barrier and max-over-ranks timing the benchmark uses around
its timed region (one independent replica per GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist

    r, local, ws = bench.dist_setup(world)
    bench.barrier(ws)
    # each rank reports its own step time; the job's time is the slowest rank's
    got = bench.max_over_ranks(10.0 + 5.0 * r, ws)
    bench.barrier(ws)
    out[r] = (r, local, ws, got)
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert sorted(out.values()) == [(0, 0, 2, 15.0), (1, 1, 2, 15.0)]
