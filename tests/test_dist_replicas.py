"""`bench.py --gpus N` runs N independent replicas ("replicas only": the layer
has no exchange step on one GPU).  Its multi-rank plumbing -- process group
set-up from the torchrun environment, the barrier around the timed region and
the max-over-ranks time -- is checked here with two gloo ranks on the CPU."""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank), "BENCH_BACKEND": "gloo"})
    sys.path.insert(0, str(ROOT))
    import bench
    dist, r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(dist)
    # each replica reports its own time; the slowest one defines the step
    out[rank] = bench.max_over_ranks(1.5 + rank, dist)
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a gloo rank did not finish")
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_group():
    sys.path.insert(0, str(ROOT))
    import bench
    env = os.environ.pop("WORLD_SIZE", None)
    try:
        dist, r, w, local = bench.dist_setup(1)
        assert dist is None and (r, w, local) == (0, 1, 0)
        assert bench.max_over_ranks(3.25, None) == 3.25
    finally:
        if env is not None:
            os.environ["WORLD_SIZE"] = env
