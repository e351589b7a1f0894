"""The bench's multi-rank logic on CPU with the gloo backend, world size 2
(one GPU per rank on a GPU node; here plain processes): the job time is the
slowest rank's, every rank sees the same value, and the reference arm runs on
rank 0 only.  Replicas only: the product path has no collective."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.max_over_ranks(values[rank], world, "cpu")
        bench.barrier(world)
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("values", [(3.5, 7.25), (9.0, 1.0)])
def test_slowest_rank_sets_the_time_on_every_rank(values):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: max(values), 1: max(values)}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, 1, "cpu") == 4.0
    bench.barrier(1)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    args = argparse.Namespace(workload="q6k_sweep", steps=1, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None
