"""The multi-GPU path of bench.py is replicas only: every rank runs the whole
step on its own GPU, a barrier brackets the timed region, the slowest rank's
time is taken and rank 0 alone prints.  These CPU tests run that host logic as
two gloo ranks (no GPU): the max-over-ranks reduction, the whole-job
throughput, and the reference arm leaving ranks other than 0 without work."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        # each rank's own step time and e2e time; the job takes the slowest
        mine = [1.0 + rank, 5.0 - rank]
        ms = bench.max_over_ranks(mine, "cpu")
        dist.barrier()

        class Args:
            workload = "c1_single_linear_256x512x512"
            steps, warmup, cpu_sample = 1, 3, 16
            fuse_shared_input, linear = False, []
        ref = bench.run_reference(Args) if rank != 0 else "rank 0 runs the oracle"
        out[rank] = (ms, ref)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_only_rank0_reports():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == [2.0, 5.0] and res[1][0] == [2.0, 5.0]
    assert res[1][1] is None   # the reference arm does no work on rank 1


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    flops = 6 * 8192 * 2048 * 5504
    one = bench.job_throughput(1, flops, 0.5)
    assert one == pytest.approx(flops / 0.5e-3 / 1e12)
    assert bench.job_throughput(4, flops, 0.5) == pytest.approx(4 * one)
    assert bench.max_over_ranks([3.0, 1.5], "cpu") == [3.0, 1.5]   # no process group: unchanged
