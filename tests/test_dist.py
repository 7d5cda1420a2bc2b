"""bench.py's multi-process path on CPU: gloo, world size 2, 127.0.0.1.

The attention path has no exchange step, so N GPUs run N independent
replicas; the only cross-rank traffic is the host-side barrier and the
max-over-ranks of the timed region, which these tests exercise."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, loc = bench.dist_setup()
    assert (w, r, loc) == (world, rank, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(w, 10.0 * (rank + 1))     # this rank's "timed region" in ms
    bench.barrier(w)
    dist.destroy_process_group()


def test_replica_coordination_gloo_two_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a threaded process
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        assert out[0] == out[1] == 20.0          # both ranks see the slowest rank's time


def test_whole_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tflops(1, 9.6e11, 10, 10.0)
    two = bench.whole_job_tflops(2, 9.6e11, 10, 10.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(9.6e11 * 10 / 0.01 / 1e12)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload, steps, warmup, gpus = "tiny", 1, 3, 2
    bench.run_reference(A, world=2, rank=1)
    assert capsys.readouterr().out == ""
