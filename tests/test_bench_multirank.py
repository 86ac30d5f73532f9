"""bench.py's multi-rank logic on CPU: two gloo ranks (world size 2).

With N GPUs every rank runs an independent replica of the workload (the
path shards over (batch, head) with no exchange), so the only cross-rank
steps are the barrier around the timed region and the max over ranks of the
measured time; the job's rate is the units of all ranks over the slowest
rank's time."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier()
        assert bench.world_size() == world
        # rank r measured (r + 1) seconds for 100 tokens
        rate, slowest = bench.job_throughput(100.0, float(rank + 1))
        mx = bench.max_over_ranks(float(10 * rank - 3))
        bench.barrier()
        out[rank] = (rate, slowest, mx)
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        rate, slowest, mx = out[r]
        assert slowest == 2.0               # both ranks see the slowest rank's time
        assert rate == pytest.approx(100.0)  # 2 ranks x 100 tokens / 2 s
        assert mx == 7.0


def test_single_process_needs_no_group():
    import bench
    assert not torch.distributed.is_initialized()
    assert bench.world_size() == 1
    assert bench.job_throughput(50.0, 0.5) == (100.0, 0.5)
    bench.barrier()  # no-op
