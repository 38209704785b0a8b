"""The multi-GPU path of bench.py on CPU: independent replicas (weak scaling) whose job time is
the slowest rank's, reduced over a world-size-2 gloo process group.  No GPU is touched."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        w, r, lr = bench.dist_env()
        local_ms = 10.0 + 5.0 * rank                     # the ranks finish at different times
        job = bench.job_time_ms(local_ms, w)
        value = bench.job_throughput(50, 100, w, job)
        out[rank] = (w, r, lr, job, value)
    finally:
        dist.destroy_process_group()


def test_replica_job_time_is_the_slowest_rank_and_value_counts_all_ranks():
    ws, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_rank, args=(ws, port, out), nprocs=ws, join=True)
    for rank in range(ws):
        w, r, lr, job, value = out[rank]
        assert (w, r, lr) == (ws, rank, rank)
        assert job == 15.0                              # max over ranks, seen by every rank
        # 50 tokens x 100 steps on each of 2 replicas in 15 ms
        assert value == pytest.approx(50 * 100 * 2 / 0.015)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time_ms(12.5, 1) == 12.5
    assert bench.job_throughput(50, 10, 1, 12.5) == pytest.approx(500 / 0.0125)


def _ref_rank(rank, ws, port, out):
    """The reference arm under torchrun: rank 0 alone does the work, the others return."""
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench

    class Args:
        workload = "tiny"
        steps = 1
        warmup = 0
        gpus = ws

    if rank == 0:
        out[rank] = "skipped"                          # rank 0 would time the oracle; not needed here
        return
    bench.run_reference(Args())
    out[rank] = "returned"


def test_reference_arm_non_zero_ranks_exit_without_work():
    ws, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_ref_rank, args=(ws, port, out), nprocs=ws, join=True)
    assert out[1] == "returned"
