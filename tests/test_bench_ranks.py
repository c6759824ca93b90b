"""The bench's multi-process path, on CPU with gloo (world size 2).

With N GPUs the bench runs N independent replicas of the decode + gather step
(the path has no exchange step, so no collective sits on the data path); the
only cross-rank operations are the barriers and the max over ranks of the
timed step, and only rank 0 prints.  These run here without a GPU.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.0 + 0.5 * rank            # rank 1 is the slower one
        dist.barrier()
        got = bench.max_over_ranks(ms, dist, "cpu")
        q.put((rank, got, bench.whole_job_gbps(1e9, world, got)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [1.5, 1.5]
    # Whole-job GB/s: 2 ranks x 1e9 bytes per step over the slowest 1.5 ms.
    assert res[0][2] == pytest.approx(2e9 / 1.5e-3 / 1e9)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    assert bench.whole_job_gbps(1e9, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        steps, warmup = 1, 0
    assert bench.run_reference(Args, world=2, rank=1) == 0
    assert capsys.readouterr().out == ""
