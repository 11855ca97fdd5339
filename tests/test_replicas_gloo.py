"""Host-side logic of the multi-process (replica) bench path, run as two
gloo ranks on the CPU: the max-over-ranks timing, the whole-job aggregate,
the reference arm's rank-0-only rule, and that a rank leaving before the
barrier surfaces on the other rank as an error within a short timeout
(no GPU is involved anywhere here)."""
import datetime
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port, timeout_s=30):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))


def _aggregate_worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    _init(rank, world, port)
    bench.barrier(world)
    local_ms = [40.0, 55.0][rank]            # rank 1 is the slow replica
    per_s, total = bench.job_throughput(local_ms, 10, 1.0e9, world, torch.device("cpu"))
    out[rank] = (per_s, total)
    dist.destroy_process_group()


def test_two_rank_throughput_uses_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_aggregate_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        per_s, total = out[r]
        assert total == 55.0                  # max over ranks, seen by every rank
        assert per_s == pytest.approx(2 * 10 * 1.0e9 / 0.055)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        pass
    # a non-zero rank returns at once, without touching the oracle or inputs
    assert bench.run_reference(Args(), 2, 1) == 0


def _leaver_worker(rank, world, port, out):
    _init(rank, world, port, timeout_s=3)
    if rank == 1:
        return                                # leaves between steps, never joins the barrier
    try:
        dist.barrier()
        out[rank] = "joined"
    except Exception as e:                    # the survivor learns of it as an error
        out[rank] = type(e).__name__


def test_rank_that_leaves_is_reported_not_hung():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    ctx = mp.start_processes(_leaver_worker, args=(world, port, out), nprocs=world, join=False,
                             start_method="spawn")
    for p in ctx.processes:
        p.join(timeout=60)
    alive = [p for p in ctx.processes if p.is_alive()]
    for p in alive:
        p.kill()
    assert not alive, "a rank was still waiting after the process-group timeout"
    assert out.get(0) not in (None, "joined")
