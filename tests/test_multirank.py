"""The multi-rank host logic of bench.py, on CPU with the gloo backend (world size 2).

The decode step shards by batch with no exchange (replicas, weak scaling), so the
only collectives are the timing barrier and the max / sum over ranks that turn
per-rank step times and bytes into the whole-job number. Each rank runs as its own
process, as under torchrun.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import torch.distributed as dist

    class Args:
        pass

    w, r, _ = bench.dist_setup(Args())
    try:
        bench.barrier(w)
        step_ms = 1.0 + r  # rank 1 is slower
        mx = bench.max_over_ranks(w, step_ms)
        total = bench.sum_over_ranks(w, 100.0 * (r + 1))
        q.put((r, w, mx, total))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, w, mx, total in res:
        assert w == 2
        assert mx == pytest.approx(2.0)  # the slowest rank's time is the job's time
        assert total == pytest.approx(300.0)  # whole-job bytes add up over ranks


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(1, 3.5) == 3.5
    assert bench.sum_over_ranks(1, 7.0) == 7.0
