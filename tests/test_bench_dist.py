"""Host logic of bench.py's multi-process mode, on CPU with gloo ranks.

With N processes the bench runs N replicas of the workload (weak scaling);
the only cross-rank steps are a barrier around the timed region and the
maximum of the per-rank step times.  These run here on two gloo ranks.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        bench.barrier(w)
        step_ms = 2.0 + rank  # rank 1 is the slower one
        ms = bench.max_over_ranks(step_ms, w)
        bench.barrier(w)
        q.put((r, w, local, ms, bench.job_value(1.0e9, w, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    import torch.multiprocessing as mp

    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, (r, w, local, ms, value) in enumerate(got):
        assert (r, w, local) == (rank, world, rank)
        assert ms == pytest.approx(3.0)  # every rank sees the slowest rank's time
        # 2 ranks x 1e9 units in 3 ms
        assert value == pytest.approx(2 * 1.0e9 / 3.0e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(5.0, 1) == 5.0
    bench.barrier(1)
    assert bench.job_value(10.0, 1, 1000.0) == pytest.approx(10.0)
