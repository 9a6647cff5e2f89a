"""Host logic of bench.py's multi-rank run (replicas, one process per GPU),
exercised with two gloo ranks on the CPU: the timed region's time is the
slowest rank's, and the reported rate is the whole job's."""
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup(None)
        secs = bench.max_over_ranks(dist, 1.0 + 0.5 * rank, "cpu")
        rate = bench.whole_job_rate(3.514e11, 10, w, secs, 1e12)
        out.put((r, w, local, secs, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_the_whole_job_rate():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for r, (rank, world, local, secs, rate) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert secs == 1.5  # the slower rank's time on both
        assert rate == pytest.approx(3.514e11 * 10 * 2 / 1.5 / 1e12)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 0.25, "cpu") == 0.25
    assert bench.whole_job_rate(2.0, 5, 1, 2.0, 1.0) == 5.0
