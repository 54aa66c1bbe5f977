"""The N > 1 path of bench.py on CPU ranks (gloo, world size 2): every rank
runs one replica; the timing is the slowest rank's, and the whole-job value
adds the work of all ranks over that time."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [12.5, 20.0][rank]
    ms_max = bench.max_over_ranks(ms, world)
    q.put((rank, ms_max, bench.whole_job_tflops(world, 4e12, ms_max)))
    dist.barrier()
    dist.destroy_process_group()


def test_bench_aggregates_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, ms_max, tf in out:
        assert ms_max == pytest.approx(20.0)
        assert tf == pytest.approx(2 * 4e12 / 0.020 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
