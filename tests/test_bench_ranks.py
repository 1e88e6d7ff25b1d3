"""The bench's multi-rank host logic on CPU: two gloo ranks agree on the
slowest rank's time, draw different batches and report the whole-job value."""

import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, ws, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, _ = bench._dist()
        slowest = bench.max_over_ranks(times[rank], got_ws, "cpu")
        out.put((got_rank, slowest, bench.rank_seed(7, got_rank),
                 bench.whole_job_tbps(got_ws, 1e9, 10, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [3.0, 5.0]
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 5.0 for r in res)             # both see the slowest rank
    assert res[0][2] != res[1][2]                     # each rank its own batch
    assert res[0][3] == pytest.approx(2 * 1e9 * 10 / 5e-3 / 1e12)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.5, 1, "cpu") == 4.5
    assert bench.whole_job_tbps(1, 2e9, 4, 2.0) == pytest.approx(4.0)
