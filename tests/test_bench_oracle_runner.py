"""The benchmark's CPU baseline runner on the host (no GPU): the oracle run as
(sequence, KV head) units by worker processes over a shared-memory copy of
the cache pages.  Every unit must be run exactly once, the bytes and tokens
must add up to the sampled sequences, and a step's time is its slowest
worker's."""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.mark.parametrize("workers", [1, 3])
def test_oracle_runner_covers_every_unit(workers):
    import bench
    from paged_gqa_decode_rope_gb300.workloads import Workload
    lengths = [1, 63, 130, 300]
    wl = Workload("custom", seed=3, lengths=lengths, kv_dtype=0, device="cpu")
    steps = [[0, 1, 2, 3], [2]]
    res, used = bench.run_oracle_steps(wl, steps, 0.0, workers=workers)
    assert used == workers
    assert len(res) == 2
    # one KV head's K and V per unit: 128 x 2 x 2 bytes per token (BF16)
    assert res[0]["units"] == 8 * len(lengths)
    assert res[0]["tokens"] == sum(lengths)
    assert res[0]["bytes"] == sum(lengths) * 8 * 128 * 2 * 2
    assert res[1]["units"] == 8 and res[1]["tokens"] == 130
    assert all(r["seconds"] > 0 for r in res)


def test_oracle_runner_fp8_and_host_cores():
    import bench
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=4, lengths=[70, 5], kv_dtype=1, device="cpu")
    res, used = bench.run_oracle_steps(wl, [[0, 1]], 0.0, workers=2)
    assert used == 2
    assert res[0]["bytes"] == 75 * 8 * 128 * 2 * 1
    assert bench.host_cores() >= 1
