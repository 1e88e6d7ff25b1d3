"""GPU planner vs the oracle planner: bit-exact work lists and coverage."""

import numpy as np
import pytest
import torch

from oracle import plan as op
import gpu_util as gu

pytestmark = pytest.mark.gpu


def _mixes():
    rng = np.random.default_rng(5)
    yield [1, 63, 64, 300]
    yield [4096] * 32
    yield [131072] + [4096] * 31
    yield [0, 5, 0, 64 * 7 + 1]
    yield [0, 0, 0]
    yield [65, 1]
    yield list(rng.integers(1, 5000, size=50))
    yield list(np.floor(np.exp(rng.uniform(np.log(128), np.log(262144), 64))).astype(int))
    yield list(rng.integers(0, 200, size=3000))            # many sequences, > 1 per thread


def _run_dynamic(lens, C, min_tiles, capacity=None, J=0, kmin=1):
    from paged_gqa_decode_rope_gb300 import ops
    B = len(lens)
    max_blocks = max(1, max(-(-L // 64) for L in lens))
    cap = C * (1 + J) + 8 * B if capacity is None else capacity
    plan = ops.DecodePlan(B, C, cap, "cuda", pool_chunks=J, pool_min_tiles=kmin)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.decode_plan(torch.tensor(lens, dtype=torch.int32, device="cuda"), max_blocks, plan,
                    status, min_tiles)
    torch.cuda.synchronize()
    return plan, int(status.item())


def _host(plan, n_items):
    items = [tuple(x) for x in plan.items[:n_items].cpu().tolist()]
    return items, plan.cta_ptr.cpu().tolist(), plan.seg_ptr.cpu().tolist()


@pytest.mark.parametrize("J,kmin", [(0, 1), (1, 1), (6, 1), (4, 2), (4, 16)])
@pytest.mark.parametrize("C", [1, 7, 152, 304, 1000])
def test_dynamic_plan_bit_exact(C, J, kmin):
    gu.require_gpu()
    for lens in _mixes():
        for min_tiles in (1, 4):
            plan, st = _run_dynamic(lens, C, min_tiles, J=J, kmin=kmin)
            assert st == 0
            items, cta_ptr, seg_ptr, home_end, pool = op.plan_dynamic(lens, C, min_tiles, J, kmin)
            got = _host(plan, len(items))
            assert got[1] == cta_ptr, "cta_ptr"
            assert got[2] == seg_ptr, "seg_ptr"
            assert got[0] == [tuple(i) for i in items], "items"
            assert plan.home_end.cpu().tolist() == home_end, "home_end"
            pl = plan.pool.cpu().tolist()
            assert pl[:3] == [0, 0, len(pool)] and pl[3:3 + len(pool)] == pool, "pool"
            op.check_coverage(lens, *got, home_end, pool)


def test_dynamic_plan_random_configs():
    """Many seeded (lengths, CTAs, min_tiles, pool) draws: every divisor the
    planner sets up a multiplicative inverse for (range, chunk, pieces per
    range) takes many values, including ranges near 2^31 from a huge
    min_tiles."""
    gu.require_gpu()
    rng = np.random.default_rng(11)
    for trial in range(160):
        B = int(rng.choice([1, 2, 5, 33, 200]))
        hi = int(rng.choice([100, 5000, 300000]))
        lens = [int(x) for x in rng.integers(0, hi, size=B)]
        C = int(rng.choice([1, 3, 152, 999, 4096]))
        min_tiles = int(rng.choice([1, 1, 3, 1000003, 2 ** 30 + 12345, 2 ** 31 - 1]))
        J = int(rng.choice([0, 1, 3, 4, 64]))
        kmin = int(rng.choice([1, 16]))
        plan, st = _run_dynamic(lens, C, min_tiles, J=J, kmin=kmin)
        assert st == 0
        items, cta_ptr, seg_ptr, home_end, pool = op.plan_dynamic(lens, C, min_tiles, J, kmin)
        got = _host(plan, len(items))
        ctx = (trial, B, C, min_tiles, J, kmin)
        assert got[0] == [tuple(i) for i in items], ctx
        assert got[1] == cta_ptr and got[2] == seg_ptr, ctx
        assert plan.home_end.cpu().tolist() == home_end, ctx
        pl = plan.pool.cpu().tolist()
        assert pl[:3] == [0, 0, len(pool)] and pl[3:3 + len(pool)] == pool, ctx


@pytest.mark.parametrize("S", [1, 2, 3, 64])
def test_static_plan_bit_exact(S):
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    for lens in _mixes():
        B = len(lens)
        if B * 8 * S > 400000:
            continue
        max_blocks = max(1, max(-(-L // 64) for L in lens))
        plan = ops.DecodePlan.static(B, S, "cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ops.decode_plan_static(torch.tensor(lens, dtype=torch.int32, device="cuda"), max_blocks,
                               S, plan, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        items, cta_ptr, seg_ptr, C = op.plan_static(lens, S)
        got = _host(plan, len(items))
        assert got[0] == [tuple(i) for i in items]
        assert got[1] == cta_ptr and got[2] == seg_ptr
        assert plan.home_end.cpu().tolist() == [min(c + 1, len(items)) for c in range(C)]
        assert plan.pool.cpu().tolist()[:3] == [0, 0, 0]
        op.check_coverage(lens, *got)


def test_plan_overflow_and_bad_lengths_set_status():
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    lens = [4096] * 32
    plan, st = _run_dynamic(lens, 152, 1, capacity=10)
    assert st & 16, "PLAN_OVERFLOW"
    assert plan.cta_ptr.cpu().tolist() == [0] * 153      # empty plan
    # a length beyond max_blocks*64 and a negative one are treated as empty
    B = 3
    plan = ops.DecodePlan(B, 16, 16 + 24, "cuda")       # no pool chunks
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.decode_plan(torch.tensor([100, 10 ** 6, -5], dtype=torch.int32, device="cuda"), 4, plan,
                    status, 1)
    torch.cuda.synchronize()
    assert int(status.item()) & 4, "BAD_SEQ_LEN"
    want = op.plan_dynamic([100, 0, 0], 16, 1)[:3]
    got = _host(plan, len(want[0]))
    assert got[0] == [tuple(i) for i in want[0]] and got[1] == want[1] and got[2] == want[2]
