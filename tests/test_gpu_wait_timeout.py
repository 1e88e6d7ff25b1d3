"""Failure detection without a fault: the pipeline's bounded wait (and its
polling form) runs out on barrier phases nothing completes, the kernel records
WAIT_TIMEOUT and returns, and the same context then runs a decode step
normally."""

import pytest
import torch

import gpu_util as gu

pytestmark = pytest.mark.gpu

HPC_STATUS_WAIT_TIMEOUT = 32


def test_bounded_wait_times_out_and_context_survives():
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 2_000_000                                   # 2 ms
    ops.selftest_wait_timeout(limit, status, waited)
    torch.cuda.synchronize()
    assert int(status.item()) & HPC_STATUS_WAIT_TIMEOUT
    assert limit <= int(waited.item()) < 1_000_000_000

    # the context is still usable: a full decode step afterwards is correct
    wl = Workload("tiny", seed=0)
    cos_sin = ops.rope_cos_sin_cache(wl.max_pos + 1)
    step = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks)
    out = step(wl.q, wl.k, wl.v, wl.positions, cos_sin, wl.q_norm_w, wl.k_norm_w, wl.cache,
               wl.slot_mapping, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.isfinite(out.float()).all()


def test_bounded_polling_wait_times_out_and_context_survives():
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 2_000_000                                   # 2 ms
    ops.selftest_poll_timeout(limit, status, waited)
    torch.cuda.synchronize()
    assert int(status.item()) & HPC_STATUS_WAIT_TIMEOUT
    assert limit <= int(waited.item()) < 1_000_000_000

    # the context is still usable: multi-token decode (the tensor-core form
    # whose MMA warp polls) runs correctly afterwards
    wl = Workload("custom", seed=11, lengths=[300, 1, 4096], kv_dtype=1, include_new_token=True)
    q = torch.randn((wl.batch, 4, 64, 128), device="cuda").to(torch.bfloat16)
    step = ops.DecodeStepMT(wl.batch, 4, wl.kv_dtype, wl.max_blocks)
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.isfinite(out.float()).all()
