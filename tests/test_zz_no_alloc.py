"""The no-allocation entry point (hpc_decode_attn_merge_noalloc).

It serves callers that cannot allocate device memory: the split-KV scratch
lives in the library's own device array instead of caller buffers.  Called
through the C ABI, twice in a row on different batches (so that anything the
first call left in the shared array would show up in the second), its output
must match the allocating path (hpc_decode_attn + hpc_merge with
caller-owned partials) within the attention tolerance used by the other
tests, and the float64 oracle on every output row.  Collected last on
purpose; it also passes alone in a fresh process.
"""

import ctypes
import math

import pytest
import torch

import gpu_util as gu

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, wl, plan, out, status):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.hpc_decode_attn_merge_noalloc(
        _p(wl.q), _p(wl.cache), wl.kv_dtype, _p(wl.kv_scale), wl.num_blocks, _p(wl.block_table),
        wl.max_blocks, _p(wl.seq_lens), wl.batch, ctypes.byref(plan.c), _p(out),
        1.0 / math.sqrt(128), _p(status), stream)


def _allocating(wl):
    from paged_gqa_decode_rope_gb300 import ops
    step = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks)
    step.plan_step(wl.seq_lens)
    out = step.attend(wl.q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens).clone()
    return step, out


def test_noalloc_matches_allocating_path_on_two_calls_in_a_row():
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import _lib
    from paged_gqa_decode_rope_gb300.workloads import Workload
    lib = _lib.lib()
    batches = [
        Workload("mixed", seed=21, include_new_token=True),                      # BF16, 408 items
        Workload("custom", seed=22, lengths=[1, 63, 64, 300, 5000, 17, 2049],    # FP8, other plan
                 kv_dtype=1, include_new_token=True),
    ]
    for wl in batches:
        step, ref = _allocating(wl)             # the plan of this batch, and the reference
        out = torch.full_like(ref, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert step.plan.capacity <= _lib.NOALLOC_MAX_ITEMS
        assert _noalloc(lib, wl, step.plan, out, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got, want = gu.bf16_host(out), gu.bf16_host(ref)
        tol = (gu.TOL_BF16_MAX, gu.TOL_BF16_MEAN) if wl.kv_dtype == 0 else (gu.TOL_FP8_MAX, None)
        gu.compare(got, want, *tol, label="noalloc vs allocating, %s" % wl.name)
        gu.compare(got, gu.oracle_outputs(wl, wl.q, range(wl.batch)), *tol,
                   label="noalloc vs oracle, %s" % wl.name)


def test_noalloc_rejects_a_plan_beyond_its_array():
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import _lib, ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    lib = _lib.lib()
    wl = Workload("custom", seed=23, lengths=[100, 200], kv_dtype=0, include_new_token=True)
    plan = ops.DecodePlan(wl.batch, 152, _lib.NOALLOC_MAX_ITEMS + 1, "cuda")
    out = torch.zeros((wl.batch, 64, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, wl, plan, out, status) == _lib.HPC_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and bool((out == 0).all()), "nothing was launched"
