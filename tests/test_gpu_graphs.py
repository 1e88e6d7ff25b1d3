"""CUDA-graph capture of the prefill and multi-token calls: every call is
asynchronous on the caller's stream and allocates nothing, so a captured
plan + attention replays to the eager result bit for bit, and replays reset
their own claim counters (a plan can run again)."""

import numpy as np
import pytest
import torch

import gpu_util as gu

pytestmark = pytest.mark.gpu


def _capture(fn):
    """fn() run once eagerly on a side stream (warm-up: attribute opt-ins and
    map encoders resolved), then captured; returns the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("kv", [0, 1])
def test_prefill_plan_and_attention_in_a_graph(kv):
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    lengths = [1, 65, 300, 1000, 2200]
    q_lens = [1, 65, 37, 200, 33]
    wl = Workload("custom", seed=51 + kv, lengths=lengths, kv_dtype=kv, include_new_token=True)
    qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    qst = torch.as_tensor(qs, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(51)
    q = torch.randn((int(qs[-1]), 64, 128), generator=gen, device="cuda").to(torch.bfloat16)
    pf = ops.PrefillAttention(wl.batch)
    eager = torch.empty_like(q)
    pf.plan(qst)
    pf(q, qst, wl.cache, kv, wl.kv_scale, wl.block_table, wl.seq_lens, eager)
    torch.cuda.synchronize()
    out = torch.empty_like(q)

    def run():
        pf.plan(qst)
        pf(q, qst, wl.cache, kv, wl.kv_scale, wl.block_table, wl.seq_lens, out)

    g = _capture(run)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(pf.status.item()) == 0
    assert int(pf.counters.abs().sum().item()) == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("q_len,kv", [(2, 0), (4, 1)])
def test_multi_token_plan_and_attention_in_a_graph(q_len, kv):
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=61 + kv, lengths=[3, 64, 65, 1000, 5000, 20000], kv_dtype=kv,
                  include_new_token=True)
    gen = torch.Generator(device="cuda").manual_seed(61)
    q = torch.randn((wl.batch, q_len, 64, 128), generator=gen, device="cuda").to(torch.bfloat16)
    step = ops.DecodeStepMT(wl.batch, q_len, kv, wl.max_blocks)
    step.plan_step(wl.seq_lens)
    eager = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens).clone()
    torch.cuda.synchronize()

    def run():
        step.plan_step(wl.seq_lens)
        step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)

    g = _capture(run)
    step.out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(step.out.view(torch.int16), eager.view(torch.int16))
