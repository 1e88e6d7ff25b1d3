"""End to end: fused prologue -> plan -> attention -> merge vs the oracle's own
prologue, cache write and attention (on host copies taken before the step)."""

import numpy as np
import pytest
import torch

from oracle import decode as od
import gpu_util as gu

pytestmark = pytest.mark.gpu


def _step_vs_oracle(wl, seqs, two_launch, label):
    """One step over the workload; the sampled sequences against the oracle's
    prologue, cache write and attention on host copies of their pages taken
    before the step."""
    from paged_gqa_decode_rope_gb300 import ops
    views = {b: gu.seq_view(wl.cache, wl.block_table_np[b], int(wl.lengths[b]), wl.kv_dtype)
             for b in seqs}
    cos_sin = ops.rope_cos_sin_cache(wl.max_pos + 1)
    step = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks)
    out = step(wl.q, wl.k, wl.v, wl.positions, cos_sin, wl.q_norm_w, wl.k_norm_w, wl.cache,
               wl.slot_mapping, wl.kv_scale, wl.block_table, wl.seq_lens, two_launch=two_launch)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got = gu.bf16_host(out)
    assert np.all(np.isfinite(got)), "%s: NaN/inf in outputs" % label
    q, k, v = gu.bf16_host(wl.q), gu.bf16_host(wl.k), gu.bf16_host(wl.v)
    qw, kw = gu.bf16_host(wl.q_norm_w), gu.bf16_host(wl.k_norm_w)
    scale = wl.kv_scale.cpu().numpy().astype(np.float64)
    tol = (gu.TOL_BF16_MAX, gu.TOL_BF16_MEAN) if wl.kv_dtype == od.KV_BF16 else (gu.TOL_FP8_MAX, None)
    wants = []
    for b in seqs:
        L = int(wl.lengths[b])
        sub, row = views[b]
        slot = (L - 1) // 64 * 64 + (L - 1) % 64          # the new token's slot in the view
        q_out, want = od.decode_step(q[b:b + 1], k[b:b + 1], v[b:b + 1], [L - 1], qw, kw, sub,
                                     row[None, :], [L], [slot], wl.kv_dtype, scale)
        wants.append(want[0])
    # the bounds hold over every output of the checked sequences together
    gu.compare(got[list(seqs)], np.stack(wants), *tol, label="%s, %d sequences" % (label, len(seqs)))


@pytest.mark.parametrize("name,two_launch", [("tiny", True), ("tiny", False), ("mixed", True),
                                             ("mixed", False), ("heavy_tail", True)])
def test_decode_step_end_to_end(name, two_launch):
    """The whole step on every sequence of the workload: the oracle's own
    prologue, cache write and attention against the GPU step, over all
    batch x 64 x 128 outputs."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload(name, seed=0)                 # history holds tokens 0 .. L-2
    _step_vs_oracle(wl, list(range(wl.batch)), two_launch, name)


@pytest.mark.parametrize("kv", [0, 1])
def test_decode_step_at_the_batch_limit(kv):
    """The whole step for HPC_MAX_BATCH (8192) sequences of ragged lengths
    1 .. 129: 73 729 prologue blocks beside the planner block, 8192 new tokens
    written into the cache, then the attention and merge."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300.workloads import Workload
    rng = np.random.default_rng(31 + kv)
    wl = Workload("custom", seed=31 + kv, lengths=rng.integers(1, 130, 8192).tolist(), kv_dtype=kv)
    seqs = sorted(set(rng.choice(8192, 6, replace=False).tolist()) | {0, 8191})
    _step_vs_oracle(wl, seqs, True, "batch limit kv %d" % kv)


@pytest.mark.parametrize("two_launch", [True, False])
def test_decode_step_in_cuda_graph(two_launch):
    """The step is capturable: graph replays give the eager step's output bit
    for bit (the step is deterministic), and replays of a captured plan reset
    their own counters."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("mixed", seed=1)
    cos_sin = ops.rope_cos_sin_cache(wl.max_pos + 1)
    step = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks)

    def run():
        return step(wl.q, wl.k, wl.v, wl.positions, cos_sin, wl.q_norm_w, wl.k_norm_w, wl.cache,
                    wl.slot_mapping, wl.kv_scale, wl.block_table, wl.seq_lens,
                    two_launch=two_launch)

    eager = run().clone()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        run()                                    # warm on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            out = run()
    step.out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(out, eager)
