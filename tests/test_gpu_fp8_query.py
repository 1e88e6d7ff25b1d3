"""E4M3 query (q quantised to E4M3 codes, its products with the E4M3 cache
on the tensor cores) and the caller-chosen output type, against the float64
oracle on the same dequantised values."""


import numpy as np
import pytest
import torch

from oracle import decode as od
from oracle import numerics as nx
import gpu_util as gu

pytestmark = pytest.mark.gpu

LENGTHS = [1, 2, 63, 64, 65, 300, 4097, 9000]


def _q_codes(B, qn, seed):
    """E4M3 codes of a N(0,1) q with a per-tensor scale max|q|/448 (host)."""
    rng = np.random.default_rng(seed)
    qf = rng.standard_normal((B, qn, 64, 128))
    scale = float(np.abs(qf).max() / 448.0)
    codes = od.encode_kv(qf, od.KV_FP8, scale).astype(np.uint8)
    return codes, scale


def _oracle_mt(wl, qvals, b, heads=None):
    L = int(wl.lengths[b])
    sub, row = gu.seq_view(wl.cache, wl.block_table_np[b], L, wl.kv_dtype)
    sc = wl.kv_scale.cpu().numpy().astype(np.float64)
    return od.decode_attention_mt(qvals[b], sub, row, L, wl.kv_dtype, sc[0], sc[1], heads=heads)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("q_len", [1, 2, 3, 4])
def test_fp8_query_attention_matches_oracle(q_len, fused):
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=80 + q_len, lengths=LENGTHS, kv_dtype=od.KV_FP8,
                  include_new_token=True)
    codes, qs = _q_codes(wl.batch, q_len, 3 + q_len)
    q = torch.as_tensor(codes, device="cuda")
    qvals = od.decode_kv(codes, od.KV_FP8, qs)
    step = ops.DecodeStepEx(wl.batch, od.KV_FP8, wl.max_blocks, q_len=q_len, q_dtype=ops.Q_FP8,
                            q_scale=qs, fused=fused)
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got = gu.bf16_host(out)
    assert np.all(np.isfinite(got))
    for b in range(wl.batch):
        gu.compare(got[b], _oracle_mt(wl, qvals, b), gu.TOL_FP8_MAX, None,
                   label="q_len %d seq %d (L=%d)" % (q_len, b, wl.lengths[b]))


def test_fp8_query_queue_count_follows_the_form():
    """An E4M3 q at q_len 2 on an E4M3 cache runs the tensor-core form (two
    queues per CTA), a BF16 q at q_len 2 the 2-token mma.sync layout (three),
    and q_len 3-4 the tensor-core form for both q types."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ops.num_ctas(od.KV_FP8, 2, ops.Q_FP8) == 2 * sms
    assert ops.num_ctas(od.KV_FP8, 2, ops.Q_BF16) == 3 * sms
    assert ops.num_ctas(od.KV_FP8, 1, ops.Q_FP8) == 3 * sms
    for qn in (3, 4):
        for qd in (ops.Q_BF16, ops.Q_FP8):
            assert ops.num_ctas(od.KV_FP8, qn, qd) == 2 * sms
    assert ops.num_ctas(od.KV_BF16, 2, ops.Q_BF16) == 2 * sms


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("q_len", [2, 4])
def test_fp8_query_bad_block_is_reported_and_skipped(q_len, fused):
    """A block id past the cache under an E4M3 q (the tensor-core form): the
    status says BAD_BLOCK, the other sequences match the oracle and the bad
    sequence's outputs stay finite."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=40 + q_len, lengths=[300, 200, 4097, 70], kv_dtype=od.KV_FP8,
                  include_new_token=True)
    wl.block_table[1, 2] = wl.num_blocks + 5          # tile 2 of sequence 1 points past the cache
    codes, qs = _q_codes(wl.batch, q_len, 50 + q_len)
    q = torch.as_tensor(codes, device="cuda")
    qvals = od.decode_kv(codes, od.KV_FP8, qs)
    step = ops.DecodeStepEx(wl.batch, od.KV_FP8, wl.max_blocks, q_len=q_len, q_dtype=ops.Q_FP8,
                            q_scale=qs, fused=fused)
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) & 1, "BAD_BLOCK"
    got = gu.bf16_host(out)
    assert np.all(np.isfinite(got[1]))
    for b in (0, 2, 3):
        gu.compare(got[b], _oracle_mt(wl, qvals, b), gu.TOL_FP8_MAX, None, label="seq %d" % b)


@pytest.mark.parametrize("q_len", [1, 2])
def test_fp8_query_full_mixed(q_len):
    """The E4M3 q on the full mixed FP8 batch, sampled rows (q_len 2 runs the
    tensor-core form)."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("mixed_fp8", seed=4, include_new_token=True)
    codes, qs = _q_codes(wl.batch, q_len, 17 + q_len)
    q = torch.as_tensor(codes, device="cuda")
    qvals = od.decode_kv(codes, od.KV_FP8, qs)
    step = ops.DecodeStepEx(wl.batch, od.KV_FP8, wl.max_blocks, q_len=q_len, q_dtype=ops.Q_FP8,
                            q_scale=qs)
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got = gu.bf16_host(out)
    for b in (0, 5, 31):
        heads = list(range(0, 64, 9)) if wl.lengths[b] > 65536 else None
        gu.compare(got[b], _oracle_mt(wl, qvals, b, heads), gu.TOL_FP8_MAX, None, label="seq %d" % b)


@pytest.mark.parametrize("kv", [0, 1])
def test_output_types(kv):
    """FP32, FP16 and BF16 outputs of one run: the FP32 output matches the
    oracle, and the FP16 / BF16 outputs are the FP32 values rounded to nearest
    (fused and standalone merges alike)."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=90 + kv, lengths=[5, 64, 700, 5000], kv_dtype=kv,
                  include_new_token=True)
    g = torch.Generator(device="cuda").manual_seed(2)
    q = torch.randn((wl.batch, 2, 64, 128), generator=g, device="cuda").to(torch.bfloat16)
    outs = {}
    for fused in (True, False):
        for od_ in (ops.OUT_FP32, ops.OUT_FP16, ops.OUT_BF16):
            step = ops.DecodeStepEx(wl.batch, kv, wl.max_blocks, q_len=2, out_dtype=od_, fused=fused)
            step.plan_step(wl.seq_lens)
            outs[(fused, od_)] = step.attend(q, wl.cache, wl.kv_scale, wl.block_table,
                                             wl.seq_lens).clone()
            torch.cuda.synchronize()
            assert int(step.status.item()) == 0
    for fused in (True, False):
        f32 = outs[(fused, ops.OUT_FP32)]
        assert outs[(fused, ops.OUT_FP32)].dtype == torch.float32
        assert torch.equal(outs[(fused, ops.OUT_FP16)], f32.to(torch.float16))
        assert torch.equal(outs[(fused, ops.OUT_BF16)], f32.to(torch.bfloat16))
    qv = gu.bf16_host(q)
    got = outs[(True, ops.OUT_FP32)].cpu().numpy().astype(np.float64)
    tol = (gu.TOL_BF16_MAX, gu.TOL_BF16_MEAN) if kv == 0 else (gu.TOL_FP8_MAX, None)
    for b in range(wl.batch):
        gu.compare(got[b], _oracle_mt(wl, qv, b), *tol, label="fp32 out seq %d" % b)


def test_fp8_query_step_end_to_end():
    """Prologue storing E4M3 q codes (within one code of the oracle's), plan
    and attention against the oracle on the cache and q codes the GPU wrote."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    qn = 2
    wl = Workload("custom", seed=95, lengths=[2, 64, 65, 1000], kv_dtype=od.KV_FP8)
    B = wl.batch
    g = torch.Generator(device="cuda").manual_seed(13)
    q = torch.randn((B, qn, 64, 128), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, qn, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, qn, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
    pos = np.array([[L - qn + t for t in range(qn)] for L in wl.lengths], dtype=np.int32)
    slots = np.array([[wl.block_table_np[b][p // 64] * 64 + p % 64 for p in pos[b]]
                      for b in range(B)], dtype=np.int64)
    cos_sin = ops.rope_cos_sin_cache(int(wl.lengths.max()) + 1)
    qs = 0.02
    step = ops.DecodeStepEx(B, od.KV_FP8, wl.max_blocks, q_len=qn, q_dtype=ops.Q_FP8, q_scale=qs)
    out = step(q, k, v, torch.as_tensor(pos, device="cuda"), cos_sin, wl.q_norm_w, wl.k_norm_w,
               wl.cache, torch.as_tensor(slots, device="cuda"), wl.kv_scale, wl.block_table,
               wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got = gu.bf16_host(out)
    codes = step.q_out.cpu().numpy()
    qh, kh, vh = gu.bf16_host(q), gu.bf16_host(k), gu.bf16_host(v)
    qw, kw = gu.bf16_host(wl.q_norm_w), gu.bf16_host(wl.k_norm_w)
    for b in range(B):
        for t in range(qn):
            qo, _, _ = od.prologue_token(qh[b, t], kh[b, t], vh[b, t], int(pos[b, t]), qw, kw)
            mine = od.decode_kv(od.encode_kv(qo, od.KV_FP8, qs), od.KV_FP8, 1.0)
            gpu = od.decode_kv(codes[b, t], od.KV_FP8, 1.0)
            assert np.all(np.abs(gpu - mine) <= nx.e4m3_step(np.maximum(np.abs(gpu), np.abs(mine))))
    qvals = od.decode_kv(codes, od.KV_FP8, qs)
    for b in range(B):
        gu.compare(got[b], _oracle_mt(wl, qvals, b), gu.TOL_FP8_MAX, None, label="step seq %d" % b)
