"""Multi-token decode (q_len = 2 .. 4 new tokens per sequence) against the
float64 oracle: each new token sees the history and the new tokens up to
itself.  Lengths include sequences shorter than q_len (whose first new tokens
see no key and must give zeros) and lengths around the 64-token tile edges;
unused cache entries are NaN, so a key read past a token's causal limit
shows up as a non-finite output."""

import numpy as np
import pytest
import torch

from oracle import decode as od
import gpu_util as gu

pytestmark = pytest.mark.gpu

LENGTHS = [1, 2, 3, 4, 63, 64, 65, 66, 130, 300, 4097, 5000]


def _q(B, qn, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn((B, qn, 64, 128), generator=g, device="cuda").to(torch.bfloat16)


def _oracle(wl, q, b, heads=None):
    L = int(wl.lengths[b])
    sub, row = gu.seq_view(wl.cache, wl.block_table_np[b], L, wl.kv_dtype)
    sc = wl.kv_scale.cpu().numpy().astype(np.float64)
    return od.decode_attention_mt(gu.bf16_host(q[b]), sub, row, L, wl.kv_dtype, sc[0], sc[1],
                                  heads=heads)


def _tol(kv):
    return (gu.TOL_BF16_MAX, gu.TOL_BF16_MEAN) if kv == od.KV_BF16 else (gu.TOL_FP8_MAX, None)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("kv", [0, 1])
@pytest.mark.parametrize("q_len", [2, 3, 4])
def test_multi_token_attention_matches_oracle(q_len, kv, fused):
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=40 + q_len, lengths=LENGTHS, kv_dtype=kv, include_new_token=True)
    q = _q(wl.batch, q_len, 7 + q_len)
    step = ops.DecodeStepMT(wl.batch, q_len, kv, wl.max_blocks, fused=fused)
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got = gu.bf16_host(out)
    assert np.all(np.isfinite(got))
    for b in range(wl.batch):
        want = _oracle(wl, q, b)
        gu.compare(got[b], want, *_tol(kv), label="q_len %d kv %d seq %d (L=%d)"
                   % (q_len, kv, b, wl.lengths[b]))
        for t in range(q_len):   # tokens that see no key give exact zeros
            if wl.lengths[b] - q_len + 1 + t <= 0:
                assert np.all(got[b, t] == 0.0)


@pytest.mark.parametrize("kv", [0, 1])
@pytest.mark.parametrize("q_len", [2, 4])
def test_multi_token_pooled_plan_and_reproducible(q_len, kv):
    """A plan with many pooled chunks (many items per segment, merged by the
    last queue to finish) gives the unpooled result within the split
    tolerance, and two runs of one plan are bit-identical."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    # long enough for pooled chunks on either grid (304 BF16 or 456 FP8 queues)
    wl = Workload("custom", seed=61, lengths=[60000, 300, 7, 4096, 1], kv_dtype=kv,
                  include_new_token=True)
    q = _q(wl.batch, q_len, 99)
    ref = ops.DecodeStepMT(wl.batch, q_len, kv, wl.max_blocks, pool_chunks=0)
    ref.plan_step(wl.seq_lens)
    a = ref.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens).clone()
    pooled = ops.DecodeStepMT(wl.batch, q_len, kv, wl.max_blocks, pool_chunks=3, pool_min_tiles=1)
    pooled.plan_step(wl.seq_lens)
    b1 = pooled.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens).clone()
    b2 = pooled.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens).clone()
    torch.cuda.synchronize()
    assert int(ref.status.item()) == 0 and int(pooled.status.item()) == 0
    assert int(pooled.plan.pool[2].item()) > 0
    assert torch.equal(b1.view(torch.int16), b2.view(torch.int16))
    d = (a.float() - b1.float()).abs()
    assert float(d.max()) <= 4e-3 and float(d.mean()) <= 2e-4
    got = gu.bf16_host(b1)
    gu.compare(got[0], _oracle(wl, q, 0, heads=list(range(0, 64, 7))), *_tol(kv), label="seq 0")
    gu.compare(got[1:], np.stack([_oracle(wl, q, b) for b in range(1, wl.batch)]), *_tol(kv),
               label="seqs 1..")


@pytest.mark.parametrize("name,q_len", [("mixed", 2), ("mixed_fp8", 4)])
def test_multi_token_mixed_full_size(name, q_len):
    """Multi-token decode on the full mixed batch (1 x 128K + 31 x 4K tokens),
    BF16 at q_len 2 and FP8 at q_len 4, in the launch configuration of the
    benchmark; every output row against the oracle, the bounds over all of
    them."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload(name, seed=3, include_new_token=True)
    q = _q(wl.batch, q_len, 5)
    step = ops.DecodeStepMT(wl.batch, q_len, wl.kv_dtype, wl.max_blocks)
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got = gu.bf16_host(out)
    assert np.all(np.isfinite(got))
    want = np.stack([_oracle(wl, q, b) for b in range(wl.batch)])
    gu.compare(got, want, *_tol(wl.kv_dtype), label="%s q_len %d" % (name, q_len))


@pytest.mark.parametrize("kv", [0, 1])
def test_multi_token_step_end_to_end(kv):
    """Prologue of every new token (its own position and slot), plan and
    attention.  The stored q and the written K/V codes match the oracle's
    multi-token step (q within one BF16 ulp, cache codes within one code: the
    fp32 and fp64 roundings may part at a tie), and the attention matches the
    oracle run on the cache bytes the GPU wrote; for BF16 the whole step also
    matches the oracle's own end-to-end composition."""
    gu.require_gpu()
    from oracle import numerics as nx
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    qn = 3
    wl = Workload("custom", seed=70 + kv, lengths=[3, 64, 65, 700, 2049], kv_dtype=kv)
    B = wl.batch
    q = _q(B, qn, 11)
    g = torch.Generator(device="cuda").manual_seed(12)
    k = torch.randn((B, qn, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, qn, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
    pos = np.array([[L - qn + t for t in range(qn)] for L in wl.lengths], dtype=np.int32)
    slots = np.array([[wl.block_table_np[b][p // 64] * 64 + p % 64 for p in pos[b]]
                      for b in range(B)], dtype=np.int64)
    positions = torch.as_tensor(pos, device="cuda")
    slot_mapping = torch.as_tensor(slots, device="cuda")
    cos_sin = ops.rope_cos_sin_cache(int(wl.lengths.max()) + 1)
    before = [gu.seq_view(wl.cache, wl.block_table_np[b], int(wl.lengths[b]), kv) for b in range(B)]
    step = ops.DecodeStepMT(B, qn, kv, wl.max_blocks)
    out = step(q, k, v, positions, cos_sin, wl.q_norm_w, wl.k_norm_w, wl.cache, slot_mapping,
               wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got = gu.bf16_host(out)
    q_gpu = gu.bf16_host(step.q_out)
    qh, kh, vh = gu.bf16_host(q), gu.bf16_host(k), gu.bf16_host(v)
    qw, kw = gu.bf16_host(wl.q_norm_w), gu.bf16_host(wl.k_norm_w)
    sc = wl.kv_scale.cpu().numpy().astype(np.float64)
    for b in range(B):
        L = int(wl.lengths[b])
        sub, row = before[b]
        mine = sub.copy()
        local = [[row[p // 64] * 64 + p % 64 for p in pos[b]]]
        q_ref, want = od.decode_step_mt(qh[b:b + 1], kh[b:b + 1], vh[b:b + 1], pos[b:b + 1], qw, kw,
                                        mine, row[None, :], [L], local, kv, sc)
        # the stored q and the written codes
        ulp = np.abs(q_gpu[b] - q_ref[0]) / np.maximum(np.abs(q_ref[0]), 1e-30)
        assert np.all(ulp <= 2.0 ** -7), "q_out of seq %d" % b
        after, _ = gu.seq_view(wl.cache, wl.block_table_np[b], L, kv)
        for p_ in pos[b]:
            blk, off = divmod(int(p_), 64)
            a_ = after[blk, :, :, off].astype(np.int64)
            m_ = mine[blk, :, :, off].astype(np.int64)
            if kv == od.KV_BF16:
                assert np.max(np.abs(a_ - m_)) <= 1, "bf16 code of seq %d pos %d" % (b, p_)
            else:
                da = od.decode_kv(after[blk, :, :, off], kv, 1.0)
                dm = od.decode_kv(mine[blk, :, :, off], kv, 1.0)
                assert np.all(np.abs(da - dm) <= nx.e4m3_step(np.maximum(np.abs(da), np.abs(dm))) + 0.0)
        # attention on the cache the GPU wrote, with the GPU's q
        att = od.decode_attention_mt(q_gpu[b], after, row, L, kv, sc[0], sc[1])
        gu.compare(got[b], att, *_tol(kv), label="attention kv %d seq %d (L=%d)" % (kv, b, L))
        if kv == od.KV_BF16:
            gu.compare(got[b], want[0], *_tol(kv), label="step seq %d (L=%d)" % (b, L))


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("kv", [0, 1])
@pytest.mark.parametrize("q_len", [3, 4])
def test_multi_token_bad_block_is_reported_and_skipped(q_len, kv, fused):
    """A block id past the cache (the 4-token layout's tensor-core form): the
    status says BAD_BLOCK, the other sequences are exact to the oracle, and
    the bad sequence's outputs stay finite."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=60 + q_len, lengths=[300, 200, 4097, 70], kv_dtype=kv,
                  include_new_token=True)
    wl.block_table[1, 2] = wl.num_blocks + 5          # tile 2 of sequence 1 points past the cache
    q = _q(wl.batch, q_len, 70 + q_len)
    step = ops.DecodeStepMT(wl.batch, q_len, kv, wl.max_blocks, fused=fused)
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) & 1, "BAD_BLOCK"
    got = gu.bf16_host(out)
    assert np.all(np.isfinite(got[1]))
    for b in (0, 2, 3):
        gu.compare(got[b], _oracle(wl, q, b), *_tol(kv), label="seq %d" % b)


@pytest.mark.parametrize("q_len", [3, 4])
def test_multi_token_e4m3_pages_wide_range_q(q_len):
    """Over E4M3 pages the 4-token layout's Q K^T runs on E4M3 products, a BF16
    q split per row into two E4M3 terms under a power-of-two row scale.  The
    split is exact for elements within 2^10 of the row's largest and off by at
    most 2^-17 of it below that.  Rows whose elements span 2^-20 .. 2^4 (and
    whole rows of zeros) must still match the float64 oracle within the FP8
    tolerance."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=80 + q_len, lengths=[300, 4097, 65, 1], kv_dtype=1,
                  include_new_token=True)
    rng = np.random.default_rng(90 + q_len)
    mag = np.exp2(rng.uniform(-20.0, 4.0, size=(wl.batch, q_len, 64, 128)))
    qf = rng.standard_normal((wl.batch, q_len, 64, 128)) * mag
    qf[0, 0, 3, :] = 0.0                        # a row of zeros
    q = torch.as_tensor(qf, dtype=torch.float32, device="cuda").to(torch.bfloat16)
    step = ops.DecodeStepMT(wl.batch, q_len, 1, wl.max_blocks)
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got = gu.bf16_host(out)
    assert np.all(np.isfinite(got))
    for b in range(wl.batch):
        gu.compare(got[b], _oracle(wl, q, b), *_tol(1), label="seq %d (L=%d)" % (b, wl.lengths[b]))
