"""Prefill and mixed prefill + decode batches through the same paged cache,
against the float64 oracle (each new token sees its history and the new
tokens up to itself).  The cache holds every token of every sequence (the new
ones included) and NaN elsewhere, so any read past a sequence's length shows
up as a non-finite output."""

import numpy as np
import pytest
import torch

from oracle import decode as od
import gpu_util as gu

pytestmark = pytest.mark.gpu


def _batch(lengths, q_lens, seed, kv_dtype=0):
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=seed, lengths=lengths, kv_dtype=kv_dtype, include_new_token=True)
    qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((int(qs[-1]), 64, 128), generator=g, device="cuda").to(torch.bfloat16)
    return wl, q, torch.as_tensor(qs, device="cuda"), qs


def _check(wl, q, qs, out, seqs=None, heads=None, tol=None):
    """Against the oracle over the cache as it is on the device (an E4M3
    cache through the oracle's own decoder and the per-tensor scales)."""
    if tol is None:
        tol = (gu.TOL_BF16_MAX, gu.TOL_BF16_MEAN) if wl.kv_dtype == 0 else (gu.TOL_FP8_MAX, None)
    ks, vs = [float(x) for x in wl.kv_scale.cpu().numpy()] if wl.kv_dtype == 1 else (1.0, 1.0)
    got = out.float().cpu().numpy().astype(np.float64)
    qh = gu.bf16_host(q)
    for b in (range(wl.batch) if seqs is None else seqs):
        a, e = int(qs[b]), int(qs[b + 1])
        if e == a:
            continue
        L = int(wl.lengths[b])
        sub, row = gu.seq_view(wl.cache, wl.block_table_np[b], L, wl.kv_dtype)
        want = od.decode_attention_mt(qh[a:e], sub, row, L, wl.kv_dtype, ks, vs, heads=heads)
        gu.compare(got[a:e], want, *tol, label="seq %d (L=%d, q_len=%d)" % (b, L, e - a))


def test_prefill_at_the_batch_limit():
    """HPC_MAX_BATCH (8192) sequences, each with 1 .. 3 new tokens after a
    ragged history (the decode side of a mixed batch at its largest): 64K
    units dealt to the persistent grid; sampled sequences against the oracle."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    rng = np.random.default_rng(21)
    q_lens = rng.integers(1, 4, 8192)
    lengths = (q_lens + rng.integers(0, 127, 8192)).tolist()
    wl, q, qst, qs = _batch(lengths, q_lens.tolist(), 21)
    pf = ops.PrefillAttention(wl.batch)
    pf.plan(qst)
    out = torch.empty_like(q)
    pf(q, qst, wl.cache, 0, wl.kv_scale, wl.block_table, wl.seq_lens, out)
    torch.cuda.synchronize()
    assert int(pf.status.item()) == 0
    assert int(pf.counters.abs().sum().item()) == 0
    assert torch.isfinite(out.float()).all()
    seqs = sorted(set(rng.choice(8192, 8, replace=False).tolist()) | {0, 8191})
    _check(wl, q, qs, out, seqs=seqs)


def test_prefill_prompts_and_chunks():
    """Whole prompts (q_len = L, tile and block edges) and chunks after a
    history, one launch; a second launch of the same plan gives the same bits."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    lengths = [1, 16, 17, 64, 65, 130, 300, 1000, 2200]
    q_lens = [1, 16, 17, 64, 65, 130, 37, 200, 33]
    wl, q, qst, qs = _batch(lengths, q_lens, 5)
    pf = ops.PrefillAttention(wl.batch)
    pf.plan(qst)
    out = torch.empty_like(q)
    pf(q, qst, wl.cache, 0, wl.kv_scale, wl.block_table, wl.seq_lens, out)
    again = pf(q, qst, wl.cache, 0, wl.kv_scale, wl.block_table, wl.seq_lens, torch.empty_like(q))
    torch.cuda.synchronize()
    assert int(pf.status.item()) == 0
    assert int(pf.counters.abs().sum().item()) == 0
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    assert torch.isfinite(out.float()).all()
    _check(wl, q, qs, out)


def test_mixed_batch_prefill_and_decode_kernels_on_one_cache():
    """A mixed batch: decode sequences (one new token, long histories) through
    the split-KV decode path, prompt chunks through the prefill kernel; both
    over the one cache, both against the oracle; the prefill kernel run on the
    decode sequences too gives the decode path's result."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    lengths = [20000, 4096, 513, 700, 90, 3000]
    q_lens = [1, 1, 1, 120, 90, 64]
    wl, q, qst, qs = _batch(lengths, q_lens, 8)
    out = torch.empty_like(q)
    pf = ops.PrefillAttention(wl.batch)
    pf.plan(qst)
    pf(q, qst, wl.cache, 0, wl.kv_scale, wl.block_table, wl.seq_lens, out)
    torch.cuda.synchronize()
    assert int(pf.status.item()) == 0
    _check(wl, q, qs, out, seqs=[1, 2, 3, 4, 5])
    _check(wl, q, qs, out, seqs=[0], heads=list(range(0, 64, 9)))
    # the decode sequences through the decode path (split-KV), same cache
    dec = [0, 1, 2]
    sub = Workload("custom", seed=8, lengths=[lengths[i] for i in dec], kv_dtype=0,
                   include_new_token=True)
    step = ops.DecodeStep(len(dec), 0, wl.max_blocks)
    bt = wl.block_table[dec].contiguous()
    sl = wl.seq_lens[dec].contiguous()
    qd = torch.stack([q[int(qs[b])] for b in dec])
    step.plan_step(sl)
    od_out = step.attend(qd, wl.cache, wl.kv_scale, bt, sl)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    d = (od_out.float() - torch.stack([out[int(qs[b])] for b in dec]).float()).abs()
    assert float(d.max()) <= 4e-3 and float(d.mean()) <= 2e-4


def test_prefill_output_types_and_empty_sequences():
    """FP32 output matches the oracle; FP16 output is it rounded; sequences
    without new tokens take no unit and write nothing."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    lengths = [100, 50, 600, 70]
    q_lens = [20, 0, 48, 0]
    wl, q, qst, qs = _batch(lengths, q_lens, 11)
    outs = {}
    for od_ in (ops.OUT_FP32, ops.OUT_FP16):
        pf = ops.PrefillAttention(wl.batch, out_dtype=od_)
        pf.plan(qst)
        o = torch.full((q.shape[0], 64, 128), float("nan"), device="cuda",
                       dtype=torch.float32 if od_ == ops.OUT_FP32 else torch.float16)
        outs[od_] = pf(q, qst, wl.cache, 0, wl.kv_scale, wl.block_table, wl.seq_lens, o)
        torch.cuda.synchronize()
        assert int(pf.status.item()) == 0
        assert int(pf.unit_ptr[-1].item()) == 8 * (1 + 2)   # ceil(q_len / 32) per kv head
    assert torch.equal(outs[ops.OUT_FP16], outs[ops.OUT_FP32].to(torch.float16))
    _check(wl, q, qs, outs[ops.OUT_FP32])


def test_prefill_bad_lengths_set_status_and_skip():
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    lengths = [64, 100]
    q_lens = [80, 10]                         # sequence 0 has more new tokens than tokens
    wl, q, qst, qs = _batch(lengths, q_lens, 13)
    pf = ops.PrefillAttention(wl.batch)
    pf.plan(qst)
    out = torch.zeros_like(q)
    pf(q, qst, wl.cache, 0, wl.kv_scale, wl.block_table, wl.seq_lens, out)
    torch.cuda.synchronize()
    assert int(pf.status.item()) & 4          # HPC_STATUS_BAD_SEQ_LEN
    assert not out[:80].float().abs().any()   # skipped
    _check(wl, q, qs, out, seqs=[1])


@pytest.mark.parametrize("bad_page", [2, 3])
@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_prefill_bad_block_is_reported_and_skipped(kv_dtype, staged, bad_page):
    """A block id past the cache: the status says BAD_BLOCK, the page's keys
    are left out of that sequence's attention, the other sequences are
    untouched (BF16 and E4M3 caches; E4M3 also through staged pages, where the
    real block table still marks the tile).  The bad page is page 2 or page 3
    of sequence 1, an even and an odd page of its pages 0..4."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    if staged and kv_dtype == 0:
        pytest.skip("staging applies to E4M3 caches")
    lengths = [300, 260, 100]
    q_lens = [40, 70, 100]
    wl, q, qst, qs = _batch(lengths, q_lens, 17, kv_dtype)
    wl.block_table[1, bad_page] = wl.num_blocks + 5    # keys 64 p .. 64 p + 63 of sequence 1
    pf = ops.PrefillAttention(wl.batch, staging_pages=ops.PrefillAttention.pages_for(lengths)
                              if staged else 0)
    pf.plan(qst)
    out = torch.empty_like(q)
    pf(q, qst, wl.cache, kv_dtype, wl.kv_scale, wl.block_table, wl.seq_lens, out)
    torch.cuda.synchronize()
    assert int(pf.status.item()) & 1                   # HPC_STATUS_BAD_BLOCK
    _check(wl, q, qs, out, seqs=[0, 2])
    L, n = lengths[1], q_lens[1]
    sub, row = gu.seq_view(wl.cache, wl.block_table_np[1], L, kv_dtype)
    ks, vs = [float(x) for x in wl.kv_scale.cpu().numpy()] if kv_dtype == 1 else (1.0, 1.0)
    qh = gu.bf16_host(q)[int(qs[1]):int(qs[2])]
    keep = np.r_[0:64 * bad_page, 64 * bad_page + 64:L]
    want = np.zeros((n, 64, 128))
    for h in range(8):
        K, V = od.gather_kv(sub, row, L, h, kv_dtype, ks, vs)
        for t in range(n):
            vis = keep[keep <= L - n + t]
            for j in range(8 * h, 8 * h + 8):
                want[t, j] = od.attention_head(qh[t, j], K[vis], V[vis], 1.0 / np.sqrt(128))
    tol = (gu.TOL_BF16_MAX, gu.TOL_BF16_MEAN) if kv_dtype == 0 else (gu.TOL_FP8_MAX, None)
    gu.compare(out[int(qs[1]):int(qs[2])].float().cpu().numpy().astype(np.float64), want,
               *tol, label="seq 1 without page %d" % bad_page)


def test_prefill_fp8_cache_prompts_and_chunks():
    """An E4M3 cache: whole prompts and chunks after a history (tile and block
    edges, a lane without tokens), against the oracle over the device's cache
    codes and scales; FP16 and FP32 outputs are the same values."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    lengths = [1, 16, 17, 64, 65, 130, 300, 1000, 2200]
    q_lens = [1, 16, 17, 64, 65, 130, 37, 200, 33]
    wl, q, qst, qs = _batch(lengths, q_lens, 23, kv_dtype=1)
    outs = {}
    for od_ in (ops.OUT_BF16, ops.OUT_FP32, ops.OUT_FP16):
        pf = ops.PrefillAttention(wl.batch, out_dtype=od_)
        pf.plan(qst)
        o = torch.full((q.shape[0], 64, 128), float("nan"), device="cuda",
                       dtype={ops.OUT_BF16: torch.bfloat16, ops.OUT_FP32: torch.float32,
                              ops.OUT_FP16: torch.float16}[od_])
        outs[od_] = pf(q, qst, wl.cache, 1, wl.kv_scale, wl.block_table, wl.seq_lens, o)
        torch.cuda.synchronize()
        assert int(pf.status.item()) == 0
        assert int(pf.counters.abs().sum().item()) == 0
    assert torch.equal(outs[ops.OUT_FP16], outs[ops.OUT_FP32].to(torch.float16))
    assert torch.equal(outs[ops.OUT_BF16], outs[ops.OUT_FP32].to(torch.bfloat16))
    _check(wl, q, qs, outs[ops.OUT_FP32])
    _check(wl, q, qs, outs[ops.OUT_BF16])


def test_prefill_fp8_cache_staged_pages():
    """An E4M3 cache through hpc_prefill_attn_staged: every page the batch
    reads converted once into BF16 staging, then the BF16 kernel with the K and
    V scales.  The page prefix is ceil(L / 64) per sequence; the output matches
    the oracle over the device's codes, and the direct E4M3 kernel to within
    the FP8 tolerance (P is BF16 here, F16 there); a second launch gives the
    same bits."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    lengths = [1, 16, 17, 64, 65, 130, 300, 1000, 2200]
    q_lens = [1, 16, 17, 64, 65, 130, 37, 200, 33]
    wl, q, qst, qs = _batch(lengths, q_lens, 23, kv_dtype=1)
    need = ops.PrefillAttention.pages_for(lengths)
    pf = ops.PrefillAttention(wl.batch, staging_pages=need)
    pf.plan(qst)
    out = torch.full_like(q, float("nan"))
    pf(q, qst, wl.cache, 1, wl.kv_scale, wl.block_table, wl.seq_lens, out)
    again = pf(q, qst, wl.cache, 1, wl.kv_scale, wl.block_table, wl.seq_lens, torch.empty_like(q))
    torch.cuda.synchronize()
    assert int(pf.status.item()) == 0
    assert int(pf.counters.abs().sum().item()) == 0
    pages = [(L + 63) // 64 for L in lengths]
    assert pf.page_ptr.cpu().tolist() == [0] + np.cumsum(pages).tolist()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    _check(wl, q, qs, out)
    direct = ops.PrefillAttention(wl.batch)
    direct.plan(qst)
    ref = direct(q, qst, wl.cache, 1, wl.kv_scale, wl.block_table, wl.seq_lens, torch.empty_like(q))
    torch.cuda.synchronize()
    # both are within the oracle's FP8 tolerance; between them the BF16 P
    # moves an output by at most a few BF16 ulps (1 ulp is 2^-6 at |x| in [2, 4))
    diff = (out.float() - ref.float()).abs()
    assert float(diff.max()) <= gu.TOL_FP8_MAX and float(diff.mean()) <= 5e-4, \
        (float(diff.max()), float(diff.mean()))


def test_prefill_staging_overflow_skips_the_sequences_that_do_not_fit():
    """Staging with room for the first sequences' pages only: PLAN_OVERFLOW,
    the sequences that fit are computed, the others skipped (left as they were)."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    lengths = [300, 130, 2200, 65]
    q_lens = [37, 130, 33, 65]
    wl, q, qst, qs = _batch(lengths, q_lens, 29, kv_dtype=1)
    room = ops.PrefillAttention.pages_for(lengths[:2])    # sequences 0 and 1 fit, 2 and 3 do not
    pf = ops.PrefillAttention(wl.batch, staging_pages=room)
    pf.plan(qst)
    out = torch.full_like(q, float("nan"))
    pf(q, qst, wl.cache, 1, wl.kv_scale, wl.block_table, wl.seq_lens, out)
    torch.cuda.synchronize()
    assert int(pf.status.item()) & 16                    # HPC_STATUS_PLAN_OVERFLOW
    assert int(pf.counters.abs().sum().item()) == 0
    _check(wl, q, qs, out, seqs=[0, 1])
    assert torch.isnan(out[int(qs[2]):].float()).all()
