"""Seeded random configurations of the decode attention against the float64
oracle.  Each case draws:
- the batch size and ragged lengths (zeros, tile edges, lengths below q_len);
- the cache type and the number of new tokens (q_len 1 .. 4);
- the query type (BF16, or E4M3 codes with an E4M3 cache) and the output type;
- whether the merge is fused into the attention or run as its own call.

Every output row of every sequence is compared, and the new tokens that see no
key must be exact zeros."""

import numpy as np
import pytest
import torch

from oracle import decode as od
import gpu_util as gu

pytestmark = pytest.mark.gpu

CASES = 16
EDGE_LENGTHS = [0, 1, 2, 3, 63, 64, 65, 127, 128, 129, 300, 1000, 2500]


def _config(seed):
    from paged_gqa_decode_rope_gb300 import ops
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 24))
    lengths = np.array(rng.choice(EDGE_LENGTHS, size=B)) + rng.integers(0, 3, size=B) * (rng.random(B) < 0.5)
    kv = int(rng.integers(0, 2))
    return dict(
        lengths=[int(x) for x in lengths], kv=kv, q_len=int(rng.integers(1, 5)),
        q8=bool(kv == 1 and rng.random() < 0.4),
        out_dtype=int(rng.choice([ops.OUT_BF16, ops.OUT_FP16, ops.OUT_FP32])),
        fused=bool(rng.random() < 0.6), seed=int(seed))


@pytest.mark.parametrize("seed", range(CASES))
def test_random_decode_configurations(seed):
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    cfg = _config(seed)
    qn, kv = cfg["q_len"], cfg["kv"]
    wl = Workload("custom", seed=2000 + seed, lengths=cfg["lengths"], kv_dtype=kv,
                  include_new_token=True)
    rng = np.random.default_rng(3000 + seed)
    qf = rng.standard_normal((wl.batch, qn, 64, 128))
    if cfg["q8"]:
        q_scale = float(np.abs(qf).max() / 448.0)
        codes = od.encode_kv(qf, od.KV_FP8, q_scale).astype(np.uint8)
        q = torch.as_tensor(codes, device="cuda")
        qvals = od.decode_kv(codes, od.KV_FP8, q_scale)
    else:
        q_scale = 1.0
        q = torch.as_tensor(qf, dtype=torch.float32, device="cuda").to(torch.bfloat16)
        qvals = gu.bf16_host(q)
    step = ops.DecodeStepEx(wl.batch, kv, wl.max_blocks, q_len=qn,
                            q_dtype=ops.Q_FP8 if cfg["q8"] else ops.Q_BF16, q_scale=q_scale,
                            out_dtype=cfg["out_dtype"], fused=cfg["fused"])
    step.plan_step(wl.seq_lens)
    out = step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0, cfg
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), cfg
    tol = (gu.TOL_BF16_MAX, gu.TOL_BF16_MEAN) if kv == od.KV_BF16 else (gu.TOL_FP8_MAX, None)
    sc = wl.kv_scale.cpu().numpy().astype(np.float64)
    for b in range(wl.batch):
        L = int(wl.lengths[b])
        for t in range(qn):   # tokens that see no key give exact zeros
            if L - qn + 1 + t <= 0:
                assert np.all(got[b, t] == 0.0), (cfg, b, t)
        if L == 0:
            continue
        sub, row = gu.seq_view(wl.cache, wl.block_table_np[b], L, kv)
        want = od.decode_attention_mt(qvals[b], sub, row, L, kv, sc[0], sc[1])
        gu.compare(got[b], want, *tol, label="case %d seq %d (L=%d) %s" % (seed, b, L, cfg))


PREFILL_CASES = 10


@pytest.mark.parametrize("seed", range(PREFILL_CASES))
def test_random_prefill_configurations(seed):
    """Random packed batches through the prefill call: per sequence a length
    and a number of new tokens 0 .. L (whole prompts, chunks, single decode
    tokens, sequences without new tokens), the cache type, staged pages for
    E4M3 caches or not, and the output type; every new token's row against
    the oracle over the cache as it is on the device."""
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    rng = np.random.default_rng(4000 + seed)
    B = int(rng.integers(1, 12))
    lengths = [int(x) for x in np.array(rng.choice(EDGE_LENGTHS[1:], size=B)) + rng.integers(0, 3, size=B)]
    q_lens = [int(rng.choice([0, 1, 2, 17, 32, 33, 64, L])) for L in lengths]
    q_lens = [min(n, L) for n, L in zip(q_lens, lengths)]
    kv = int(rng.integers(0, 2))
    staged = bool(kv == 1 and rng.random() < 0.5)
    out_dtype = int(rng.choice([ops.OUT_BF16, ops.OUT_FP16, ops.OUT_FP32]))
    wl = Workload("custom", seed=5000 + seed, lengths=lengths, kv_dtype=kv, include_new_token=True)
    qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(qs[-1])
    if T == 0:
        pytest.skip("no new tokens drawn")
    q = torch.as_tensor(rng.standard_normal((T, 64, 128)), dtype=torch.float32,
                        device="cuda").to(torch.bfloat16)
    qst = torch.as_tensor(qs, device="cuda")
    pf = ops.PrefillAttention(wl.batch, out_dtype=out_dtype,
                              staging_pages=ops.PrefillAttention.pages_for(lengths) if staged else 0)
    pf.plan(qst)
    dt = {ops.OUT_BF16: torch.bfloat16, ops.OUT_FP16: torch.float16, ops.OUT_FP32: torch.float32}
    out = torch.full((T, 64, 128), float("nan"), dtype=dt[out_dtype], device="cuda")
    pf(q, qst, wl.cache, kv, wl.kv_scale, wl.block_table, wl.seq_lens, out)
    torch.cuda.synchronize()
    label = "case %d: lengths %s q_lens %s kv %d staged %s out %d" % (seed, lengths, q_lens, kv, staged, out_dtype)
    assert int(pf.status.item()) == 0, label
    assert int(pf.counters.abs().sum().item()) == 0, label
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), label
    tol = (gu.TOL_BF16_MAX, gu.TOL_BF16_MEAN) if kv == od.KV_BF16 else (gu.TOL_FP8_MAX, None)
    ks, vs = [float(x) for x in wl.kv_scale.cpu().numpy()] if kv == 1 else (1.0, 1.0)
    qh = gu.bf16_host(q)
    for b in range(wl.batch):
        a, e = int(qs[b]), int(qs[b + 1])
        if e == a:
            continue
        L = lengths[b]
        sub, row = gu.seq_view(wl.cache, wl.block_table_np[b], L, kv)
        want = od.decode_attention_mt(qh[a:e], sub, row, L, kv, ks, vs)
        gu.compare(got[a:e], want, *tol, label="%s seq %d" % (label, b))
