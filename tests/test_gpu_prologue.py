"""GPU fused prologue and RoPE table vs the oracle."""

import numpy as np
import pytest
import torch

from oracle import decode as od
from oracle import numerics as nx
import gpu_util as gu

pytestmark = pytest.mark.gpu


def _bf16_ulp(r):
    """BF16 spacing at |r|: the float32 spacing times 2^16."""
    return np.spacing(np.abs(r).astype(np.float32)).astype(np.float64) * 65536.0


def test_rope_table_matches_float64_angles():
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    max_pos = 262144
    t = ops.rope_cos_sin_cache(max_pos).cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(0)
    for pos in list(rng.integers(0, max_pos, 200)) + [0, 1, max_pos - 1]:
        x = np.eye(128)[:64]                       # e_i for i < 64
        y = od.rope_neox(x, int(pos))              # (cos, sin) on the diagonal pairs
        cos = y[np.arange(64), np.arange(64)]
        sin = y[np.arange(64), 64 + np.arange(64)]
        # float32 rounding of the float64 value: half an ulp of float32
        assert np.all(np.abs(t[pos, :64] - cos) <= 2.0 ** -24 + 1e-15), pos
        assert np.all(np.abs(t[pos, 64:] - sin) <= 2.0 ** -24 + 1e-15), pos


def _run_prologue(wl, cache_fill_bits):
    from paged_gqa_decode_rope_gb300 import ops
    cos_sin = ops.rope_cos_sin_cache(wl.max_pos + 1)
    if wl.kv_dtype == od.KV_BF16:
        wl.cache.view(torch.int16).fill_(cache_fill_bits)
    else:
        wl.cache.fill_(cache_fill_bits)
    q_out = torch.empty_like(wl.q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.rope_norm_kvwrite(wl.q, wl.k, wl.v, wl.positions, cos_sin, wl.q_norm_w, wl.k_norm_w,
                          wl.cache, wl.kv_dtype, wl.slot_mapping, wl.kv_scale, q_out, status)
    torch.cuda.synchronize()
    return q_out, int(status.item())


@pytest.mark.parametrize("kv", [0, 1])
@pytest.mark.parametrize("lengths", [[1, 63, 64, 300], list(range(1, 200, 7)), [131072, 5, 4096]])
def test_prologue_slots_and_values(kv, lengths):
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=3, lengths=lengths, kv_dtype=kv)
    if kv == od.KV_FP8:
        wl.kv_scale = torch.tensor([0.0123, 0.0071], dtype=torch.float32, device="cuda")
    sentinel = 0x7FC1 if kv == od.KV_BF16 else 0x7F
    q_out, st = _run_prologue(wl, sentinel)
    assert st == 0
    raw = gu.raw_cache_host(wl.cache, kv)
    B = wl.batch
    q = gu.bf16_host(wl.q); k = gu.bf16_host(wl.k); v = gu.bf16_host(wl.v)
    qw = gu.bf16_host(wl.q_norm_w); kw = gu.bf16_host(wl.k_norm_w)
    ks, vs = (wl.kv_scale.cpu().numpy().astype(np.float64) if kv == od.KV_FP8 else (1.0, 1.0))
    slots = wl.slot_mapping.cpu().numpy()
    # 1) the set of written (block, token) slots is exactly {slot_mapping[b]}
    touched = np.argwhere(raw != sentinel)
    written = set(map(tuple, touched[:, [0, 3]].tolist()))
    assert written == {(int(s) // 64, int(s) % 64) for s in slots}
    # 2) values: q_out and the K/V entries vs the oracle, within one rounding step
    qg = gu.bf16_host(q_out)
    n_tie = 0
    for b in range(B):
        qo, ko, vo = od.prologue_token(q[b], k[b], v[b], int(wl.positions[b]), qw, kw)
        rq = nx.bf16_round(qo)
        dq = np.abs(qg[b] - rq)
        ulp = _bf16_ulp(rq)
        assert np.all(dq <= ulp + 1e-30), b
        n_tie += int(np.count_nonzero(dq))
        blk, off = divmod(int(slots[b]), 64)
        got_k = od.decode_kv(raw[blk, 0, :, off], kv, ks)
        got_v = od.decode_kv(raw[blk, 1, :, off], kv, vs)
        if kv == od.KV_BF16:
            for got, want in ((got_k, ko), (got_v, vo)):
                r = nx.bf16_round(want)
                assert np.all(np.abs(got - r) <= _bf16_ulp(r)), b
        else:
            for got, want, s in ((got_k, ko, ks), (got_v, vo, vs)):
                r = nx.e4m3_decode(nx.e4m3_encode(want / s)) * s
                step = nx.e4m3_step(np.minimum(np.abs(want / s), 448.0)) * s
                assert np.all(np.abs(got - r) <= step + 1e-30), b
    # rounding differences from float32 vs float64 arithmetic must be rare
    assert n_tie <= max(4, qg.size // 200), n_tie


def test_prologue_aliasing_padding_and_bad_inputs():
    gu.require_gpu()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    wl = Workload("custom", seed=4, lengths=[10, 70, 130], kv_dtype=0)
    cos_sin = ops.rope_cos_sin_cache(256)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_ref = torch.empty_like(wl.q)
    ops.rope_norm_kvwrite(wl.q, wl.k, wl.v, wl.positions, cos_sin, wl.q_norm_w, wl.k_norm_w,
                          wl.cache, 0, wl.slot_mapping, wl.kv_scale, q_ref, status)
    q_alias = wl.q.clone()
    ops.rope_norm_kvwrite(q_alias, wl.k, wl.v, wl.positions, cos_sin, wl.q_norm_w, wl.k_norm_w,
                          wl.cache, 0, wl.slot_mapping, wl.kv_scale, q_alias, status)
    torch.cuda.synchronize()
    assert torch.equal(q_alias.view(torch.int16), q_ref.view(torch.int16)), "q_out may alias q"
    # slot -1: no cache write; slot past the cache: BAD_SLOT; position past the table: BAD_POSITION
    before = wl.cache.clone()
    slots = torch.tensor([-1, wl.num_blocks * 64 + 3, int(wl.slot_mapping[2])], dtype=torch.int64, device="cuda")
    pos = wl.positions.clone()
    pos[2] = 256
    status.zero_()
    ops.rope_norm_kvwrite(wl.q, wl.k, wl.v, pos, cos_sin, wl.q_norm_w, wl.k_norm_w,
                          wl.cache, 0, slots, wl.kv_scale, q_ref, status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & 2 and st & 8
    assert torch.equal(before.view(torch.int16), wl.cache.view(torch.int16)), "nothing written"
