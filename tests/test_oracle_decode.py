"""Oracle pins: RoPE, RMSNorm, cache write, attention, split/merge (CPU only)."""

import math

import numpy as np
import pytest

from oracle import decode as od
from oracle import numerics as nx
import oracle_pins as pins


@pytest.fixture
def rng():
    return np.random.default_rng(1234)


def test_rope_special_angles():
    pins.check_rope_special_angles(od.rope_neox)


def test_rope_norm_and_identity(rng):
    pins.check_rope_norm_and_identity(od.rope_neox, rng)


def test_rope_group_properties(rng):
    pins.check_rope_group(od.rope_neox, rng)


def test_rms_norm_against_library(rng):
    pins.check_rms_norm_library(od.rms_norm, rng)


def test_prologue_order_hand_derived():
    """RoPE first, then the weighted RMSNorm: hand-derived values at an angle
    of exactly 1 rad for a q head and a k head."""
    pins.check_prologue_order(od.prologue_token)


def test_prologue_order_only_matters_through_the_weight(rng):
    """The mean square is rotation invariant: with unit weights RoPE and the
    norm commute; with non-unit weights they do not."""
    q, k, v = rng.standard_normal((64, 128)), rng.standard_normal((8, 128)), rng.standard_normal((8, 128))
    one = np.ones(128)
    a = od.prologue_token(q, k, v, 777, one, one)
    b = od.prologue_token(q, k, v, 777, one, one, norm_before_rope=True)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=0, atol=1e-12)
    w = 1.0 + 0.1 * rng.standard_normal(128)
    a = od.prologue_token(q, k, v, 777, w, w)
    b = od.prologue_token(q, k, v, 777, w, w, norm_before_rope=True)
    assert np.max(np.abs(a[0] - b[0])) > 1e-3
    assert np.array_equal(a[2], v) and np.array_equal(b[2], v), "v passes through"


def test_attention_closed_forms(rng):
    pins.check_attention_closed_forms(od.attention_head, rng)


def test_attention_brute_force(rng):
    for L in (1, 2, 5, 13):
        q = rng.standard_normal(6)
        K = rng.standard_normal((L, 6))
        V = rng.standard_normal((L, 6))
        got = od.attention_head(q, K, V, 0.37)
        want = od.brute_force_attention(q.tolist(), K.tolist(), V.tolist(), 0.37)
        assert np.allclose(got, want, rtol=0, atol=1e-13)


def test_attention_matches_sdpa_gqa(rng):
    pins.check_attention_sdpa(od.decode_attention, rng)


def test_multi_token_attention_matches_masked_sdpa(rng):
    pins.check_attention_mt_sdpa(od.decode_attention_mt, rng)


def test_prefill_blocks_match_causal_sdpa(rng):
    pins.check_attention_prefill_sdpa(od.decode_attention_mt, rng)


def test_multi_token_attention_is_causal(rng):
    pins.check_attention_mt_causal(od.decode_attention_mt, od.decode_attention, rng)


def test_split_merge_equals_unsplit(rng):
    pins.check_split_merge(od.partial_attention, od.merge_partials, rng)


def test_block_table_permutation_invariance(rng):
    """Moving pages around, with the block table updated to match, leaves the
    output unchanged."""
    nb, L = 9, 300
    cache = od.encode_kv(rng.standard_normal((nb, 2, 8, 64, 128)), od.KV_BF16)
    bt = rng.permutation(nb)[:5]
    q = rng.standard_normal((64, 128))
    out1 = od.decode_attention(q, cache, bt, L, od.KV_BF16)
    perm = rng.permutation(nb)                   # page p moves to perm[p]
    cache2 = np.empty_like(cache)
    cache2[perm] = cache
    out2 = od.decode_attention(q, cache2, perm[bt], L, od.KV_BF16)
    assert np.array_equal(out1, out2)


def test_gqa_head_mapping(rng):
    """q head j reads KV head j // 8: putting distinct constant values in each
    KV head's V makes every output row equal to its group's constant."""
    nb, L = 2, 70
    V = np.zeros((nb, 8, 64, 128))
    for h in range(8):
        V[:, h] = h + 1.0
    K = rng.standard_normal((nb, 8, 64, 128))
    cache = np.stack([od.encode_kv(K, 0), od.encode_kv(V, 0)], axis=1)
    out = od.decode_attention(rng.standard_normal((64, 128)), cache, [1, 0], L, 0)
    for j in range(64):
        assert np.allclose(out[j], j // 8 + 1.0, rtol=0, atol=1e-12)


def test_write_kv_touches_only_its_slot(rng):
    for kv in (od.KV_BF16, od.KV_FP8):
        dt = np.uint16 if kv == od.KV_BF16 else np.uint8
        sentinel = 0x7FC1 if kv == od.KV_BF16 else 0x7F
        cache = np.full((4, 2, 8, 64, 128), sentinel, dt)
        k, v = rng.standard_normal((8, 128)), rng.standard_normal((8, 128))
        od.write_kv(cache, 2 * 64 + 37, k, v, kv, 0.01, 0.02)
        touched = np.argwhere(cache != sentinel)
        assert set(map(tuple, touched[:, [0, 3]])) == {(2, 37)}
        got_k = od.decode_kv(cache[2, 0, :, 37], kv, 0.01)
        if kv == od.KV_BF16:
            assert np.array_equal(got_k, nx.bf16_round(k))
        else:
            assert np.all(np.abs(got_k - np.clip(k, -4.48, 4.48)) <= nx.e4m3_step(k / 0.01) * 0.01 / 2 + 1e-15)
        od.write_kv(cache, -1, k, v, kv)          # padding slot: no write
        assert set(map(tuple, np.argwhere(cache != sentinel)[:, [0, 3]])) == {(2, 37)}


def test_fp8_single_key_returns_dequantised_value(rng):
    cache = np.full((1, 2, 8, 64, 128), 0x7F, np.uint8)        # NaN everywhere
    k, v = rng.standard_normal((8, 128)), rng.standard_normal((8, 128))
    od.write_kv(cache, 0, k, v, od.KV_FP8, 0.02, 0.03)
    out = od.decode_attention(rng.standard_normal((64, 128)), cache, [0], 1, od.KV_FP8, 0.02, 0.03)
    want = nx.e4m3_decode(nx.e4m3_encode(v / 0.03)) * 0.03
    for j in range(64):
        assert np.array_equal(out[j], want[j // 8])


def test_decode_step_tiny_matches_composition(rng):
    """End to end on the tiny shape: the new token lands in its slot and the
    output equals attention over the history plus that token."""
    lengths = [1, 63, 64, 300]
    n = [-(-L // 64) for L in lengths]
    nb = sum(n) + 2
    perm = rng.permutation(nb)
    bt = np.zeros((4, max(n)), np.int64)
    o = 0
    for b in range(4):
        bt[b, :n[b]] = perm[o:o + n[b]]
        o += n[b]
    cache = od.encode_kv(rng.standard_normal((nb, 2, 8, 64, 128)), 0)
    q = rng.standard_normal((4, 64, 128))
    k = rng.standard_normal((4, 8, 128))
    v = rng.standard_normal((4, 8, 128))
    qw = nx.bf16_round(1 + 0.1 * rng.standard_normal(128))
    kw = nx.bf16_round(1 + 0.1 * rng.standard_normal(128))
    pos = [L - 1 for L in lengths]
    slots = [bt[b, (L - 1) // 64] * 64 + (L - 1) % 64 for b, L in enumerate(lengths)]
    c0 = cache.copy()
    q_out, out = od.decode_step(q, k, v, pos, qw, kw, cache, bt, lengths, slots, 0)
    for b, L in enumerate(lengths):
        qo, ko, vo = od.prologue_token(q[b], k[b], v[b], pos[b], qw, kw)
        assert np.array_equal(q_out[b], nx.bf16_round(qo))
        blk, off = divmod(slots[b], 64)
        assert np.array_equal(cache[blk, 0, :, off], od.encode_kv(ko, 0))
        assert np.array_equal(cache[blk, 1, :, off], od.encode_kv(vo, 0))
        for h in (0, 5):
            K, V = od.gather_kv(cache, bt[b], L, h, 0)
            j = 8 * h + 3
            assert np.allclose(out[b, j], od.attention_head(q_out[b, j], K, V, 1 / math.sqrt(128)))
    mask = np.ones(cache.shape[:1] + cache.shape[3:4], bool)
    for s in slots:
        mask[s // 64, s % 64] = False
    assert np.array_equal(cache.transpose(0, 3, 1, 2, 4)[mask], c0.transpose(0, 3, 1, 2, 4)[mask])


def test_multi_token_step_writes_every_new_token_and_is_the_single_step_at_one(rng):
    """The multi-token step writes each new token into its own slot at its own
    position, and with q_len = 1 it is the single-token step."""
    lengths = [3, 66, 130]
    qn = 3
    n = [-(-L // 64) for L in lengths]
    nb = sum(n) + 1
    bt = np.zeros((3, max(n)), np.int64)
    perm = rng.permutation(nb)
    o = 0
    for b in range(3):
        bt[b, :n[b]] = perm[o:o + n[b]]
        o += n[b]
    cache = od.encode_kv(rng.standard_normal((nb, 2, 8, 64, 128)), 0)
    q = rng.standard_normal((3, qn, 64, 128))
    k = rng.standard_normal((3, qn, 8, 128))
    v = rng.standard_normal((3, qn, 8, 128))
    qw = nx.bf16_round(1 + 0.1 * rng.standard_normal(128))
    kw = nx.bf16_round(1 + 0.1 * rng.standard_normal(128))
    pos = [[L - qn + t for t in range(qn)] for L in lengths]
    slots = [[bt[b, p // 64] * 64 + p % 64 for p in pos[b]] for b in range(3)]
    c1 = cache.copy()
    q_out, out = od.decode_step_mt(q, k, v, pos, qw, kw, c1, bt, lengths, slots, 0)
    for b in range(3):
        for t in range(qn):
            qo, ko, vo = od.prologue_token(q[b, t], k[b, t], v[b, t], pos[b][t], qw, kw)
            assert np.array_equal(q_out[b, t], nx.bf16_round(qo))
            blk, off = divmod(slots[b][t], 64)
            assert np.array_equal(c1[blk, 0, :, off], od.encode_kv(ko, 0))
            assert np.array_equal(c1[blk, 1, :, off], od.encode_kv(vo, 0))
    # q_len = 1: the last new token alone, after the others were written
    c2 = c1.copy()
    last = [[p[-1]] for p in pos]
    lslots = [[s[-1]] for s in slots]
    q1, o1 = od.decode_step_mt(q[:, -1:], k[:, -1:], v[:, -1:], last, qw, kw, c2, bt, lengths, lslots, 0)
    c3 = c1.copy()
    q2, o2 = od.decode_step(q[:, -1], k[:, -1], v[:, -1], [p[0] for p in last], qw, kw, c3, bt,
                            lengths, [s[0] for s in lslots], 0)
    assert np.array_equal(o1[:, 0], o2) and np.array_equal(q1[:, 0], q2)
    assert np.allclose(out[:, -1], o2, rtol=0, atol=1e-12)



def test_fp8_query_step_quantises_q_with_the_cache_encoder(rng):
    """With an E4M3 q the step stores code(q / q_scale) and attends with
    code * q_scale; a q_scale that makes q exact on the E4M3 grid gives the
    BF16-q result of the same values."""
    lengths = [70, 5]
    qn = 2
    bt = np.array([[0, 1], [2, 0]])
    cache = od.encode_kv(rng.standard_normal((3, 2, 8, 64, 128)) * 0.5, od.KV_FP8, 0.01)
    q = rng.standard_normal((2, qn, 64, 128))
    k = rng.standard_normal((2, qn, 8, 128))
    v = rng.standard_normal((2, qn, 8, 128))
    w = np.ones(128)
    pos = [[L - qn + t for t in range(qn)] for L in lengths]
    slots = [[bt[b, p // 64] * 64 + p % 64 for p in pos[b]] for b in range(2)]
    c1 = cache.copy()
    qs = 0.004
    q_used, out = od.decode_step_mt(q, k, v, pos, w, w, c1, bt, lengths, slots, od.KV_FP8,
                                    (0.01, 0.01), q_scale=qs)
    for b in range(2):
        for t in range(qn):
            qo, _, _ = od.prologue_token(q[b, t], k[b, t], v[b, t], pos[b][t], w, w)
            codes = od.encode_kv(qo, od.KV_FP8, qs)
            assert np.array_equal(q_used[b, t], od.decode_kv(codes, od.KV_FP8, qs))
    # attention is decode_attention_mt of those values
    for b in range(2):
        want = od.decode_attention_mt(q_used[b], c1, bt[b], lengths[b], od.KV_FP8, 0.01, 0.01)
        assert np.array_equal(out[b], want)
    # a q already on the E4M3 grid (scaled by a power of two) is stored exactly
    grid = od.decode_kv(od.encode_kv(rng.standard_normal((64, 128)), od.KV_FP8, 1.0), od.KV_FP8, 1.0)
    back = od.decode_kv(od.encode_kv(grid * 0.25, od.KV_FP8, 0.25), od.KV_FP8, 0.25)
    assert np.array_equal(back, grid * 0.25)
