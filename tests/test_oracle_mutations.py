"""Pin sensitivity: plant a plausible mistake in a copy of an oracle function
(on the CPU) and show that at least one pin rejects it.

A pin that passes every mutant would prove nothing; these tests keep the pins
honest.  Each mutant is a small local rewrite of the oracle function with one
defect: a wrong pairing, sign, exponent, index, scale, dropped term or
rounding rule.
"""


import numpy as np
import pytest
import torch

from oracle import decode as od
from oracle import numerics as nx
from oracle import plan as op
import oracle_pins as pins


def _rope(x, pos, theta=1e6, pair="half", expo=2.0, sign=1.0):
    x = np.asarray(x, dtype=np.float64)
    i = np.arange(64, dtype=np.float64)
    ang = float(pos) * theta ** (-expo * i / 128)
    c, s = np.cos(ang), sign * np.sin(ang)
    out = np.empty_like(x)
    if pair == "half":
        lo, hi = x[..., :64], x[..., 64:]
        out[..., :64], out[..., 64:] = lo * c - hi * s, hi * c + lo * s
    else:                                   # GPT-J interleaved pairs (2i, 2i+1)
        ev, odd = x[..., 0::2], x[..., 1::2]
        out[..., 0::2], out[..., 1::2] = ev * c - odd * s, odd * c + ev * s
    return out


@pytest.mark.parametrize("mutant", [
    lambda x, p: _rope(x, p, pair="interleaved"),
    lambda x, p: _rope(x, p, expo=1.0),          # theta^(-i/d)
    lambda x, p: _rope(x, p, sign=-1.0),         # rotation the wrong way
    lambda x, p: _rope(x, p, theta=1e4),         # wrong base
    lambda x, p: _rope(x, p + 1),                # off-by-one position
])
def test_rope_mutants_fail(mutant):
    assert np.allclose(_rope(np.eye(128)[3], 5), od.rope_neox(np.eye(128)[3], 5))
    with pytest.raises(AssertionError):
        pins.check_rope_special_angles(mutant)


@pytest.mark.parametrize("mutant", [
    lambda x, w, eps=1e-6: x / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps) * w,   # sum, not mean
    lambda x, w, eps=1e-6: x / np.sqrt(np.mean(x * x, -1, keepdims=True)) * w,        # eps dropped
    lambda x, w, eps=1e-6: x / (np.mean(np.abs(x), -1, keepdims=True) + eps) * w,     # L1 norm
    lambda x, w, eps=1e-6: x / np.sqrt(np.mean(x * x, -1, keepdims=True) + eps),      # weight dropped
])
def test_rms_norm_mutants_fail(mutant):
    with pytest.raises(AssertionError):
        pins.check_rms_norm_library(mutant, np.random.default_rng(0))


def _prologue_mutant(kind):
    """Copies of the prologue with one defect each: the norm before RoPE, the
    q and k weight vectors swapped, or the weight taken at the rotation
    partner of each element."""
    def f(q, k, v, pos, q_w, k_w):
        q_w, k_w = np.asarray(q_w, np.float64), np.asarray(k_w, np.float64)
        if kind == "norm_first":
            return (od.rope_neox(od.rms_norm(q, q_w), pos), od.rope_neox(od.rms_norm(k, k_w), pos),
                    np.asarray(v, np.float64).copy())
        if kind == "weights_swapped":
            q_w, k_w = k_w, q_w
        if kind == "partner_weight":
            q_w, k_w = np.roll(q_w, 64), np.roll(k_w, 64)
        return (od.rms_norm(od.rope_neox(q, pos), q_w), od.rms_norm(od.rope_neox(k, pos), k_w),
                np.asarray(v, np.float64).copy())
    return f


@pytest.mark.parametrize("kind", ["norm_first", "weights_swapped", "partner_weight"])
def test_prologue_mutants_fail_order_pin(kind):
    with pytest.raises(AssertionError):
        pins.check_prologue_order(_prologue_mutant(kind))


def _attn(q, K, V, scale, scale_mut=None, drop_last=False):
    if drop_last and len(K) > 1:
        K, V = K[:-1], V[:-1]
    s = (K @ q) * (scale if scale_mut is None else scale_mut)
    p = np.exp(s - s.max())
    return (p @ V) / p.sum()


@pytest.mark.parametrize("mutant", [
    lambda q, K, V, s: _attn(q, K, V, s, scale_mut=1.0 / 128),
    lambda q, K, V, s: _attn(q, K, V, s, scale_mut=1.0),
    lambda q, K, V, s: _attn(q, K, V, s, drop_last=True),
    lambda q, K, V, s: (np.exp((K @ q) * s) @ V),                        # no normalisation
])
def test_attention_mutants_fail_closed_forms(mutant):
    with pytest.raises(AssertionError):
        pins.check_attention_closed_forms(mutant, np.random.default_rng(0))


def _decode_attention_mut(q, cache, block_row, length, kv_dtype, mode):
    out = np.zeros((64, 128))
    for j in range(64):
        h = j % 8 if mode == "gqa_mod" else j // 8
        L = length - 1 if mode == "short" and length > 1 else length
        K, V = od.gather_kv(cache, block_row, L, h, kv_dtype)
        if mode == "kv_swapped":
            K, V = V, K
        out[j] = od.attention_head(q[j], K, V)
    return out


@pytest.mark.parametrize("mode", ["gqa_mod", "short", "kv_swapped"])
def test_paged_attention_mutants_fail_sdpa(mode):
    with pytest.raises(AssertionError):
        pins.check_attention_sdpa(
            lambda q, c, b, L, kv: _decode_attention_mut(q, c, b, L, kv, mode),
            np.random.default_rng(0))


@pytest.mark.parametrize("which", ["plain_mean", "no_max_weighting", "lse_without_log_l"])
def test_merge_mutants_fail(which):
    def partial(q, K, V, s):
        O, lse = od.partial_attention(q, K, V, s)
        if which == "lse_without_log_l":
            sc = (q @ K.T) * s
            lse = sc.max(1)
        return O, lse

    def merge(parts):
        if which == "plain_mean":
            return np.mean([p[0] for p in parts], axis=0)
        if which == "no_max_weighting":
            return sum(p[0] for p in parts) / len(parts)
        return od.merge_partials(parts)

    with pytest.raises(AssertionError):
        pins.check_split_merge(partial, merge, np.random.default_rng(0))


def test_e4m3_mutants_fail():
    g = pins.load_golden("e4m3_spec_values.json")

    def round_half_up(x):                       # ties away from zero
        x = np.asarray(x, float)
        a = np.minimum(np.abs(x), 448.0)
        grid = nx.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
        idx = np.searchsorted(grid, a, side="left")
        idx = np.clip(idx, 1, len(grid) - 1)
        lo, hi = grid[idx - 1], grid[idx]
        code = np.where(a - lo < hi - a, idx - 1, idx)
        return (code | (np.signbit(x).astype(int) << 7)).astype(np.uint8)

    bad = [int(round_half_up(np.array([float(c["x"])]))[0]) != int(c["code"], 16)
           for c in g["encode_rne_saturating"]]
    assert any(bad)

    def decode_bias8(codes):
        return nx.e4m3_decode(codes) / 2.0

    bad = [decode_bias8(np.array([int(c["code"], 16)], np.uint8))[0] != float(c["value"])
           for c in g["decode"] if c["value"] not in ("nan", "0")]
    assert any(bad)


def test_bf16_truncation_mutant_fails():
    vals = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    trunc = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert not np.array_equal(trunc, ref)


def test_plan_mutants_fail():
    g = pins.load_golden("plan_hand_example.json")["dynamic"]

    def plan_floor_quota(lens, C, m):          # q = floor(T / C): units overflow
        n = [op.num_tiles(L) for L in lens]
        T = 8 * sum(n)
        q = max(m, T // C)
        items, owner = [], []
        s = 0
        for b in range(len(lens)):
            for h in range(8):
                t = s
                while t < s + n[b]:
                    c = t // q
                    e = min(s + n[b], (c + 1) * q)
                    items.append((b, h, t - s, e - s))
                    t = e
                s += n[b]
        return items

    def plan_per_sequence(lens, C, m):         # one item per (seq, head): static
        return [(b, h, 0, op.num_tiles(L)) for b, L in enumerate(lens) for h in range(8)]

    for mutant in (plan_per_sequence,):
        assert [list(i) for i in mutant(g["seq_lens"], g["num_ctas"], 1)] != g["items"]
    # the floor quota happens to give q = 3 here too; it differs on 25 tiles
    lens = [65, 1, 1]   # T = 8 * 4 = 32 -> ceil(32/6) = 6, floor = 5
    a = op.plan_dynamic(lens, 6, 1)[0]
    b = plan_floor_quota(lens, 6, 1)
    assert [tuple(i) for i in a] != [tuple(i) for i in b]


def _mt_mutant(kind):
    """A copy of the multi-token attention with one plausible mistake."""
    def fn(q, cache, block_row, length, kv_dtype, k_scale=1.0, v_scale=1.0):
        q = np.asarray(q, dtype=np.float64)
        qn = q.shape[0]
        out = np.zeros((qn, od.HQ, od.D))
        for h in range(od.HKV):
            K, V = od.gather_kv(cache, block_row, length, h, kv_dtype, k_scale, v_scale)
            for t in range(qn):
                if kind == "no_mask":
                    seen = length
                elif kind == "self_hidden":
                    seen = length - qn + t
                elif kind == "from_start":              # positions counted from the sequence start
                    seen = min(t + 1, length)
                else:                                   # "reversed": new tokens in the wrong order
                    seen = length - t
                for j in range(h * 8, h * 8 + 8):
                    if seen > 0:
                        out[t, j] = od.attention_head(q[t, j], K[:seen], V[:seen])
        return out
    return fn


@pytest.mark.parametrize("kind", ["no_mask", "self_hidden", "reversed"])
def test_multi_token_mutants_fail_masked_sdpa(kind):
    with pytest.raises(AssertionError):
        pins.check_attention_mt_sdpa(_mt_mutant(kind), np.random.default_rng(3))


def test_prefill_position_mutant_fails_chunk_pin():
    """New tokens placed at positions 0 .. q_len-1 instead of L-q_len .. L-1:
    the same as the right rule for a whole prompt, wrong for a chunk after a
    history; the prefill pin (which has chunks) must catch it."""
    with pytest.raises(AssertionError):
        pins.check_attention_prefill_sdpa(_mt_mutant("from_start"), np.random.default_rng(5))
