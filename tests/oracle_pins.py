"""Pins that tie the oracle to facts outside itself.

Each ``check_*`` takes the function under test as an argument, so that
``test_oracle_mutations.py`` can hand it a copy of the oracle with a planted
mistake and show that at least one pin fails.  Sources of truth used here:
hand-derived fixtures (tests/golden/), closed forms, group/invariance
properties of the mathematics, library routines (torch SDPA, torch rms_norm,
scipy logsumexp, torch float casts) and brute force on tiny inputs.
"""

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
D = 128
HALF = 64


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ RoPE --

def check_rope_special_angles(rope):
    """e_i rotated at position pos lands on (cos a, sin a) in the (i, i+64)
    plane with the hand-derived angle a (fixture), and nowhere else."""
    g = load_golden("rope_special_angles.json")
    for c in g["cases"]:
        i, pos, a = c["i"], c["pos"], float(c["angle"])
        x = np.zeros(D)
        x[i] = 1.0
        y = rope(x, pos)
        want = np.zeros(D)
        want[i], want[i + HALF] = math.cos(a), math.sin(a)
        # the angle is pos * inv_freq; float64 rounding of the product grows
        # with pos, so allow a few ulp of the angle itself
        tol = 1e-14 + 4 * np.spacing(max(a, 1.0))
        assert np.max(np.abs(y - want)) <= tol, (c, y[i], y[i + HALF])
        # the partner e_{i+64} turns to (-sin a, cos a)
        x = np.zeros(D)
        x[i + HALF] = 1.0
        y = rope(x, pos)
        want = np.zeros(D)
        want[i], want[i + HALF] = -math.sin(a), math.cos(a)
        assert np.max(np.abs(y - want)) <= tol, c


def check_rope_norm_and_identity(rope, rng):
    x = rng.standard_normal((5, D))
    assert np.allclose(rope(x, 0), x, rtol=0, atol=0), "pos 0 must be the identity"
    for pos in (1, 17, 4095, 262143):
        y = rope(x, pos)
        n_in = x[:, :HALF] ** 2 + x[:, HALF:] ** 2
        n_out = y[:, :HALF] ** 2 + y[:, HALF:] ** 2
        assert np.allclose(n_in, n_out, rtol=1e-12, atol=1e-12), "pair norms change"


def check_rope_group(rope, rng):
    """R(a) R(b) = R(a+b), and <R(m) q, R(n) k> depends only on m - n."""
    x = rng.standard_normal(D)
    for a, b in ((3, 5), (1000, 24), (70000, 123)):
        assert np.allclose(rope(rope(x, a), b), rope(x, a + b), rtol=0, atol=1e-9)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for m, n, s in ((10, 3, 100), (4096, 17, 5000)):
        d1 = rope(q, m) @ rope(k, n)
        d2 = rope(q, m + s) @ rope(k, n + s)
        assert abs(d1 - d2) < 1e-9 * (1 + abs(d1)), (m, n, s)


# --------------------------------------------------------------- RMSNorm --

def check_rms_norm_library(rms, rng):
    x = rng.standard_normal((7, D)) * 3.0
    w = 1.0 + 0.1 * rng.standard_normal(D)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (D,), torch.from_numpy(w), eps=1e-6)
    assert np.allclose(rms(x, w), ref.numpy(), rtol=1e-13, atol=1e-13)
    # with unit weights and eps -> 0 the output has RMS exactly 1 and keeps
    # the input's direction
    y = rms(x, np.ones(D), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)
    cos = np.sum(x * y, -1) / np.linalg.norm(x, axis=-1) / np.linalg.norm(y, axis=-1)
    assert np.allclose(cos, 1.0, rtol=1e-13)


# -------------------------------------------------------------- prologue --

def check_prologue_order(prologue):
    """prologue(q [64,128], k [8,128], v [8,128], pos, q_w, k_w) -> (q', k', v').

    Hand-derived fixture (tests/golden/prologue_order.json): a unit vector
    rotated by RoPE and then normalised with a weight that differs between
    the two elements of its rotation pair.  Rotating first puts w[i] on the
    cosine part and w[i+64] on the sine part; normalising first would put
    one weight on both.  The q and k weight vectors differ at the checked
    elements, so using one for the other also fails."""
    g = load_golden("prologue_order.json")
    for which in ("q", "k"):
        q = np.zeros((64, D))
        k = np.zeros((8, D))
        v = np.arange(8 * D, dtype=np.float64).reshape(8, D) / 100.0
        q_w, k_w = np.ones(D), np.ones(D)
        for i, w in g["q_weight"].items():
            q_w[int(i)] = float(w)
        for i, w in g["k_weight"].items():
            k_w[int(i)] = float(w)
        head = g[which + "_head"]
        x = q if which == "q" else k
        x[head, g[which + "_in_index"]] = 1.0
        qo, ko, vo = prologue(q, k, v, g[which + "_pos"], q_w, k_w)
        got = qo if which == "q" else ko
        other = ko if which == "q" else qo
        want = np.zeros_like(got)
        for i, val in g[which + "_expected"].items():
            want[head, int(i)] = float(val)
        # the angle is exactly 1 rad; float64 sin/cos and the norm's sqrt
        # leave a few ulp of the ~30-sized results
        assert np.max(np.abs(got - want)) <= 1e-13, (which, got[head][got[head] != 0])
        assert not np.any(other), "a zero head stays zero"
        assert np.array_equal(vo, v), "v passes through"


# ------------------------------------------------------------- attention --

def check_attention_closed_forms(attn, rng):
    """attn(q, K, V, scale) -> out for one query vector."""
    s = 1.0 / math.sqrt(D)
    V = rng.standard_normal((1, D))
    K = rng.standard_normal((1, D))
    q = rng.standard_normal(D)
    assert np.allclose(attn(q, K, V, s), V[0], rtol=0, atol=1e-14), "single key must return v"
    K = np.repeat(rng.standard_normal((1, D)), 9, axis=0)
    V = rng.standard_normal((9, D))
    assert np.allclose(attn(q, K, V, s), V.mean(0), rtol=0, atol=1e-13), "identical keys -> mean V"
    # two keys whose scores differ by ln 3: weights 3/4 and 1/4
    q = np.zeros(D)
    q[0] = math.sqrt(D)
    K = np.zeros((2, D))
    K[0, 0] = math.log(3.0)
    V = rng.standard_normal((2, D))
    assert np.allclose(attn(q, K, V, s), 0.75 * V[0] + 0.25 * V[1], rtol=0, atol=1e-13)


def check_attention_sdpa(decode_attention_fn, rng, kv_dtype=0):
    """GQA decode over a paged cache equals torch SDPA (float64, enable_gqa)
    on the de-paged contiguous K/V."""
    from oracle import decode as od
    lengths = [1, 63, 64, 130]
    n_pages = [-(-L // 64) for L in lengths]
    nb = sum(n_pages) + 3
    perm = rng.permutation(nb)
    bt = np.full((len(lengths), max(n_pages)), -1, np.int64)
    o = 0
    for b, n in enumerate(n_pages):
        bt[b, :n] = perm[o:o + n]
        o += n
    Kc = rng.standard_normal((nb, 8, 64, D))
    Vc = rng.standard_normal((nb, 8, 64, D))
    cache = np.stack([od.encode_kv(Kc, 0), od.encode_kv(Vc, 0)], axis=1)   # bf16 bits
    for b, L in enumerate(lengths):
        q = rng.standard_normal((64, D))
        out = decode_attention_fn(q, cache, bt[b], L, 0)
        K = np.concatenate([od.decode_kv(cache[p, 0], 0) for p in bt[b, :n_pages[b]]], axis=1)[:, :L]
        V = np.concatenate([od.decode_kv(cache[p, 1], 0) for p in bt[b, :n_pages[b]]], axis=1)[:, :L]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, :, None, :], torch.from_numpy(K)[None],
            torch.from_numpy(V)[None], enable_gqa=True)[0, :, 0, :].numpy()
        assert np.allclose(out, ref, rtol=1e-11, atol=1e-12), (b, np.max(np.abs(out - ref)))


def check_attention_mt_sdpa(mt_fn, rng):
    """Multi-token decode over a paged cache equals torch SDPA (float64,
    enable_gqa) with an explicit boolean mask: query t of q_len, at position
    L - q_len + t, may attend to key s iff s <= L - q_len + t.  A query that
    sees no key (L < q_len) must give zeros."""
    from oracle import decode as od
    cases = [(2, 2), (2, 65), (3, 64), (3, 130), (4, 4), (4, 129), (2, 1), (4, 2)]
    n_pages = [-(-L // 64) for _, L in cases]
    nb = sum(n_pages) + 2
    perm = rng.permutation(nb)
    Kc = rng.standard_normal((nb, 8, 64, D))
    Vc = rng.standard_normal((nb, 8, 64, D))
    cache = np.stack([od.encode_kv(Kc, 0), od.encode_kv(Vc, 0)], axis=1)
    o = 0
    for (qn, L), n in zip(cases, n_pages):
        bt = perm[o:o + n]
        o += n
        q = rng.standard_normal((qn, 64, D))
        out = mt_fn(q, cache, bt, L, 0)
        K = np.concatenate([od.decode_kv(cache[pg, 0], 0) for pg in bt], axis=1)[:, :L]
        V = np.concatenate([od.decode_kv(cache[pg, 1], 0) for pg in bt], axis=1)[:, :L]
        mask = np.arange(L)[None, :] <= (L - qn + np.arange(qn))[:, None]      # [q_len, L]
        for t in range(qn):
            if not mask[t].any():
                assert np.all(out[t] == 0.0), (qn, L, t)
                continue
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[t])[None, :, None, :], torch.from_numpy(K)[None],
                torch.from_numpy(V)[None], attn_mask=torch.from_numpy(mask[t:t + 1]),
                enable_gqa=True)[0, :, 0, :].numpy()
            assert np.allclose(out[t], ref, rtol=1e-11, atol=1e-12), (qn, L, t)


def check_attention_prefill_sdpa(mt_fn, rng):
    """Prompt-sized blocks of new tokens (a whole prompt, L = q_len, and a
    chunk after a history) equal torch SDPA with the causal mask of their
    positions; for a whole prompt that is SDPA's own is_causal."""
    from oracle import decode as od
    for qn, L in ((70, 70), (45, 200)):
        n_pages = -(-L // 64)
        Kc = rng.standard_normal((n_pages + 1, 8, 64, D))
        Vc = rng.standard_normal((n_pages + 1, 8, 64, D))
        cache = np.stack([od.encode_kv(Kc, 0), od.encode_kv(Vc, 0)], axis=1)
        bt = rng.permutation(n_pages + 1)[:n_pages]
        q = rng.standard_normal((qn, 64, D)) * 0.5
        out = mt_fn(q, cache, bt, L, 0)
        K = np.concatenate([od.decode_kv(cache[pg, 0], 0) for pg in bt], axis=1)[:, :L]
        V = np.concatenate([od.decode_kv(cache[pg, 1], 0) for pg in bt], axis=1)[:, :L]
        qt = torch.from_numpy(q.transpose(1, 0, 2))[None]            # [1, 64, q_len, 128]
        if qn == L:
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, torch.from_numpy(K)[None], torch.from_numpy(V)[None], is_causal=True,
                enable_gqa=True)
        else:
            mask = np.arange(L)[None, :] <= (L - qn + np.arange(qn))[:, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, torch.from_numpy(K)[None], torch.from_numpy(V)[None],
                attn_mask=torch.from_numpy(mask), enable_gqa=True)
        ref = ref[0].numpy().transpose(1, 0, 2)                        # [q_len, 64, 128]
        assert np.allclose(out, ref, rtol=1e-11, atol=1e-12), (qn, L)


def check_attention_mt_causal(mt_fn, single_fn, rng):
    """Changing the value of the last new token changes only the last query's
    output; with q_len = 1 the multi-token form is the single-token one."""
    from oracle import decode as od
    L, qn = 200, 3
    Kc = rng.standard_normal((4, 8, 64, D))
    Vc = rng.standard_normal((4, 8, 64, D))
    cache = np.stack([od.encode_kv(Kc, 0), od.encode_kv(Vc, 0)], axis=1)
    bt = np.array([2, 0, 3, 1])
    q = rng.standard_normal((qn, 64, D))
    a = mt_fn(q, cache, bt, L, 0)
    c2 = cache.copy()
    last = L - 1
    c2[bt[last // 64], 1, :, last % 64] = od.encode_kv(rng.standard_normal((8, D)) * 5, 0)
    b = mt_fn(q, c2, bt, L, 0)
    assert np.array_equal(a[:qn - 1], b[:qn - 1])
    assert np.abs(a[qn - 1] - b[qn - 1]).max() > 1e-3
    one = mt_fn(q[:1], cache, bt, L, 0)[0]
    assert np.array_equal(one, single_fn(q[0], cache, bt, L, 0))


def check_split_merge(partial_fn, merge_fn, rng):
    """Splitting the keys at arbitrary cut points and merging the partials
    equals the unsplit result; lse equals scipy's logsumexp."""
    from scipy.special import logsumexp
    s = 1.0 / math.sqrt(D)
    L = 700
    q = rng.standard_normal((8, D)) * 2.0
    K = rng.standard_normal((L, D))
    V = rng.standard_normal((L, D))
    O_all, lse_all = partial_fn(q, K, V, s)
    ref_lse = logsumexp((q @ K.T) * s, axis=1)
    assert np.allclose(lse_all, ref_lse, rtol=0, atol=1e-12)
    for trial in range(6):
        cuts = sorted(set(rng.integers(1, L, size=trial + 1).tolist()))
        bounds = [0] + cuts + [L]
        parts = [partial_fn(q, K[a:b], V[a:b], s) for a, b in zip(bounds, bounds[1:])]
        assert np.allclose(merge_fn(parts), O_all, rtol=0, atol=1e-12), cuts
