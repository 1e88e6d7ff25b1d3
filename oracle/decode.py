"""The decode step in float64, step by step, as the pages describe it.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources (public web pages on vLLM's HPC_ATTN backend):

* [news] "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA Hopper"
  (24-ai.news, 2026-07-06).  Intro of "Two new HPC backends in the vLLM
  ecosystem": 64 query heads, 8 KV heads, head_dim 128.  "Why does dynamic
  scheduling matter for attention?": split-KV over 64-token tiles; the fused
  prologue does RoPE rotation, then QK-Norm, then the KV write, in one pass.
* [pr] "[vllm] Introducing the HPC-Ops attention backend" (analysis of vLLM PR
  #46020), "Code analysis" section 2 and "General lessons" item 1: RoPE,
  QK-Norm and the KV-cache write fused into one kernel.

Readings where the pages are silent (each is also listed in the design notes):

* RoPE is the NeoX half rotation: element i pairs with element i+64 and the
  pair turns by pos * theta^(-2i/128), theta = 1e6.
* QK-Norm is a per-head RMSNorm, eps = 1e-6, with separate q and k weight
  vectors of length 128; it runs after RoPE (the order the pages list).
  ``norm_before_rope=True`` gives the other order for comparison.
* V gets neither RoPE nor the norm.  q is not written to the cache.
* Softmax scale 1/sqrt(128); q head j reads KV head j // 8.
* The paged cache is ``[num_blocks][2 (K, V)][8 kv heads][64 tokens][128]``;
  ``slot = block * 64 + offset``.  BF16 caches store RNE-rounded values; FP8
  caches store E4M3 codes of x / scale (scale per tensor, K and V separate).
* Only length masks the keys: the decode query (q_len = 1) sees tokens
  0 .. L-1 of its sequence, the new token included.
"""

import math

import numpy as np

from . import numerics as nx

HQ = 64          # query heads
HKV = 8          # KV heads
GROUP = HQ // HKV
D = 128          # head dim
PAGE = 64        # tokens per cache block (= one KV tile)
THETA = 1.0e6
EPS = 1.0e-6

KV_BF16 = 0
KV_FP8 = 1


# ------------------------------------------------------------- prologue ---

def rope_neox(x, pos, theta=THETA):
    """Rotate x[..., 128] by position ``pos`` (NeoX half rotation).

    For i in 0..63 the pair (x[i], x[i+64]) turns by the angle
    pos * theta^(-2i/128):  x'[i] = x[i] cos - x[i+64] sin,
    x'[i+64] = x[i+64] cos + x[i] sin.  Angles are formed in float64.
    """
    x = np.asarray(x, dtype=np.float64)
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    ang = float(pos) * theta ** (-2.0 * i / D)
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rms_norm(x, w, eps=EPS):
    """Per-vector RMSNorm: x / sqrt(mean(x^2) + eps) * w over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def prologue_token(q, k, v, pos, q_w, k_w, norm_before_rope=False, theta=THETA, eps=EPS):
    """One sequence's prologue: returns (q_out, k_out, v_out) in float64.

    q [64,128], k [8,128], v [8,128].  RoPE then RMSNorm on every q and k head
    (or the reverse with ``norm_before_rope``); v passes through unchanged.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if norm_before_rope:
        qo = rope_neox(rms_norm(q, q_w, eps), pos, theta)
        ko = rope_neox(rms_norm(k, k_w, eps), pos, theta)
    else:
        qo = rms_norm(rope_neox(q, pos, theta), q_w, eps)
        ko = rms_norm(rope_neox(k, pos, theta), k_w, eps)
    return qo, ko, np.asarray(v, dtype=np.float64).copy()


def encode_kv(x, kv_dtype, scale=1.0):
    """Stored representation of cache values: BF16 bits or E4M3 codes."""
    if kv_dtype == KV_BF16:
        return nx.bf16_bits(nx.bf16_round(x))
    return nx.e4m3_encode(np.asarray(x, dtype=np.float64) / scale)


def decode_kv(raw, kv_dtype, scale=1.0):
    """float64 values of stored cache entries (dequantised for FP8)."""
    if kv_dtype == KV_BF16:
        return nx.bf16_from_bits(raw)
    return nx.e4m3_decode(raw) * scale


def write_kv(cache, slot, k_new, v_new, kv_dtype, k_scale=1.0, v_scale=1.0):
    """Write one token's K and V ([8,128] each) into ``cache`` at ``slot``.

    ``cache`` is the raw array [num_blocks, 2, 8, 64, 128] (uint16 BF16 bits or
    uint8 E4M3 codes).  A negative slot means "no write" (padding entry).
    """
    if slot < 0:
        return
    blk, off = divmod(int(slot), PAGE)
    cache[blk, 0, :, off, :] = encode_kv(k_new, kv_dtype, k_scale)
    cache[blk, 1, :, off, :] = encode_kv(v_new, kv_dtype, v_scale)


# ------------------------------------------------------------ attention ---

def gather_kv(cache, block_row, length, kv_head, kv_dtype, k_scale=1.0, v_scale=1.0):
    """De-page one sequence's K and V for one KV head: two [length, 128] arrays."""
    n_pages = -(-int(length) // PAGE)
    pages = np.asarray(block_row[:n_pages], dtype=np.int64)
    k_raw = cache[pages, 0, kv_head].reshape(n_pages * PAGE, D)[:length]
    v_raw = cache[pages, 1, kv_head].reshape(n_pages * PAGE, D)[:length]
    return decode_kv(k_raw, kv_dtype, k_scale), decode_kv(v_raw, kv_dtype, v_scale)


def attention_head(q, K, V, scale=1.0 / math.sqrt(D)):
    """Exact softmax attention of one query vector over keys K and values V.

    out = sum_t softmax_t(scale * q . K[t]) V[t]; the max is subtracted before
    exponentiating.  An empty key set gives zeros.
    """
    if K.shape[0] == 0:
        return np.zeros(V.shape[-1])
    s = (K @ np.asarray(q, dtype=np.float64)) * scale
    p = np.exp(s - np.max(s))
    return (p @ V) / np.sum(p)


def partial_attention(q_group, K, V, scale=1.0 / math.sqrt(D)):
    """Attention of several query heads over one slice of keys.

    Returns (O, lse): O [h,128] is the slice's normalised output and
    lse [h] = log(sum_t exp(scale * q . K[t])), natural log.  These are the
    split partials that a split-KV schedule produces per work item.
    """
    s = (np.asarray(q_group, dtype=np.float64) @ K.T) * scale     # [h, t]
    m = np.max(s, axis=1, keepdims=True)
    p = np.exp(s - m)
    l = np.sum(p, axis=1, keepdims=True)
    return (p @ V) / l, (m + np.log(l))[:, 0]


def merge_partials(partials):
    """Log-sum-exp merge of split partials [(O_k [h,128], lse_k [h]), ...].

    M = max_k lse_k, w_k = exp(lse_k - M), out = sum_k w_k O_k / sum_k w_k.
    """
    lse = np.stack([p[1] for p in partials])            # [k, h]
    O = np.stack([p[0] for p in partials])              # [k, h, 128]
    M = np.max(lse, axis=0)
    w = np.exp(lse - M)                                 # [k, h]
    return np.einsum("kh,khd->hd", w, O) / np.sum(w, axis=0)[:, None]


def decode_attention(q, cache, block_row, length, kv_dtype, k_scale=1.0, v_scale=1.0,
                     heads=None, scale=1.0 / math.sqrt(D)):
    """Decode attention of one sequence: q [64,128] -> out [64,128] (float64).

    q head j attends with KV head j // 8 over tokens 0..length-1 of the paged
    cache.  ``heads`` restricts the computation to a subset of q heads (other
    rows stay NaN), so that single outputs of very long sequences can be
    checked one by one.
    """
    out = np.full((HQ, D), np.nan)
    heads = range(HQ) if heads is None else heads
    by_kv = {}
    for j in heads:
        by_kv.setdefault(j // GROUP, []).append(j)
    for h, js in by_kv.items():
        if length <= 0:
            out[js] = 0.0
            continue
        K, V = gather_kv(cache, block_row, length, h, kv_dtype, k_scale, v_scale)
        for j in js:
            out[j] = attention_head(q[j], K, V, scale)
    return out


def decode_attention_mt(q, cache, block_row, length, kv_dtype, k_scale=1.0, v_scale=1.0,
                        heads=None, scale=1.0 / math.sqrt(D)):
    """Multi-token decode attention of one sequence: q [q_len,64,128] ->
    out [q_len,64,128] (float64).

    The sequence holds ``length`` tokens, the last q_len of them new in this
    step (a multi-token-prediction layer decodes its draft tokens together).
    New token t sits at position p_t = length - q_len + t and sees the keys at
    positions 0..p_t: the whole history and the new tokens up to itself.  A
    token that sees no key (length < q_len) gets zeros.  q_len = 1 is
    ``decode_attention``.
    """
    q = np.asarray(q, dtype=np.float64)
    qn = q.shape[0]
    out = np.full((qn, HQ, D), np.nan)
    heads = range(HQ) if heads is None else heads
    by_kv = {}
    for j in heads:
        by_kv.setdefault(j // GROUP, []).append(j)
    for h, js in by_kv.items():
        if length > 0:
            K, V = gather_kv(cache, block_row, length, h, kv_dtype, k_scale, v_scale)
        for t in range(qn):
            seen = int(length) - qn + 1 + t          # keys visible to new token t
            for j in js:
                out[t, j] = attention_head(q[t, j], K[:seen], V[:seen], scale) if seen > 0 else 0.0
    return out


def brute_force_attention(q, K, V, scale):
    """Pure-Python triple loop version of ``attention_head`` for tiny inputs."""
    L, d = len(K), len(q)
    s = [scale * sum(q[i] * K[t][i] for i in range(d)) for t in range(L)]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = sum(e)
    return [sum(e[t] * V[t][i] for t in range(L)) / z for i in range(d)]


# --------------------------------------------------------- end to end -----

def decode_step(q, k, v, positions, q_w, k_w, cache, block_table, seq_lens,
                slot_mapping, kv_dtype, kv_scale=(1.0, 1.0), heads=None,
                seqs=None, norm_before_rope=False):
    """The whole step for the listed sequences, in the pages' order.

    1. fused prologue per sequence: RoPE -> RMSNorm on q and k, q output stored
       as BF16, k and v written into the paged cache (modifies ``cache``);
    2. decode attention of the BF16 q over the cache (the new token included).

    Returns (q_out float64 of the stored BF16 q [B,64,128], out [B,64,128]);
    rows of sequences not in ``seqs`` (or heads not in ``heads``) are NaN.
    """
    B = len(seq_lens)
    seqs = range(B) if seqs is None else seqs
    q_out = np.full((B, HQ, D), np.nan)
    out = np.full((B, HQ, D), np.nan)
    ks, vs = float(kv_scale[0]), float(kv_scale[1])
    for b in seqs:
        qo, ko, vo = prologue_token(q[b], k[b], v[b], positions[b], q_w, k_w,
                                    norm_before_rope=norm_before_rope)
        write_kv(cache, slot_mapping[b], ko, vo, kv_dtype, ks, vs)
        q_out[b] = nx.bf16_round(qo)
    for b in seqs:
        out[b] = decode_attention(q_out[b], cache, block_table[b], int(seq_lens[b]),
                                  kv_dtype, ks, vs, heads=heads)
    return q_out, out


def decode_step_mt(q, k, v, positions, q_w, k_w, cache, block_table, seq_lens, slot_mapping,
                   kv_dtype, kv_scale=(1.0, 1.0), heads=None, seqs=None, q_scale=None):
    """The multi-token step: q [B,q_len,64,128], k and v [B,q_len,8,128],
    positions and slot_mapping [B,q_len].

    1. the prologue of every new token (RoPE at its own position, RMSNorm,
       q stored, k and v written into its cache slot), tokens in order; q is
       stored as BF16, or with ``q_scale`` as the E4M3 code of q / q_scale
       (the same encoder as the FP8 cache: RNE, saturating);
    2. ``decode_attention_mt`` of the stored q (dequantised: code * q_scale)
       over the cache.

    Returns (q_out [B,q_len,64,128], out [B,q_len,64,128]); q_out holds the
    values the attention used (BF16 values, or dequantised E4M3 codes); rows
    of sequences not in ``seqs`` are NaN.
    """
    B, qn = len(seq_lens), q.shape[1]
    seqs = range(B) if seqs is None else seqs
    q_out = np.full((B, qn, HQ, D), np.nan)
    out = np.full((B, qn, HQ, D), np.nan)
    ks, vs = float(kv_scale[0]), float(kv_scale[1])
    for b in seqs:
        for t in range(qn):
            qo, ko, vo = prologue_token(q[b, t], k[b, t], v[b, t], positions[b][t], q_w, k_w)
            write_kv(cache, slot_mapping[b][t], ko, vo, kv_dtype, ks, vs)
            if q_scale is None:
                q_out[b, t] = nx.bf16_round(qo)
            else:
                q_out[b, t] = decode_kv(encode_kv(qo, KV_FP8, q_scale), KV_FP8, q_scale)
    for b in seqs:
        out[b] = decode_attention_mt(q_out[b], cache, block_table[b], int(seq_lens[b]),
                                     kv_dtype, ks, vs, heads=heads)
    return q_out, out
