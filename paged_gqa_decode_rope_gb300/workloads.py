"""Seeded synthetic inputs of the decode step, shared by the tests, the
benchmark and the smoke run.

This module holds none of the method's arithmetic.  It makes lengths, page
permutations, slot indices, N(0,1) values, the NaN fill of unused cache
entries, and the per-tensor FP8 scales of the synthetic history.  Every
consumer (CUDA path or CPU oracle) then reads the same tensors.

Workloads (64 query heads, 8 KV heads, head_dim 128, 64-token pages):

    tiny        4 sequences of {1, 63, 64, 300} tokens, BF16 KV
    uniform     32 x 4096 tokens, BF16 KV
    mixed       1 x 131072 + 31 x 4096 tokens, BF16 KV
    mixed_fp8   the same mix, FP8 E4M3 KV
    heavy_tail  64 lengths floor(exp(U(ln 128, ln 262144))) from
                numpy default_rng(seed), FP8 E4M3 KV

Recipe: new-token q, k, v ~ N(0,1) rounded to BF16; q/k norm weights
1 + 0.1 N(0,1) rounded to BF16; positions = length - 1; the block table is a
seeded random permutation of a pool of sum(ceil(L/64)) pages plus 5% spares;
history K/V ~ N(0,1) (BF16, or E4M3 codes of x / scale with
scale = max|x| / 448 over that tensor's history, made with torch's float8
cast); every cache entry that holds no history (spare pages, slots at or past
the history length) is NaN.
"""

import numpy as np
import torch

KV_BF16 = 0
KV_FP8 = 1
HQ, HKV, D, PAGE = 64, 8, 128, 64
BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F

WORKLOADS = {
    "tiny": ("fixed", [1, 63, 64, 300], KV_BF16),
    "uniform": ("fixed", [4096] * 32, KV_BF16),
    "mixed": ("fixed", [131072] + [4096] * 31, KV_BF16),
    "mixed_fp8": ("fixed", [131072] + [4096] * 31, KV_FP8),
    "heavy_tail": ("loguniform", (64, 128, 262144), KV_FP8),
}


def seq_lengths(name, seed=0):
    kind, arg, _ = WORKLOADS[name]
    if kind == "fixed":
        return np.asarray(arg, dtype=np.int32)
    n, lo, hi = arg
    rng = np.random.default_rng(seed)
    return np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi), n))).astype(np.int32)


def kv_dtype_of(name):
    return WORKLOADS[name][2]


def pages_of(length):
    return -(-int(length) // PAGE) if length > 0 else 0


def block_table_for(lengths, seed=0, spare_frac=0.05):
    """Seeded random page assignment: (block_table int32 [B, max_blocks], num_blocks).

    Entries past a sequence's last page are -1 (never read)."""
    n = [pages_of(L) for L in lengths]
    total = sum(n)
    num_blocks = total + int(np.ceil(spare_frac * total)) + 1
    perm = np.random.default_rng(seed + 7919).permutation(num_blocks).astype(np.int32)
    max_blocks = max(1, max(n) if n else 1)
    bt = np.full((len(lengths), max_blocks), -1, dtype=np.int32)
    o = 0
    for b, nb in enumerate(n):
        bt[b, :nb] = perm[o:o + nb]
        o += nb
    return bt, num_blocks


def slot_mapping_for(lengths, block_table):
    """Cache slot of each sequence's newest token (position length-1); -1 if empty."""
    out = np.full(len(lengths), -1, dtype=np.int64)
    for b, L in enumerate(lengths):
        if L > 0:
            out[b] = int(block_table[b, (L - 1) // PAGE]) * PAGE + (L - 1) % PAGE
    return out


def new_token(batch, seed=0, device="cuda"):
    """(q [B,64,128], k [B,8,128], v [B,8,128], q_norm_w [128], k_norm_w [128]), BF16."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn((batch, HQ, D), generator=g).to(torch.bfloat16)
    k = torch.randn((batch, HKV, D), generator=g).to(torch.bfloat16)
    v = torch.randn((batch, HKV, D), generator=g).to(torch.bfloat16)
    qw = (1.0 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    kw = (1.0 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    return tuple(t.to(device) for t in (q, k, v, qw, kw))


def _history_values(b, length, which, seed, device):
    """N(0,1) history of sequence b, whole pages: float32 [pages*64, 8, 128].
    Rows at or past ``length`` are NaN.  Regenerated identically on demand."""
    g = torch.Generator(device=device).manual_seed(seed * 1000003 + 2 * b + which)
    n = pages_of(length) if length > 0 else 0
    x = torch.randn((n * PAGE, HKV, D), generator=g, device=device, dtype=torch.float32)
    x = x.to(torch.bfloat16).to(torch.float32)
    x[length:] = float("nan")
    return x


def history_values(b, length, which, seed=0, device="cuda"):
    """Public accessor of the unquantised history (which: 0 = K, 1 = V)."""
    return _history_values(b, length, which, seed, device)


def make_cache(lengths, block_table, num_blocks, kv_dtype, seed=0, device="cuda",
               include_new_token=False):
    """Paged cache [num_blocks, 2, 8, 64, 128] holding the history of every
    sequence: tokens 0 .. L-2 (or 0 .. L-1 with include_new_token), NaN
    elsewhere.  Returns (cache, kv_scale float32 [2] on device)."""
    if kv_dtype == KV_BF16:
        cache = torch.full((num_blocks, 2, HKV, PAGE, D), BF16_NAN_BITS, dtype=torch.int16,
                           device=device).view(torch.bfloat16)
    else:
        cache = torch.full((num_blocks, 2, HKV, PAGE, D), E4M3_NAN_CODE, dtype=torch.uint8,
                           device=device)
    hist = [int(L) if include_new_token else max(int(L) - 1, 0) for L in lengths]
    bt = torch.as_tensor(block_table, dtype=torch.int64, device=device)

    scale = [1.0, 1.0]
    if kv_dtype == KV_FP8:
        amax = [0.0, 0.0]
        for b, L in enumerate(hist):
            if L == 0:
                continue
            for w in (0, 1):
                x = _history_values(b, L, w, seed, device)[:L]
                amax[w] = max(amax[w], float(x.abs().max()))
        scale = [a / 448.0 if a > 0 else 1.0 for a in amax]

    for b, L in enumerate(hist):
        n = pages_of(L)
        if n == 0:
            continue
        pages = bt[b, :n]
        for w in (0, 1):
            x = _history_values(b, L, w, seed, device)                 # [n*64, 8, 128]
            x = x.view(n, PAGE, HKV, D).permute(0, 2, 1, 3)            # [n, 8, 64, 128]
            if kv_dtype == KV_BF16:
                cache[pages, w] = x.to(torch.bfloat16)
            else:
                codes = (x / scale[w]).to(torch.float8_e4m3fn).view(torch.uint8)
                codes = torch.where(torch.isnan(x), torch.full_like(codes, E4M3_NAN_CODE), codes)
                cache[pages, w] = codes
    kv_scale = torch.tensor(scale, dtype=torch.float32, device=device)
    return cache, kv_scale


def raw_cache_host(cache, kv_dtype):
    """A cache (or some of its pages) as a host numpy array of raw codes:
    uint16 BF16 bit patterns or uint8 E4M3 codes."""
    if kv_dtype == KV_BF16:
        return cache.view(torch.int16).cpu().numpy().view(np.uint16)
    return cache.view(torch.uint8).cpu().numpy()


def host_pages(cache, block_row, length, kv_dtype):
    """(sub_cache, row): a host copy of the raw codes of one sequence's pages,
    renumbered 0 .. n-1, and the block row that reads them in order."""
    n = pages_of(length)
    pages = torch.as_tensor(np.asarray(block_row[:n], dtype=np.int64), device=cache.device)
    return raw_cache_host(cache[pages], kv_dtype), np.arange(n)


def host_f64(t):
    """A BF16 (or any float) tensor as a float64 host array."""
    return t.float().cpu().numpy().astype(np.float64)


class Workload:
    """Everything one decode step of a named workload needs, on ``device``."""

    def __init__(self, name, seed=0, device="cuda", include_new_token=False, lengths=None,
                 kv_dtype=None):
        self.name = name
        self.seed = seed
        self.lengths = np.asarray(lengths if lengths is not None else seq_lengths(name, seed),
                                  dtype=np.int32)
        self.kv_dtype = kv_dtype if kv_dtype is not None else kv_dtype_of(name)
        self.block_table_np, self.num_blocks = block_table_for(self.lengths, seed)
        self.max_blocks = self.block_table_np.shape[1]
        B = len(self.lengths)
        self.batch = B
        self.q, self.k, self.v, self.q_norm_w, self.k_norm_w = new_token(B, seed, device)
        self.positions = torch.as_tensor(np.maximum(self.lengths - 1, 0), dtype=torch.int32, device=device)
        self.slot_mapping = torch.as_tensor(slot_mapping_for(self.lengths, self.block_table_np),
                                            dtype=torch.int64, device=device)
        self.block_table = torch.as_tensor(self.block_table_np, dtype=torch.int32, device=device)
        self.seq_lens = torch.as_tensor(self.lengths, dtype=torch.int32, device=device)
        self.cache, self.kv_scale = make_cache(self.lengths, self.block_table_np, self.num_blocks,
                                               self.kv_dtype, seed, device, include_new_token)
        self.max_pos = int(max(int(self.lengths.max()) if B else 1, 1))

    @property
    def tokens(self):
        return int(self.lengths.sum())

    def kv_bytes(self):
        """KV bytes the step must read: 8 heads x 128 x (K, V) x element size per token."""
        elem = 2 if self.kv_dtype == KV_BF16 else 1
        return self.tokens * HKV * D * 2 * elem

    def qo_bytes(self):
        return self.batch * HQ * D * 2 * 2
