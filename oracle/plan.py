"""Split-KV schedules: the length-proportional planner and the static one.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
Hopper" (24-ai.news, 2026-07-06), section "Why does dynamic scheduling matter
for attention?".  A static split-KV schedule assumes uniform lengths and leaves
compute units idle on mixed batches; the HPC_ATTN scheduler instead deals
64-token tiles to compute units in proportion to each sequence's current
length at every step.

Reading (the pages give no formula): flatten every (sequence, KV head) tile in
(sequence, kv_head, tile) order; compute unit c is given the contiguous flat
range [c*q, min((c+1)*q, T)) with q = max(min_tiles, ceil(T / C)); a work item
is a piece of that range cut at (sequence, kv_head) boundaries.  Each unit then
streams the same number of tiles, so work is proportional to length.  When every
sequence has the same number of tiles n and the B*8 segments are no more than
the units, q is raised to n: each unit takes whole segments (the page notes
that a static split suits uniform lengths; splitting equal segments further
only adds partial results to merge).

Runtime dealing of the tail (``pool_chunks`` = J > 0): units do not run at
exactly the same speed, so the last P = floor(q / 8) tiles of every unit's
range are cut into chunks of k = ceil(P / J) tiles and pooled; a unit that
has finished its home part [c*q, c*q + q - P) claims pool chunks, in pool
order, until none is left.  Chunks shorter than ``pool_min_tiles`` are not
worth dealing at run time: then nothing is pooled.  Every tile is still dealt
exactly once.  J = 0 gives the plain plan above.

The static comparator splits every (sequence, kv_head) into S chunks of
ceil(n/S) tiles, one chunk per compute unit, whatever the length.

A work item is (seq, kv_head, tile_begin, tile_end), tile_end exclusive.
"""

PAGE = 64
HKV = 8


def num_tiles(length):
    """64-token tiles of a sequence of ``length`` tokens (the last may be partial)."""
    return -(-int(length) // PAGE) if length > 0 else 0


def plan_dynamic(seq_lens, num_ctas, min_tiles=1, pool_chunks=0, pool_min_tiles=1):
    """Length-proportional plan.

    Returns (items, cta_ptr, seg_ptr, home_end, pool):
      items     4-tuples in flat (seq, kv_head, tile) order
      cta_ptr   [C+1]: unit c's range holds items cta_ptr[c] .. cta_ptr[c+1]-1
      seg_ptr   [B*8+1]: segment s = seq*8 + kv_head owns items
                seg_ptr[s] .. seg_ptr[s+1]-1
      home_end  [C]: unit c runs items cta_ptr[c] .. home_end[c]-1 itself;
                items home_end[c] .. cta_ptr[c+1]-1 go to the pool
      pool      pooled item indices, in claim order (unit order, then item)
    """
    B = len(seq_lens)
    n = [num_tiles(L) for L in seq_lens]
    T = HKV * sum(n)
    q = max(int(min_tiles), -(-T // num_ctas)) if T > 0 else max(int(min_tiles), 1)
    if B > 0 and n[0] > 0 and all(x == n[0] for x in n) and B * HKV <= num_ctas:
        q = max(q, n[0])
    P = q // 8 if pool_chunks > 0 else 0
    k = -(-P // pool_chunks) if P > 0 else 1
    if k < pool_min_tiles:                     # chunks too short to deal
        P, k = 0, 1
    h = q - P                                  # home tiles of every unit

    def piece(f):
        """(unit, piece) that owns flat tile f; piece 0 is the home part."""
        c, r = divmod(f, q)
        return (c, 0) if r < h else (c, 1 + (r - h) // k)

    def piece_end(c, j):
        return c * q + (h if j == 0 else min(q, h + j * k))

    items, owner = [], []
    start = 0
    seg_ptr = []
    for b in range(B):
        for hh in range(HKV):
            s0, s1 = start, start + n[b]
            seg_ptr.append(len(items))
            t = s0
            while t < s1:
                c, j = piece(t)
                end = min(s1, piece_end(c, j))
                items.append((b, hh, t - s0, end - s0))
                owner.append((c, j))
                t = end
            start = s1
    seg_ptr.append(len(items))

    cta_ptr, home_end = [], []
    i = 0
    for c in range(num_ctas + 1):
        while i < len(items) and owner[i][0] < c:
            i += 1
        cta_ptr.append(i)
    for c in range(num_ctas):
        i = cta_ptr[c]
        while i < cta_ptr[c + 1] and owner[i][1] == 0:
            i += 1
        home_end.append(i)
    pool = [i for c in range(num_ctas) for i in range(home_end[c], cta_ptr[c + 1])]
    return items, cta_ptr, seg_ptr, home_end, pool


def plan_static(seq_lens, splits):
    """Static equal split: every segment cut into ``splits`` chunks of
    ceil(n/splits) tiles; unit c runs item c (one item per unit).

    Returns (items, cta_ptr, seg_ptr, num_ctas) with num_ctas = B*8*splits.
    """
    B = len(seq_lens)
    items, seg_ptr = [], []
    for b in range(B):
        nb = num_tiles(seq_lens[b])
        chunk = -(-nb // splits) if nb > 0 else 1
        for h in range(HKV):
            seg_ptr.append(len(items))
            for t0 in range(0, nb, chunk):
                items.append((b, h, t0, min(t0 + chunk, nb)))
    seg_ptr.append(len(items))
    num_ctas = B * HKV * splits
    cta_ptr = [min(c, len(items)) for c in range(num_ctas + 1)]
    return items, cta_ptr, seg_ptr, num_ctas


def check_coverage(seq_lens, items, cta_ptr, seg_ptr, home_end=None, pool=None):
    """Assert that a plan deals every (seq, kv_head, tile) exactly once and
    that its index arrays are consistent.  Returns the number of items."""
    B = len(seq_lens)
    want = {}
    for b in range(B):
        for h in range(HKV):
            for t in range(num_tiles(seq_lens[b])):
                want[(b, h, t)] = 0
    for (b, h, t0, t1) in items:
        assert 0 <= t0 < t1 <= num_tiles(seq_lens[b]), (b, h, t0, t1)
        for t in range(t0, t1):
            want[(b, h, t)] += 1
    assert all(v == 1 for v in want.values()), "a tile is missed or repeated"
    assert cta_ptr[0] == 0 and cta_ptr[-1] == len(items)
    assert all(a <= b for a, b in zip(cta_ptr, cta_ptr[1:]))
    assert len(seg_ptr) == B * HKV + 1 and seg_ptr[-1] == len(items)
    for s in range(B * HKV):
        for i in range(seg_ptr[s], seg_ptr[s + 1]):
            assert items[i][0] * HKV + items[i][1] == s
        # items of a segment are in tile order and contiguous
        ts = [items[i][2:] for i in range(seg_ptr[s], seg_ptr[s + 1])]
        assert all(a[1] == b[0] for a, b in zip(ts, ts[1:]))
    if home_end is not None:
        # each item is run exactly once: by its home unit or from the pool
        runs = []
        for c in range(len(cta_ptr) - 1):
            assert cta_ptr[c] <= home_end[c] <= cta_ptr[c + 1]
            runs += list(range(cta_ptr[c], home_end[c]))
        runs += list(pool)
        assert sorted(runs) == list(range(len(items))), "an item is run twice or never"
    return len(items)
