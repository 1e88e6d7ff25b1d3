"""Split-KV schedules: the length-proportional planner and the static one.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
Hopper" (24-ai.news, 2026-07-06), section "Why does dynamic scheduling matter
for attention?".  A static split-KV schedule assumes uniform lengths and leaves
compute units idle on mixed batches; the HPC_ATTN scheduler instead deals
64-token tiles to compute units in proportion to each sequence's current
length at every step.

Reading (the pages give no formula): flatten every (sequence, KV head) tile in
(sequence, kv_head, tile) order; give compute unit c the contiguous flat range
[c*q, min((c+1)*q, T)) with q = max(min_tiles, ceil(T / C)); a work item is that
range cut at (sequence, kv_head) boundaries.  Each unit then streams the same
number of tiles (up to the last one), so work is proportional to length.

The static comparator splits every (sequence, kv_head) into S chunks of
ceil(n/S) tiles, one chunk per compute unit, whatever the length.

A work item is (seq, kv_head, tile_begin, tile_end), tile_end exclusive.
"""

PAGE = 64
HKV = 8


def num_tiles(length):
    """64-token tiles of a sequence of ``length`` tokens (the last may be partial)."""
    return -(-int(length) // PAGE) if length > 0 else 0


def plan_dynamic(seq_lens, num_ctas, min_tiles=1):
    """Length-proportional plan.

    Returns (items, cta_ptr, seg_ptr): ``items`` a list of 4-tuples ordered by
    compute unit (and so by segment and tile), ``cta_ptr`` [C+1] the first item
    of each unit, ``seg_ptr`` [B*8+1] the first item of each (seq, kv_head)
    segment (segment s = seq * 8 + kv_head).
    """
    B = len(seq_lens)
    n = [num_tiles(L) for L in seq_lens]
    T = HKV * sum(n)
    q = max(int(min_tiles), -(-T // num_ctas)) if T > 0 else max(int(min_tiles), 1)

    # segments in flat order, with their start offsets
    segments = []
    start = 0
    for b in range(B):
        for h in range(HKV):
            segments.append((b, h, start, start + n[b]))
            start += n[b]

    items, owner = [], []
    cta_ptr = [0] * (num_ctas + 1)
    seg_first = []
    for (b, h, s0, s1) in segments:
        seg_first.append(len(items))
        t = s0
        while t < s1:
            c = t // q                       # the unit that owns flat tile t
            end = min(s1, (c + 1) * q)
            items.append((b, h, t - s0, end - s0))
            owner.append(c)
            t = end
    seg_ptr = seg_first + [len(items)]

    # cta_ptr[c] = index of the first item owned by a unit >= c
    i = 0
    for c in range(num_ctas + 1):
        while i < len(items) and owner[i] < c:
            i += 1
        cta_ptr[c] = i
    return items, cta_ptr, seg_ptr


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


def check_coverage(seq_lens, items, cta_ptr, seg_ptr):
    """Assert that a plan covers every (seq, kv_head, tile) exactly once and
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
    return len(items)
