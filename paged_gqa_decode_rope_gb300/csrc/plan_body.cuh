// Device code of the length-proportional split-KV planner, shared by the
// standalone planner kernel and the fused prologue + planner kernel.
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper", section "Why does dynamic scheduling matter for attention?" (64-token
// tiles dealt to compute units in proportion to each sequence's length, at
// every step).  The closed forms used here are described in plan.cu.
#pragma once

#include "common.cuh"

namespace hpc {
namespace {


// Exclusive scan of one int per thread over the CTA (kThreads threads, a
// multiple of 32, at most 1024); *total gets the sum.
template <int kThreads>
__device__ int cta_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < (kThreads / 32) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[31];
  __syncthreads();   // warp_sums is reused by the next scan
  return excl;
}

__device__ __forceinline__ int tiles_of(const int32_t* seq_lens, int b, int max_blocks,
                                        int32_t* status) {
  const int L = seq_lens[b];
  if (L < 0 || L > max_blocks * kPage) {
    atomicOr(status, HPC_STATUS_BAD_SEQ_LEN);
    return 0;
  }
  return (L + kPage - 1) / kPage;
}

template <int kThreads>
__device__ void write_empty_plan(int batch, int num_ctas, int32_t* cta_ptr, int32_t* seg_ptr) {
  for (int c = threadIdx.x; c <= num_ctas; c += kThreads) cta_ptr[c] = 0;
  for (int s = threadIdx.x; s <= batch * kHkv; s += kThreads) seg_ptr[s] = 0;
}

// floor(a * 2^32 / d) for 0 <= a < d <= 2^31 in 32-bit float and integer
// steps (double precision is slow on this part).  The estimate from an
// approximate reciprocal (relative error at most 2^-23) and two more
// roundings of at most 2^-24 on a quotient below 2^32 is within 2^10 of the
// quotient, so the exact remainder is below 2^11 d in size; one more estimate
// from that remainder (its top bits only when it passes 2^31, which needs
// d > 2^20 and so moves the estimate by less than 2^-8) lands within one of
// the quotient, and the remainder's sign and size settle the last step.
__device__ __forceinline__ uint32_t frac_quotient(uint32_t a, uint32_t d) {
  const float r = rcp_approx(static_cast<float>(d));
  uint32_t qe = __float2uint_rz(static_cast<float>(a) * r * 4294967296.0f);
  const int64_t num = static_cast<int64_t>(a) << 32;
  int64_t rem = num - static_cast<int64_t>(static_cast<uint64_t>(qe) * d);
  const float fr = (rem >= INT32_MIN && rem <= INT32_MAX)
                       ? static_cast<float>(static_cast<int32_t>(rem))
                       : static_cast<float>(static_cast<int32_t>(rem >> 12)) * 4096.0f;
  qe += static_cast<uint32_t>(__float2int_rz(fr * r));
  rem = num - static_cast<int64_t>(static_cast<uint64_t>(qe) * d);
  while (rem < 0) {
    --qe;
    rem += d;
  }
  while (rem >= static_cast<int64_t>(d)) {
    ++qe;
    rem -= d;
  }
  return qe;
}

// Division of dividends in [0, 2^31) by a divisor fixed for the whole plan,
// by multiplication: Granlund and Montgomery, "Division by invariant integers
// using multiplication" (PLDI 1994), with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(m, n) + n) >> l.  The
// planner's closed forms divide by q, k and the pieces per range in dependent
// chains; a quotient in three instructions keeps them short.
struct FastDiv {
  uint32_t d, m, l;
  // d in [1, 2^31]; 2^l - d < d, so m < 2^32
  __device__ __forceinline__ void init(uint32_t div) {
    d = div;
    l = div > 1 ? 32 - __clz(div - 1) : 0;
    m = frac_quotient((1u << l) - div, div) + 1u;
  }
  __device__ __forceinline__ int div(int n) const {
    const uint32_t un = static_cast<uint32_t>(n);
    return static_cast<int>((__umulhi(m, un) + un) >> l);
  }
};

// Pieces of the flat tile order: CTA c's range [c*q, (c+1)*q) is its home
// part [c*q, c*q + h) followed by npc - 1 pool chunks of k tiles (the last
// one may be shorter).  Pieces are numbered in flat order, npc per CTA.
struct Pieces {
  // all flat positions are < 2^31: the host keeps batch * max_blocks * 8
  // below 2^30, and a piece is formed only when it starts before T
  int q, h, k;
  int npc;   // pieces per CTA range (1 + pool chunks)
  FastDiv dq, dk, dnpc;
  // the three inverses are set up on lanes 0, 1 and 2 of every warp at once
  // and broadcast (the whole warp must call this)
  __device__ __forceinline__ void ready() {
    const int lane = threadIdx.x & 31;
    FastDiv f;
    f.init(static_cast<uint32_t>(lane == 0 ? q : (lane == 1 ? k : npc)));
    const uint32_t m = f.m, l = f.l;
    dq.d = q;
    dq.m = __shfl_sync(0xffffffffu, m, 0);
    dq.l = __shfl_sync(0xffffffffu, l, 0);
    dk.d = k;
    dk.m = __shfl_sync(0xffffffffu, m, 1);
    dk.l = __shfl_sync(0xffffffffu, l, 1);
    dnpc.d = npc;
    dnpc.m = __shfl_sync(0xffffffffu, m, 2);
    dnpc.l = __shfl_sync(0xffffffffu, l, 2);
  }
  // number of piece starts at or before flat tile x (x >= 0)
  __device__ __forceinline__ int starts_upto(int x) const {
    const int c = dq.div(x), r = x - c * q;
    int n = c * npc + 1;
    if (npc > 1 && r >= h) n += 1 + min(npc - 2, dk.div(r - h));
    return n;
  }
  __device__ __forceinline__ int id(int f) const { return starts_upto(f) - 1; }
  // first flat tile of piece p = c*npc + j
  __device__ __forceinline__ int begin(int c, int j) const {
    return c * q + (j == 0 ? 0 : h + (j - 1) * k);
  }
  // one past the last flat tile of piece p = c*npc + j (j * k stays below
  // 2 (q - h), so the sum is formed only once it is at most q)
  __device__ __forceinline__ int end(int c, int j) const {
    return c * q + h + (j == 0 ? 0 : min(q - h, j * k));
  }
};

// Shared memory of the planner, in ints: the tile prefix [batch + 1] and the
// per-CTA item bounds [num_ctas + 1] and [num_ctas].
__host__ __device__ __forceinline__ size_t plan_smem_ints(int batch, int num_ctas) {
  return static_cast<size_t>(batch) + 1 + 2 * static_cast<size_t>(num_ctas) + 1;
}

// Items of one (seq, kv_head) segment: flat tiles [s0, s0 + n) cut at piece
// starts.  Item j (global index first + j) is piece id(s0) + j clipped to the
// segment.  An item that begins on a piece start records the CTA bounds that
// start defines: the start of CTA c's range (piece c*npc) is cta_s[c]; the
// start of the piece after CTA c's home part (piece c*npc + 1) is home_s[c].
struct SegItems {
  int b, h, s0, n, first, p0;
  __device__ __forceinline__ void write(const Pieces& pc, int j, hpc_work_item* items, int* cta_s,
                                        int* home_s) const {
    const int p = p0 + j;
    const int c = pc.dnpc.div(p), jj = p - c * pc.npc;
    const int pb = pc.begin(c, jj), pe = pc.end(c, jj);
    // one 16-byte store (the item array is 16-byte aligned)
    reinterpret_cast<int4*>(items)[first + j] =
        make_int4(b, h, max(pb, s0) - s0, min(pe, s0 + n) - s0);
    if (pb >= s0) {   // the item begins on piece p's start
      if (jj == 0) cta_s[c] = first + j;
      if (pc.npc == 1 && c > 0) home_s[c - 1] = first + j;
      if (jj == 1) home_s[c] = first + j;
    }
  }
};

// The length-proportional planner, run by one CTA of kThreads threads.
// smem points at plan_smem_ints(batch, num_ctas) ints of shared memory.  One
// round trip to global memory (seq_lens); everything else is shared memory and
// arithmetic, with four block-wide scans' worth of barriers.
template <int kThreads>
__device__ void plan_dynamic_body(
    const int32_t* __restrict__ seq_lens, int batch, int max_blocks, int min_tiles, int pool_chunks,
    int pool_min_tiles, hpc_work_item* __restrict__ items, int32_t* cta_ptr, int32_t* seg_ptr,
    int32_t* home_end, int32_t* __restrict__ pool, int32_t* __restrict__ seg_done, int capacity,
    int num_ctas, int32_t* __restrict__ status, int* smem) {
  __shared__ int warp_sums[32];
  const int C = num_ctas;
  int* pre_n = smem;               // [batch + 1]
  int* cta_s = smem + batch + 1;   // [C + 1]
  int* home_s = cta_s + C + 1;     // [C]
  const int tid = threadIdx.x, lane = tid & 31;
  // read the scalar arguments into registers up front: their first reads
  // then overlap the sequence-length loads instead of stalling step 2
  asm volatile("" ::"r"(C), "r"(min_tiles), "r"(pool_chunks), "r"(pool_min_tiles), "r"(capacity));
  const int per = (batch + kThreads - 1) / kThreads;
  const int b0 = min(batch, tid * per);
  const int b1 = min(batch, b0 + per);

  // 1. tiles per sequence (staged in pre_n), then their exclusive prefix;
  //    and whether every sequence has as many tiles as sequence 0
  const int L0 = batch > 0 ? seq_lens[0] : 0;
  const int n0 = (L0 > 0 && L0 <= max_blocks * kPage) ? (L0 + kPage - 1) / kPage : -1;
  int local = 0;
  bool same = true;
  for (int b = b0; b < b1; ++b) {
    const int n = tiles_of(seq_lens, b, max_blocks, status);
    pre_n[b] = n;
    local += n;
    same = same && n == n0;
  }
  for (int x = tid; x < batch * kHkv; x += kThreads) seg_done[x] = 0;
  same = __syncthreads_and(same) != 0;
  int total_n;
  int run = cta_exclusive_scan<kThreads>(local, warp_sums, &total_n);
  for (int b = b0; b < b1; ++b) {
    const int n = pre_n[b];
    pre_n[b] = run;
    run += n;
  }
  if (tid == 0) pre_n[batch] = total_n;

  // 2. the pieces: range q, pooled tiles P in chunks of k, home part h
  //    (every thread works them out: a shared copy would cost a barrier)
  const int T = kHkv * total_n;
  Pieces pc;
  const uint32_t uC = static_cast<uint32_t>(C), uJ = static_cast<uint32_t>(pool_chunks);
  pc.q = max(min_tiles, static_cast<int>((static_cast<uint32_t>(T) + uC - 1u) / uC));
  // equal lengths with no more segments than queues: one whole segment per
  // queue (splitting them would only add partials and merges)
  if (same && batch * kHkv <= C) pc.q = max(pc.q, n0);
  uint32_t P = pool_chunks > 0 ? static_cast<uint32_t>(pc.q) / 8u : 0u;
  pc.k = P > 0 ? static_cast<int>((P + uJ - 1u) / uJ) : 1;
  if (pc.k < pool_min_tiles) {                           // chunks too short to deal
    P = 0;
    pc.k = 1;
  }
  pc.h = pc.q - static_cast<int>(P);
  pc.npc = 1 + (P > 0 ? static_cast<int>((P + pc.k - 1u) / static_cast<uint32_t>(pc.k)) : 0);
  pc.ready();
  __syncthreads();   // pre_n complete

  // 3. items per segment.  Warp w owns the segments
  //    [w * 32 * sper, (w + 1) * 32 * sper) and walks them 32 at a time (lane
  //    j takes the j-th of each group), so its segment offsets and item
  //    stores are consecutive across the lanes.  The block-wide scan gives
  //    each warp the items before its segments.
  const int nseg = batch * kHkv;
  const int sper = (nseg + kThreads - 1) / kThreads;
  const int wseg0 = (tid >> 5) * 32 * sper;
  auto seg_at = [&](int s, SegItems& g) -> int {   // fills g but first; returns the count
    g.b = s >> 3;
    g.h = s & 7;
    g.n = pre_n[g.b + 1] - pre_n[g.b];
    g.s0 = kHkv * pre_n[g.b] + g.h * g.n;
    g.p0 = g.n > 0 ? pc.id(g.s0) : 0;
    return g.n > 0 ? pc.id(g.s0 + g.n - 1) - g.p0 + 1 : 0;
  };
  local = 0;
  for (int i = 0; i < sper; ++i) {
    const int s = wseg0 + 32 * i + lane;
    SegItems g;
    if (s < nseg) local += seg_at(s, g);
  }
  int total_items;
  run = cta_exclusive_scan<kThreads>(local, warp_sums, &total_items);
  if (total_items > capacity) {
    if (tid == 0) atomicOr(status, HPC_STATUS_PLAN_OVERFLOW);
    write_empty_plan<kThreads>(batch, C, cta_ptr, seg_ptr);
    for (int c = tid; c < C; c += kThreads) home_end[c] = 0;
    if (tid == 0) pool[0] = pool[1] = pool[2] = 0;
    return;
  }
  run = __shfl_sync(0xffffffffu, run, 0);   // items before this warp's segments

  // 4. segment offsets and items.  The items of the warp's 32 segments of a
  //    group are one flat range written by the whole warp (lane j takes
  //    every 32nd), so a long segment is not left to one thread.
  for (int i = 0; i < sper; ++i) {
    const int s = wseg0 + 32 * i + lane;
    SegItems g{0, 0, 0, 0, 0, 0};
    const int cnt = s < nseg ? seg_at(s, g) : 0;
    int incl = cnt;   // inclusive scan of the counts over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int excl = incl - cnt;
    g.first = run + excl;
    if (s < nseg) seg_ptr[s] = g.first;
    const int wtotal = __shfl_sync(0xffffffffu, incl, 31);
    for (int base = 0; base < wtotal; base += 32) {
      const int v = base + lane;
      // the last lane whose range starts at or before v owns it
      int src = 0;
#pragma unroll
      for (int step = 16; step > 0; step >>= 1)
        if (__shfl_sync(0xffffffffu, excl, src + step) <= v) src += step;
      SegItems w;
      w.b = __shfl_sync(0xffffffffu, g.b, src);
      w.h = __shfl_sync(0xffffffffu, g.h, src);
      w.s0 = __shfl_sync(0xffffffffu, g.s0, src);
      w.n = __shfl_sync(0xffffffffu, g.n, src);
      w.first = __shfl_sync(0xffffffffu, g.first, src);
      w.p0 = __shfl_sync(0xffffffffu, g.p0, src);
      const int j = v - __shfl_sync(0xffffffffu, excl, src);
      if (v < wtotal) w.write(pc, j, items, cta_s, home_s);
    }
    run += wtotal;
  }
  if (tid == 0) seg_ptr[nseg] = total_items;
  //    bounds that start at or past the last tile hold no item
  for (int c = tid; c <= C; c += kThreads) {
    const int64_t f = static_cast<int64_t>(c) * pc.q;
    if (f >= T) cta_s[c] = total_items;
    if (c < C && f + (pc.npc > 1 ? pc.h : pc.q) >= T) home_s[c] = total_items;
  }
  __syncthreads();

  // 5. each CTA's range and home part; its pooled items
  //    home_end[c] .. cta_ptr[c+1]-1, listed in CTA order
  const int cper = (C + kThreads - 1) / kThreads;
  const int c0 = min(C, tid * cper), c1 = min(C, c0 + cper);
  local = 0;
  for (int c = c0; c < c1; ++c) {
    cta_ptr[c] = cta_s[c];
    home_end[c] = home_s[c];
    local += cta_s[c + 1] - home_s[c];
  }
  if (tid == 0) cta_ptr[C] = total_items;
  int pool_len;
  run = cta_exclusive_scan<kThreads>(local, warp_sums, &pool_len);
  for (int c = c0; c < c1; ++c)
    for (int i = home_s[c]; i < cta_s[c + 1]; ++i) pool[3 + run++] = i;
  if (tid == 0) {
    pool[0] = 0;          // next claim
    pool[1] = 0;          // CTAs done claiming
    pool[2] = pool_len;
  }
}

}  // namespace
}  // namespace hpc
