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

// Pieces of the flat tile order: CTA c's range [c*q, (c+1)*q) is its home
// part [c*q, c*q + h) followed by npc - 1 pool chunks of k tiles (the last
// one may be shorter).  Pieces are numbered in flat order, npc per CTA.
// Division of dividends in [0, 2^31) by a divisor fixed for the whole plan,
// by multiplication: Granlund and Montgomery, "Division by invariant integers
// using multiplication" (PLDI 1994), with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(m, n) + n) >> l.  The
// planner's closed forms divide by q, k and the pieces per range in long
// dependent chains; a hardware-free quotient keeps them short.
struct FastDiv {
  uint32_t d, m, l;
  __device__ __forceinline__ void init(uint32_t div) {
    d = div;
    l = 0;
    while ((1u << l) < d) ++l;
    m = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1);
  }
  __device__ __forceinline__ int div(int n) const {
    const uint32_t un = static_cast<uint32_t>(n);
    return static_cast<int>((__umulhi(m, un) + un) >> l);
  }
};

struct Pieces {
  // all flat positions are < 2^31: the host checks batch * max_blocks * 8
  int q, h, k;
  int npc;   // pieces per CTA range (1 + pool chunks)
  FastDiv dq, dk, dnpc;
  __device__ __forceinline__ void ready() {
    dq.init(q);
    dk.init(k);
    dnpc.init(npc);
  }
  // number of piece starts at or before flat tile x (x >= 0)
  __device__ __forceinline__ int starts_upto(int x) const {
    const int c = dq.div(x), r = x - c * q;
    int n = c * npc + 1;
    if (npc > 1 && r >= h) n += 1 + min(npc - 2, dk.div(r - h));
    return n;
  }
  __device__ __forceinline__ int id(int f) const { return starts_upto(f) - 1; }
  __device__ __forceinline__ int begin(int p) const {
    const int c = dnpc.div(p), j = p - c * npc;
    return c * q + (j == 0 ? 0 : h + (j - 1) * k);
  }
  __device__ __forceinline__ int end(int p) const {
    const int c = dnpc.div(p), j = p - c * npc;
    return c * q + (j == 0 ? h : min(q, h + j * k));
  }
};

// Shared-memory view of the plan under construction: pre_n[b] = tiles of
// sequences before b (per KV head), pre_items[b] = items before sequence b.
// Every index the planner writes is derived from these two prefixes and the
// piece arithmetic, so nothing it wrote to global memory is read back.
struct PlanView {
  const int* pre_n;
  const int* pre_items;
  int batch;
  Pieces pc;
  // items of segment (b, h)
  __device__ __forceinline__ int seg_items(int b, int h) const {
    const int n = pre_n[b + 1] - pre_n[b];
    if (n == 0) return 0;
    const int s0 = kHkv * pre_n[b] + h * n;
    return pc.id(s0 + n - 1) - pc.id(s0) + 1;
  }
  // index of the first item of segment (b, h)
  __device__ __forceinline__ int seg_first(int b, int h) const {
    int i = pre_items[b];
    for (int x = 0; x < h; ++x) i += seg_items(b, x);
    return i;
  }
  // index of the item holding flat tile f (total_items if f >= T)
  __device__ int item_at(int64_t f, int T, int total_items) const {
    if (f >= T) return total_items;
    const int ff = static_cast<int>(f);
    int lo = 0, hi = batch;   // invariant: 8*pre_n[lo] <= f < 8*pre_n[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (kHkv * pre_n[mid] <= ff) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int n = pre_n[b + 1] - pre_n[b];   // > 0 because f < 8*pre_n[b+1]
    const int h = (ff - kHkv * pre_n[b]) / n;
    const int s0 = kHkv * pre_n[b] + h * n;
    return seg_first(b, h) + pc.id(ff) - pc.id(s0);
  }
};

// The length-proportional planner, run by one CTA of kThreads threads.
// smem points at 2 * (batch + 1) ints of shared memory.  One round trip to
// global memory (seq_lens); everything else is shared memory and arithmetic.
template <int kThreads>
__device__ void plan_dynamic_body(
    const int32_t* __restrict__ seq_lens, int batch, int max_blocks, int min_tiles, int pool_chunks,
    int pool_min_tiles, hpc_work_item* __restrict__ items, int32_t* cta_ptr, int32_t* seg_ptr,
    int32_t* home_end, int32_t* __restrict__ pool, int32_t* __restrict__ seg_done, int capacity,
    int num_ctas, int32_t* __restrict__ status, int* smem) {
  __shared__ int warp_sums[32];
  int* pre_n = smem;                   // [batch + 1]
  int* pre_items = smem + batch + 1;   // [batch + 1]
  const int per = (batch + kThreads - 1) / kThreads;
  const int b0 = min(batch, static_cast<int>(threadIdx.x) * per);
  const int b1 = min(batch, b0 + per);
  for (int x = threadIdx.x; x < batch * kHkv; x += kThreads) seg_done[x] = 0;

  // 1. tiles per sequence (staged in pre_n), then their exclusive prefix
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = tiles_of(seq_lens, b, max_blocks, status);
    pre_n[b] = n;
    local += n;
  }
  int total_n;
  int run = cta_exclusive_scan<kThreads>(local, warp_sums, &total_n);
  for (int b = b0; b < b1; ++b) {
    const int n = pre_n[b];
    pre_n[b] = run;
    run += n;
  }
  if (threadIdx.x == 0) pre_n[batch] = total_n;
  __syncthreads();

  const int T = kHkv * total_n;
  PlanView v;
  v.pre_n = pre_n;
  v.pre_items = pre_items;
  v.batch = batch;
  Pieces& pc = v.pc;
  pc.q = max(min_tiles, (T + num_ctas - 1) / num_ctas);
  int P = pool_chunks > 0 ? pc.q / 8 : 0;                // pooled tiles per CTA range
  pc.k = P > 0 ? (P + pool_chunks - 1) / pool_chunks : 1;
  if (pc.k < pool_min_tiles) {                           // chunks too short to deal
    P = 0;
    pc.k = 1;
  }
  pc.h = pc.q - P;
  pc.npc = 1 + (P > 0 ? (P + pc.k - 1) / pc.k : 0);
  pc.ready();

  // 2. items per sequence (its 8 segments) and their prefix
  local = 0;
  for (int b = b0; b < b1; ++b)
    for (int h = 0; h < kHkv; ++h) local += v.seg_items(b, h);
  int total_items;
  run = cta_exclusive_scan<kThreads>(local, warp_sums, &total_items);
  if (total_items > capacity) {
    if (threadIdx.x == 0) atomicOr(status, HPC_STATUS_PLAN_OVERFLOW);
    write_empty_plan<kThreads>(batch, num_ctas, cta_ptr, seg_ptr);
    for (int c = threadIdx.x; c < num_ctas; c += kThreads) home_end[c] = 0;
    if (threadIdx.x == 0) pool[0] = pool[1] = pool[2] = 0;
    return;
  }

  // 3. segment offsets, and the first item of every sequence (in smem)
  for (int b = b0; b < b1; ++b) {
    pre_items[b] = run;
    for (int h = 0; h < kHkv; ++h) {
      seg_ptr[b * kHkv + h] = run;
      run += v.seg_items(b, h);
    }
  }
  if (threadIdx.x == 0) {
    seg_ptr[batch * kHkv] = total_items;
    pre_items[batch] = total_items;
  }
  __syncthreads();   // pre_items is read below by other threads

  //    the items, one per thread: item i lies in the last sequence b with
  //    pre_items[b] <= i and, inside it, in the segment whose range holds i
  for (int i = threadIdx.x; i < total_items; i += kThreads) {
    int lo = 0, hi = batch;   // invariant: pre_items[lo] <= i < pre_items[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre_items[mid] <= i) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int n = pre_n[b + 1] - pre_n[b];
    int h = 0, first = pre_items[b];
    for (int c = v.seg_items(b, 0); first + c <= i; c = v.seg_items(b, h)) {
      first += c;
      ++h;
    }
    const int s0 = kHkv * pre_n[b] + h * n;
    const int p = pc.id(s0) + (i - first);
    hpc_work_item it;
    it.seq = b;
    it.kv_head = h;
    it.tile_begin = max(s0, pc.begin(p)) - s0;
    it.tile_end = min(s0 + n, pc.end(p)) - s0;
    items[i] = it;
  }

  // 4. each CTA's range (its first item holds flat tile c*q), home part (the
  //    first pool item holds flat tile c*q + h) and pooled items
  //    home_end[c] .. cta_ptr[c+1]-1, listed in CTA order
  const int cper = (num_ctas + kThreads - 1) / kThreads;
  const int c0 = min(num_ctas, static_cast<int>(threadIdx.x) * cper);
  const int c1 = min(num_ctas, c0 + cper);
  local = 0;
  for (int c = c0; c < c1; ++c) {
    const int64_t f = static_cast<int64_t>(c) * pc.q;
    const int first = v.item_at(f, T, total_items);
    const int home = v.item_at(f + (P > 0 ? pc.h : pc.q), T, total_items);
    const int next = v.item_at(f + pc.q, T, total_items);
    cta_ptr[c] = first;
    home_end[c] = home;
    local += next - home;
  }
  if (threadIdx.x == 0) cta_ptr[num_ctas] = total_items;
  int pool_len;
  run = cta_exclusive_scan<kThreads>(local, warp_sums, &pool_len);
  for (int c = c0; c < c1; ++c) {
    const int64_t f = static_cast<int64_t>(c) * pc.q;
    const int home = v.item_at(f + (P > 0 ? pc.h : pc.q), T, total_items);
    const int next = v.item_at(f + pc.q, T, total_items);
    for (int i = home; i < next; ++i) pool[3 + run++] = i;
  }
  if (threadIdx.x == 0) {
    pool[0] = 0;          // next claim
    pool[1] = 0;          // CTAs done claiming
    pool[2] = pool_len;
  }
}

}  // namespace
}  // namespace hpc
