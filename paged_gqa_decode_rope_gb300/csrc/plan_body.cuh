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
struct Pieces {
  // all flat positions are < 2^31: the host checks batch * max_blocks * 8
  int q, h, k;
  int npc;   // pieces per CTA range (1 + pool chunks)
  // number of piece starts at or before flat tile x (x >= 0)
  __device__ __forceinline__ int starts_upto(int x) const {
    const int c = x / q, r = x - c * q;
    int n = c * npc + 1;
    if (npc > 1 && r >= h) n += 1 + min(npc - 2, (r - h) / k);
    return n;
  }
  __device__ __forceinline__ int id(int f) const { return starts_upto(f) - 1; }
  __device__ __forceinline__ int begin(int p) const {
    const int c = p / npc, j = p - c * npc;
    return c * q + (j == 0 ? 0 : h + (j - 1) * k);
  }
  __device__ __forceinline__ int end(int p) const {
    const int c = p / npc, j = p - c * npc;
    return c * q + (j == 0 ? h : min(q, h + j * k));
  }
};

// Index of the item holding flat tile f (total_items if f >= T).
__device__ int item_at(int64_t f, int T, int total_items, const int* pre_n, int batch,
                       const int32_t* seg_ptr, const Pieces& pc) {
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
  return seg_ptr[b * kHkv + h] + pc.id(ff) - pc.id(s0);
}

// The length-proportional planner, run by one CTA of kThreads threads.
// pre_n points at 2 * (batch + 1) ints of shared memory.
template <int kThreads>
__device__ void plan_dynamic_body(
    const int32_t* __restrict__ seq_lens, int batch, int max_blocks, int min_tiles, int pool_chunks,
    int pool_min_tiles, hpc_work_item* __restrict__ items, int32_t* cta_ptr, int32_t* seg_ptr,
    int32_t* home_end, int32_t* __restrict__ pool, int32_t* __restrict__ seg_done, int capacity,
    int num_ctas, int32_t* __restrict__ status, int* pre_n) {
  // pre_n[0..batch]: sum of n_b' for b' < b; followed by pre_items[0..batch]
  __shared__ int warp_sums[32];
  const int per = (batch + kThreads - 1) / kThreads;
  const int b0 = min(batch, static_cast<int>(threadIdx.x) * per);
  const int b1 = min(batch, b0 + per);
  for (int x = threadIdx.x; x < batch * kHkv; x += kThreads) seg_done[x] = 0;

  // 1. tiles per sequence and their prefix
  int local = 0;
  for (int b = b0; b < b1; ++b) local += tiles_of(seq_lens, b, max_blocks, status);
  int total_n;
  int run = cta_exclusive_scan<kThreads>(local, warp_sums, &total_n);
  for (int b = b0; b < b1; ++b) {
    pre_n[b] = run;
    const int L = seq_lens[b];
    run += (L < 0 || L > max_blocks * kPage) ? 0 : (L + kPage - 1) / kPage;
  }
  if (threadIdx.x == 0) pre_n[batch] = total_n;
  __syncthreads();

  const int T = kHkv * total_n;
  Pieces pc;
  pc.q = max(min_tiles, (T + num_ctas - 1) / num_ctas);
  int P = pool_chunks > 0 ? pc.q / 8 : 0;                // pooled tiles per CTA range
  pc.k = P > 0 ? (P + pool_chunks - 1) / pool_chunks : 1;
  if (pc.k < pool_min_tiles) {                           // chunks too short to deal
    P = 0;
    pc.k = 1;
  }
  pc.h = pc.q - P;
  pc.npc = 1 + (P > 0 ? (P + pc.k - 1) / pc.k : 0);

  // 2. items per sequence (its 8 segments) and their prefix
  local = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = pre_n[b + 1] - pre_n[b];
    if (n == 0) continue;
    for (int h = 0; h < kHkv; ++h) {
      const int s0 = kHkv * pre_n[b] + h * n;
      local += pc.id(s0 + n - 1) - pc.id(s0) + 1;
    }
  }
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
  int* pre_items = pre_n + batch + 1;  // [batch + 1]
  for (int b = b0; b < b1; ++b) {
    pre_items[b] = run;
    const int n = pre_n[b + 1] - pre_n[b];
    for (int h = 0; h < kHkv; ++h) {
      seg_ptr[b * kHkv + h] = run;
      if (n == 0) continue;
      const int s0 = kHkv * pre_n[b] + h * n;
      run += pc.id(s0 + n - 1) - pc.id(s0) + 1;
    }
  }
  if (threadIdx.x == 0) {
    seg_ptr[batch * kHkv] = total_items;
    pre_items[batch] = total_items;
  }
  __syncthreads();   // seg_ptr / pre_items are read below by other threads

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
    int h = kHkv - 1;
    while (seg_ptr[b * kHkv + h] > i) --h;
    const int s0 = kHkv * pre_n[b] + h * n;
    const int p = pc.id(s0) + (i - seg_ptr[b * kHkv + h]);
    hpc_work_item it;
    it.seq = b;
    it.kv_head = h;
    it.tile_begin = max(s0, pc.begin(p)) - s0;
    it.tile_end = min(s0 + n, pc.end(p)) - s0;
    items[i] = it;
  }

  // 4. each CTA's range (first item holds flat tile c*q) and home part (the
  //    first pool item holds flat tile c*q + h)
  for (int c = threadIdx.x; c <= num_ctas; c += kThreads) {
    const int64_t f = static_cast<int64_t>(c) * pc.q;
    cta_ptr[c] = c == num_ctas ? total_items : item_at(f, T, total_items, pre_n, batch, seg_ptr, pc);
    if (c < num_ctas)
      home_end[c] = item_at(f + (P > 0 ? pc.h : pc.q), T, total_items, pre_n, batch, seg_ptr, pc);
  }
  __syncthreads();   // cta_ptr / home_end are read below by other threads

  // 5. the pool: every CTA's items home_end[c] .. cta_ptr[c+1]-1, in CTA order
  const int cper = (num_ctas + kThreads - 1) / kThreads;
  const int c0 = min(num_ctas, static_cast<int>(threadIdx.x) * cper);
  const int c1 = min(num_ctas, c0 + cper);
  local = 0;
  for (int c = c0; c < c1; ++c) local += cta_ptr[c + 1] - home_end[c];
  int pool_len;
  run = cta_exclusive_scan<kThreads>(local, warp_sums, &pool_len);
  for (int c = c0; c < c1; ++c)
    for (int i = home_end[c]; i < cta_ptr[c + 1]; ++i) pool[3 + run++] = i;
  if (threadIdx.x == 0) {
    pool[0] = 0;          // next claim
    pool[1] = 0;          // CTAs done claiming
    pool[2] = pool_len;
  }
}

}  // namespace
}  // namespace hpc
