// Per-step split-KV planners: the length-proportional plan and the static
// equal-split comparator, both written on the device in one small CTA so the
// step needs no host round trip (and can sit in a CUDA graph).
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper", section "Why does dynamic scheduling matter for attention?": a
// static split-KV schedule assumes uniform lengths and leaves compute units
// idle on mixed batches; the HPC_ATTN scheduler deals 64-token tiles to the
// compute units in proportion to each sequence's current length at every
// step.
//
// Length-proportional plan.  With n_b = ceil(L_b / 64) and the flat order
// (seq, kv_head, tile), segment s = 8b + h covers flat tiles
// [S0, S0 + n_b), S0 = 8 * sum_{b'<b} n_b' + h * n_b.  CTA c owns
// [c*q, (c+1)*q) with q = max(min_tiles, ceil(T / C)).  Hence segment s is cut
// into floor((S0 + n_b - 1) / q) - floor(S0 / q) + 1 items, its j-th item runs
// on CTA floor(S0 / q) + j, and the first item of CTA c is the one that holds
// flat tile c*q.  Two block-wide scans (tiles, then items) give every index in
// closed form; no thread walks another thread's data.
#include "common.cuh"

namespace hpc {
namespace {

constexpr int kPlanThreads = 1024;

// Exclusive scan of one int per thread over the CTA; *total gets the sum.
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
    int s = lane < (kPlanThreads / 32) ? warp_sums[lane] : 0;
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

__device__ void write_empty_plan(int batch, int num_ctas, int32_t* cta_ptr, int32_t* seg_ptr) {
  for (int c = threadIdx.x; c <= num_ctas; c += kPlanThreads) cta_ptr[c] = 0;
  for (int s = threadIdx.x; s <= batch * kHkv; s += kPlanThreads) seg_ptr[s] = 0;
}

__global__ void __launch_bounds__(kPlanThreads) plan_dynamic_kernel(
    const int32_t* __restrict__ seq_lens, int batch, int max_blocks, int min_tiles,
    hpc_work_item* __restrict__ items, int32_t* __restrict__ cta_ptr, int32_t* seg_ptr,
    int capacity, int num_ctas, int32_t* __restrict__ status) {
  extern __shared__ int pre_n[];       // [batch + 1]: sum of n_b' for b' < b
  __shared__ int warp_sums[32];
  const int per = (batch + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(batch, static_cast<int>(threadIdx.x) * per);
  const int b1 = min(batch, b0 + per);

  // 1. tiles per sequence and their prefix
  int local = 0;
  for (int b = b0; b < b1; ++b) local += tiles_of(seq_lens, b, max_blocks, status);
  int total_n;
  int run = cta_exclusive_scan(local, warp_sums, &total_n);
  for (int b = b0; b < b1; ++b) {
    pre_n[b] = run;
    const int L = seq_lens[b];
    run += (L < 0 || L > max_blocks * kPage) ? 0 : (L + kPage - 1) / kPage;
  }
  if (threadIdx.x == 0) pre_n[batch] = total_n;
  __syncthreads();

  const int64_t T = static_cast<int64_t>(kHkv) * total_n;
  const int64_t q = max(static_cast<int64_t>(min_tiles), (T + num_ctas - 1) / num_ctas);

  // 2. items per sequence (its 8 segments) and their prefix
  local = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = pre_n[b + 1] - pre_n[b];
    if (n == 0) continue;
    for (int h = 0; h < kHkv; ++h) {
      const int64_t s0 = static_cast<int64_t>(kHkv) * pre_n[b] + static_cast<int64_t>(h) * n;
      local += static_cast<int>((s0 + n - 1) / q - s0 / q + 1);
    }
  }
  int total_items;
  run = cta_exclusive_scan(local, warp_sums, &total_items);
  if (total_items > capacity) {
    if (threadIdx.x == 0) atomicOr(status, HPC_STATUS_PLAN_OVERFLOW);
    write_empty_plan(batch, num_ctas, cta_ptr, seg_ptr);
    return;
  }

  // 3. segment offsets and the items themselves
  for (int b = b0; b < b1; ++b) {
    const int n = pre_n[b + 1] - pre_n[b];
    for (int h = 0; h < kHkv; ++h) {
      seg_ptr[b * kHkv + h] = run;
      if (n == 0) continue;
      const int64_t s0 = static_cast<int64_t>(kHkv) * pre_n[b] + static_cast<int64_t>(h) * n;
      const int64_t s1 = s0 + n;
      const int64_t c0 = s0 / q;
      const int cnt = static_cast<int>((s1 - 1) / q - c0 + 1);
      for (int j = 0; j < cnt; ++j) {
        const int64_t lo = max(s0, (c0 + j) * q);
        const int64_t hi = min(s1, (c0 + j + 1) * q);
        hpc_work_item it;
        it.seq = b;
        it.kv_head = h;
        it.tile_begin = static_cast<int32_t>(lo - s0);
        it.tile_end = static_cast<int32_t>(hi - s0);
        items[run + j] = it;
      }
      run += cnt;
    }
  }
  if (threadIdx.x == 0) seg_ptr[batch * kHkv] = total_items;
  __syncthreads();   // seg_ptr is read below by other threads

  // 4. first item of every CTA: the item that holds flat tile c*q
  for (int c = threadIdx.x; c <= num_ctas; c += kPlanThreads) {
    const int64_t f = static_cast<int64_t>(c) * q;
    if (c == num_ctas || f >= T) {
      cta_ptr[c] = total_items;
      continue;
    }
    // last sequence b with 8*pre_n[b] <= f (it has n_b > 0 because f < T)
    int lo = 0, hi = batch;   // invariant: 8*pre_n[lo] <= f < 8*pre_n[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<int64_t>(kHkv) * pre_n[mid] <= f) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int n = pre_n[b + 1] - pre_n[b];
    const int h = static_cast<int>((f - static_cast<int64_t>(kHkv) * pre_n[b]) / n);
    const int64_t s0 = static_cast<int64_t>(kHkv) * pre_n[b] + static_cast<int64_t>(h) * n;
    cta_ptr[c] = seg_ptr[b * kHkv + h] + static_cast<int>(c - s0 / q);
  }
}

__global__ void __launch_bounds__(kPlanThreads) plan_static_kernel(
    const int32_t* __restrict__ seq_lens, int batch, int max_blocks, int splits,
    hpc_work_item* __restrict__ items, int32_t* __restrict__ cta_ptr, int32_t* __restrict__ seg_ptr,
    int capacity, int num_ctas, int32_t* __restrict__ status) {
  __shared__ int warp_sums[32];
  const int per = (batch + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(batch, static_cast<int>(threadIdx.x) * per);
  const int b1 = min(batch, b0 + per);

  int local = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = tiles_of(seq_lens, b, max_blocks, status);
    if (n == 0) continue;
    const int chunk = (n + splits - 1) / splits;
    local += kHkv * ((n + chunk - 1) / chunk);
  }
  int total_items;
  int run = cta_exclusive_scan(local, warp_sums, &total_items);
  if (total_items > capacity) {
    if (threadIdx.x == 0) atomicOr(status, HPC_STATUS_PLAN_OVERFLOW);
    write_empty_plan(batch, num_ctas, cta_ptr, seg_ptr);
    return;
  }
  for (int b = b0; b < b1; ++b) {
    const int L = seq_lens[b];
    const int n = (L < 0 || L > max_blocks * kPage) ? 0 : (L + kPage - 1) / kPage;
    const int chunk = n > 0 ? (n + splits - 1) / splits : 1;
    for (int h = 0; h < kHkv; ++h) {
      seg_ptr[b * kHkv + h] = run;
      for (int t0 = 0; t0 < n; t0 += chunk) {
        hpc_work_item it;
        it.seq = b;
        it.kv_head = h;
        it.tile_begin = t0;
        it.tile_end = min(t0 + chunk, n);
        items[run++] = it;
      }
    }
  }
  if (threadIdx.x == 0) seg_ptr[batch * kHkv] = total_items;
  for (int c = threadIdx.x; c <= num_ctas; c += kPlanThreads) cta_ptr[c] = min(c, total_items);
}

int check_plan_args(const int32_t* seq_lens, int32_t batch, int32_t max_blocks, const hpc_plan* plan,
                    const int32_t* status) {
  HPC_CHECK_ARG(seq_lens && plan && status && plan->items && plan->cta_ptr && plan->seg_ptr);
  HPC_CHECK_ARG(batch >= 0 && max_blocks >= 1 && plan->num_ctas >= 1 && plan->capacity >= 0);
  if (batch > HPC_MAX_BATCH) return HPC_ERR_UNSUPPORTED;
  // keep the flat tile count 8 * sum(n_b) inside int32
  if (static_cast<int64_t>(batch) * max_blocks * kHkv >= (int64_t{1} << 31)) return HPC_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * kPage >= (int64_t{1} << 31)) return HPC_ERR_UNSUPPORTED;
  return HPC_OK;
}

}  // namespace
}  // namespace hpc

extern "C" int32_t hpc_plan_capacity(int32_t batch, int32_t num_ctas) {
  return num_ctas + hpc::kHkv * batch;
}

extern "C" int hpc_decode_plan(const int32_t* seq_lens, int32_t batch, int32_t max_blocks,
                               int32_t min_tiles, hpc_plan* plan, int32_t* status,
                               cudaStream_t stream) {
  const int rc = hpc::check_plan_args(seq_lens, batch, max_blocks, plan, status);
  if (rc != HPC_OK) return rc;
  HPC_CHECK_ARG(min_tiles >= 1);
  const size_t smem = sizeof(int) * (static_cast<size_t>(batch) + 1);
  hpc::plan_dynamic_kernel<<<1, hpc::kPlanThreads, smem, stream>>>(
      seq_lens, batch, max_blocks, min_tiles, plan->items, plan->cta_ptr, plan->seg_ptr,
      plan->capacity, plan->num_ctas, status);
  return HPC_LAUNCH_STATUS();
}

extern "C" int hpc_decode_plan_static(const int32_t* seq_lens, int32_t batch, int32_t max_blocks,
                                      int32_t splits, hpc_plan* plan, int32_t* status,
                                      cudaStream_t stream) {
  const int rc = hpc::check_plan_args(seq_lens, batch, max_blocks, plan, status);
  if (rc != HPC_OK) return rc;
  HPC_CHECK_ARG(splits >= 1);
  HPC_CHECK_ARG(static_cast<int64_t>(batch) * hpc::kHkv * splits == plan->num_ctas);
  HPC_CHECK_ARG(plan->capacity >= plan->num_ctas);
  hpc::plan_static_kernel<<<1, hpc::kPlanThreads, 0, stream>>>(
      seq_lens, batch, max_blocks, splits, plan->items, plan->cta_ptr, plan->seg_ptr,
      plan->capacity, plan->num_ctas, status);
  return HPC_LAUNCH_STATUS();
}
