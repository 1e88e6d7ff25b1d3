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
//
// Runtime dealing of the tail (pool_chunks = J > 0): SMs do not stream at
// exactly the same rate, so equal ranges finish apart.  The last
// P = floor(q / 8) tiles of every range are cut into chunks of ceil(P / J)
// tiles (no pool at all when that is below pool_min_tiles: short chunks cost
// more in per-item work than they save); the planner lists them, in CTA
// order, in a pool.  A CTA first runs
// its home part [c*q, c*q + q - P), then claims pool chunks through one
// atomic counter until the pool is empty.  Cutting at the piece boundaries
// just refines the cuts above, so the items stay in flat order and every
// (seq, kv_head) segment's items stay contiguous for the merge.
#include <mutex>


#include "plan_body.cuh"

namespace hpc {
namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_dynamic_kernel(
    const int32_t* __restrict__ seq_lens, int batch, int max_blocks, int min_tiles, int pool_chunks,
    int pool_min_tiles, hpc_work_item* __restrict__ items, int32_t* cta_ptr, int32_t* seg_ptr,
    int32_t* home_end, int32_t* __restrict__ pool, int32_t* __restrict__ seg_done, int capacity,
    int num_ctas, int32_t* __restrict__ status) {
  extern __shared__ int plan_smem[];
  plan_dynamic_body<kPlanThreads>(seq_lens, batch, max_blocks, min_tiles, pool_chunks, pool_min_tiles,
                                  items, cta_ptr, seg_ptr, home_end, pool, seg_done, capacity,
                                  num_ctas, status, plan_smem);
}

__global__ void __launch_bounds__(kPlanThreads) plan_static_kernel(
    const int32_t* __restrict__ seq_lens, int batch, int max_blocks, int splits,
    hpc_work_item* __restrict__ items, int32_t* __restrict__ cta_ptr, int32_t* __restrict__ seg_ptr,
    int32_t* __restrict__ home_end, int32_t* __restrict__ pool, int32_t* __restrict__ seg_done,
    int capacity, int num_ctas, int32_t* __restrict__ status) {
  __shared__ int warp_sums[32];
  const int per = (batch + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(batch, static_cast<int>(threadIdx.x) * per);
  const int b1 = min(batch, b0 + per);
  for (int x = threadIdx.x; x < batch * kHkv; x += kPlanThreads) seg_done[x] = 0;

  int local = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = tiles_of(seq_lens, b, max_blocks, status);
    if (n == 0) continue;
    const int chunk = (n + splits - 1) / splits;
    local += kHkv * ((n + chunk - 1) / chunk);
  }
  int total_items;
  int run = cta_exclusive_scan<kPlanThreads>(local, warp_sums, &total_items);
  if (threadIdx.x == 0) pool[0] = pool[1] = pool[2] = 0;   // a static plan has no pool
  if (total_items > capacity) {
    if (threadIdx.x == 0) atomicOr(status, HPC_STATUS_PLAN_OVERFLOW);
    write_empty_plan<kPlanThreads>(batch, num_ctas, cta_ptr, seg_ptr);
    for (int c = threadIdx.x; c < num_ctas; c += kPlanThreads) home_end[c] = 0;
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
  for (int c = threadIdx.x; c <= num_ctas; c += kPlanThreads) {
    cta_ptr[c] = min(c, total_items);
    if (c < num_ctas) home_end[c] = min(c + 1, total_items);
  }
}

// Dynamic shared memory above 48 KB needs a per-device opt-in; done once per
// device with the largest size the batch and CTA caps allow (160 KB).
cudaError_t plan_smem_optin() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(plan_dynamic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sizeof(int) *
                                            plan_smem_ints(HPC_MAX_BATCH, HPC_MAX_PLAN_CTAS)));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

int check_plan_args(const int32_t* seq_lens, int32_t batch, int32_t max_blocks, const hpc_plan* plan,
                    const int32_t* status) {
  HPC_CHECK_ARG(seq_lens && plan && status && plan->items && plan->cta_ptr && plan->seg_ptr &&
                plan->home_end && plan->pool && plan->seg_done);
  HPC_CHECK_ARG(batch >= 0 && max_blocks >= 1 && plan->num_ctas >= 1 && plan->capacity >= 0);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(plan->items) & 15) == 0);
  if (batch > HPC_MAX_BATCH) return HPC_ERR_UNSUPPORTED;
  // keep the flat tile count T = 8 * sum(n_b) below 2^30, so that every flat
  // position the planner forms (at most T plus one range) fits in int32
  if (static_cast<int64_t>(batch) * max_blocks * kHkv >= (int64_t{1} << 30)) return HPC_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * kPage >= (int64_t{1} << 31)) return HPC_ERR_UNSUPPORTED;
  return HPC_OK;
}

}  // namespace
}  // namespace hpc

extern "C" int32_t hpc_plan_capacity(int32_t batch, int32_t num_ctas, int32_t pool_chunks) {
  return num_ctas * (1 + (pool_chunks > 0 ? pool_chunks : 0)) + hpc::kHkv * batch;
}

extern "C" int hpc_decode_plan(const int32_t* seq_lens, int32_t batch, int32_t max_blocks,
                               const hpc_plan_params* params, hpc_plan* plan, int32_t* status,
                               cudaStream_t stream) {
  const int rc = hpc::check_plan_args(seq_lens, batch, max_blocks, plan, status);
  if (rc != HPC_OK) return rc;
  const hpc_plan_params def = {1, HPC_DEFAULT_POOL_CHUNKS, HPC_DEFAULT_POOL_MIN_TILES};
  const hpc_plan_params& pp = params != nullptr ? *params : def;
  const int min_tiles = pp.min_tiles, pool_chunks = pp.pool_chunks;
  HPC_CHECK_ARG(min_tiles >= 1 && pool_chunks >= 0 && pool_chunks <= 64 && pp.pool_min_tiles >= 1);
  if (plan->num_ctas > HPC_MAX_PLAN_CTAS) return HPC_ERR_UNSUPPORTED;
  const size_t smem = sizeof(int) * hpc::plan_smem_ints(batch, plan->num_ctas);
  if (smem > 48 * 1024 && hpc::plan_smem_optin() != cudaSuccess) return HPC_ERR_CUDA;
  hpc::plan_dynamic_kernel<<<1, hpc::kPlanThreads, smem, stream>>>(
      seq_lens, batch, max_blocks, min_tiles, pool_chunks, pp.pool_min_tiles, plan->items,
      plan->cta_ptr,
      plan->seg_ptr, plan->home_end, plan->pool, plan->seg_done, plan->capacity, plan->num_ctas,
      status);
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
      plan->home_end, plan->pool, plan->seg_done, plan->capacity, plan->num_ctas, status);
  return HPC_LAUNCH_STATUS();
}
