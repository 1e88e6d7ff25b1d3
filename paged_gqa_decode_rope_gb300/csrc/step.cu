// One decode step in two launches: the fused prologue and the planner in one
// kernel, then the attention with the merge fused in, launched as a
// programmatic dependent of the first so its CTAs are resident and its
// barriers set up by the time the plan and q are ready.
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper": section "Why does dynamic scheduling matter for attention?" (the
// per-step scheduler and the fused prologue) and "FP8 MoE pipeline as a single
// execution path" (chaining kernels with Programmatic Dependent Launch so the
// HBM round trips and launch gaps between them disappear; used there for the
// MoE path, applied here to the attention step).
#include <mutex>

#include "internal.h"
#include "plan_body.cuh"
#include "prologue_body.cuh"

namespace hpc {
namespace {

constexpr int kStepThreads = 256;   // one prologue block = 8 warps; the planner block too

// Block 0 plans, blocks 1 .. 9*batch run the prologue (sequence (blk-1)/9,
// head block (blk-1)%9).  The two parts read different inputs and write
// different outputs, so they need no ordering between them.
template <bool kFp8>
__global__ void __launch_bounds__(kStepThreads) prologue_plan_kernel(
    const uint16_t* q, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
    const int32_t* __restrict__ positions, const float* __restrict__ cos_sin, int32_t max_pos,
    const uint16_t* __restrict__ q_w, const uint16_t* __restrict__ k_w, float eps,
    uint8_t* __restrict__ kv_cache, int32_t num_blocks, const int64_t* __restrict__ slot_mapping,
    const float* __restrict__ kv_scale, uint16_t* q_out, const int32_t* __restrict__ seq_lens,
    int32_t batch, int32_t max_blocks, int32_t min_tiles, int32_t pool_chunks,
    int32_t pool_min_tiles, hpc_work_item* __restrict__ items, int32_t* cta_ptr, int32_t* seg_ptr,
    int32_t* home_end, int32_t* __restrict__ pool, int32_t* __restrict__ seg_done,
    int32_t capacity, int32_t num_ctas, int32_t* __restrict__ status) {
  pdl_trigger();
  extern __shared__ int step_smem[];
  if (blockIdx.x == 0) {
    plan_dynamic_body<kStepThreads>(seq_lens, batch, max_blocks, min_tiles, pool_chunks,
                                    pool_min_tiles, items, cta_ptr, seg_ptr, home_end, pool,
                                    seg_done, capacity, num_ctas, status, step_smem);
  } else {
    const int blk = blockIdx.x - 1;
    prologue_heads<kFp8, false>(blk / (kGroup + 1), blk % (kGroup + 1), q, k, v, positions, cos_sin,
                                max_pos, q_w, k_w, eps, kv_cache, num_blocks, slot_mapping,
                                kv_scale, q_out, 1.0f, status);
  }
}

// Dynamic shared memory above 48 KB (the planner's arrays for large batches
// or grids) needs a per-device opt-in, done once per device.
template <bool kFp8>
cudaError_t step_smem_optin() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(prologue_plan_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sizeof(int) *
                                            plan_smem_ints(HPC_MAX_BATCH, HPC_MAX_PLAN_CTAS)));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

}  // namespace
}  // namespace hpc

extern "C" int hpc_decode_step(const void* q, const void* k, const void* v,
                               const int32_t* positions, const float* cos_sin, int32_t max_pos,
                               const void* q_norm_w, const void* k_norm_w, float eps,
                               void* kv_cache, int32_t kv_dtype, int32_t num_blocks,
                               const int64_t* slot_mapping, const float* kv_scale,
                               const int32_t* block_table, int32_t max_blocks,
                               const int32_t* seq_lens, int32_t batch,
                               const hpc_plan_params* params, hpc_plan* plan, float* partial_o,
                               float* partial_lse, void* q_out, void* out, float sm_scale,
                               int32_t* status, cudaStream_t stream) {
  // the prologue's checks
  HPC_CHECK_ARG(q && k && v && positions && cos_sin && q_norm_w && k_norm_w && kv_cache &&
                slot_mapping && q_out && status && out);
  HPC_CHECK_ARG(batch >= 0 && max_pos > 0 && num_blocks > 0 && eps >= 0.0f);
  if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
  if (kv_dtype == HPC_KV_FP8_E4M3) HPC_CHECK_ARG(kv_scale != nullptr);
  // the planner's checks
  HPC_CHECK_ARG(seq_lens && plan && plan->items && plan->cta_ptr && plan->seg_ptr &&
                plan->home_end && plan->pool && plan->seg_done);
  HPC_CHECK_ARG(max_blocks >= 1 && plan->num_ctas >= 1 && plan->capacity >= 0);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(plan->items) & 15) == 0);
  if (batch > HPC_MAX_BATCH || plan->num_ctas > HPC_MAX_PLAN_CTAS) return HPC_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(batch) * max_blocks * hpc::kHkv >= (int64_t{1} << 30))
    return HPC_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * hpc::kPage >= (int64_t{1} << 31)) return HPC_ERR_UNSUPPORTED;
  const hpc_plan_params def = {1, HPC_DEFAULT_POOL_CHUNKS, HPC_DEFAULT_POOL_MIN_TILES};
  const hpc_plan_params& pp = params != nullptr ? *params : def;
  HPC_CHECK_ARG(pp.min_tiles >= 1 && pp.pool_chunks >= 0 && pp.pool_chunks <= 64 &&
                pp.pool_min_tiles >= 1);

  const size_t smem = sizeof(int) * hpc::plan_smem_ints(batch, plan->num_ctas);
  const dim3 grid(1 + (hpc::kGroup + 1) * batch);
  auto* cache = static_cast<uint8_t*>(kv_cache);
  auto args = [&](auto kernel) {
    kernel<<<grid, hpc::kStepThreads, smem, stream>>>(
        static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
        static_cast<const uint16_t*>(v), positions, cos_sin, max_pos,
        static_cast<const uint16_t*>(q_norm_w), static_cast<const uint16_t*>(k_norm_w), eps, cache,
        num_blocks, slot_mapping, kv_scale, static_cast<uint16_t*>(q_out), seq_lens, batch,
        max_blocks, pp.min_tiles, pp.pool_chunks, pp.pool_min_tiles, plan->items, plan->cta_ptr,
        plan->seg_ptr, plan->home_end, plan->pool, plan->seg_done, plan->capacity, plan->num_ctas,
        status);
  };
  if (kv_dtype == HPC_KV_BF16) {
    if (smem > 48 * 1024 && hpc::step_smem_optin<false>() != cudaSuccess) return HPC_ERR_CUDA;
    args(hpc::prologue_plan_kernel<false>);
  } else {
    if (smem > 48 * 1024 && hpc::step_smem_optin<true>() != cudaSuccess) return HPC_ERR_CUDA;
    args(hpc::prologue_plan_kernel<true>);
  }
  if (cudaPeekAtLastError() != cudaSuccess) return HPC_ERR_CUDA;
  return hpc::launch_decode_attn(q_out, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, hpc::default_attn_options(), plan,
                                 partial_o, partial_lse,
                                 sm_scale, status, nullptr, out, true, stream);
}
