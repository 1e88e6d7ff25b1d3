// Prefill and mixed prefill + decode batches through the same paged cache:
// attention of any number of new tokens per sequence (a prompt chunk), each
// new token seeing the history and the new tokens up to itself.
//
// Source: page "[vllm] Introducing the HPC-Ops attention backend" (the
// backend serves prefill, decode and mixed batches); page "vLLM and Tencent
// Hunyuan upstream two HPC backends for NVIDIA Hopper", intro of "Two new HPC
// backends in the vLLM ecosystem" (64 query heads, 8 KV heads, head_dim 128,
// paged KV in 64-token blocks).  The attention is the decode attention of
// the same pages with q_len new tokens and the causal order among them.
//
// This file holds the unit plan and the C entry points; the attention kernel
// (tcgen05, 32 new tokens x 8 query heads per unit, two 128-row tiles sharing
// each K/V page) is in prefill_tc.cuh.  Units are dealt at run time from one
// atomic counter to a persistent grid of one CTA per SM; within a sequence
// the units with the most keys come first.
#include "attn_kernel.cuh"
#include "plan_body.cuh"
#include "prefill_tc.cuh"

namespace hpc {
namespace {

// Units of every sequence (8 kv heads x blocks of 32 new tokens) and their prefix;
// zeroes the claim counters.  One CTA of kPlanThreads threads.
constexpr int kPfPlanThreads = 1024;

__global__ void __launch_bounds__(kPfPlanThreads) prefill_plan_kernel(
    const int32_t* __restrict__ query_start, int32_t batch, int32_t* __restrict__ unit_ptr,
    int32_t* __restrict__ counters, int32_t* __restrict__ status) {
  __shared__ int warp_sums[32];
  const int per = (batch + kPfPlanThreads - 1) / kPfPlanThreads;
  const int b0 = min(batch, static_cast<int>(threadIdx.x) * per);
  const int b1 = min(batch, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = query_start[b + 1] - query_start[b];
    if (n < 0) {
      atomicOr(status, HPC_STATUS_BAD_SEQ_LEN);
      continue;
    }
    local += kHkv * ((n + tc::kUnitTokens - 1) / tc::kUnitTokens);
  }
  int total;
  int run = cta_exclusive_scan<kPfPlanThreads>(local, warp_sums, &total);
  for (int b = b0; b < b1; ++b) {
    unit_ptr[b] = run;
    const int n = query_start[b + 1] - query_start[b];
    if (n > 0) run += kHkv * ((n + tc::kUnitTokens - 1) / tc::kUnitTokens);
  }
  if (threadIdx.x == 0) {
    unit_ptr[batch] = total;
    counters[0] = 0;   // next unit
    counters[1] = 0;   // CTAs done
  }
}

// Staged pages (hpc_prefill_attn_staged): page_ptr[b] = first staged page of
// sequence b (its ceil(L_b / 64) pages in order), page_ptr[batch] = all of
// them.  One CTA of kPfPlanThreads threads.
__global__ void __launch_bounds__(kPfPlanThreads) stage_plan_kernel(
    const int32_t* __restrict__ seq_lens, int32_t batch, int32_t max_blocks,
    int32_t* __restrict__ page_ptr, int32_t* __restrict__ status) {
  __shared__ int warp_sums[32];
  const int per = (batch + kPfPlanThreads - 1) / kPfPlanThreads;
  const int b0 = min(batch, static_cast<int>(threadIdx.x) * per);
  const int b1 = min(batch, b0 + per);
  auto pages = [&](int b) {
    const int L = seq_lens[b];
    if (L < 0 || L > max_blocks * kPage) return 0;   // the attention reports the sequence
    return (L + kPage - 1) / kPage;
  };
  int local = 0;
  for (int b = b0; b < b1; ++b) local += pages(b);
  int total;
  int run = cta_exclusive_scan<kPfPlanThreads>(local, warp_sums, &total);
  for (int b = b0; b < b1; ++b) {
    page_ptr[b] = run;
    run += pages(b);
  }
  if (threadIdx.x == 0) page_ptr[batch] = total;
}

// Every page the batch reads, E4M3 codes -> BF16 (exact: every E4M3 value is
// a BF16 value) into its staged page: staged page page_ptr[b] + j holds
// block block_table[b][j] of sequence b.  The work is split into 8 KB pieces
// (one K or V page of one KV head), dealt grid-stride, so a batch of few long
// pages still spreads over every SM; 256 threads, 16 codes a thread and
// step, both loads and stores coalesced.  Pages past the staging capacity are
// left (their sequences are reported by the attention); a bad block id
// stages nothing (the attention masks that tile by the real block table).
constexpr int kStageThreads = 256;
__global__ void __launch_bounds__(kStageThreads) stage_convert_kernel(
    const uint8_t* __restrict__ cache, int32_t num_blocks, const int32_t* __restrict__ block_table,
    int32_t max_blocks, int32_t batch, const int32_t* __restrict__ page_ptr, int32_t staged_pages,
    uint16_t* __restrict__ staged) {
  constexpr int kPieces = 2 * kHkv;                 // K and V of 8 heads per block
  constexpr int kPieceChunks = kPage * kD / 16;     // 16-code chunks of a piece (512)
  const int64_t total = static_cast<int64_t>(min(page_ptr[batch], staged_pages)) * kPieces;
  for (int64_t u = blockIdx.x; u < total; u += gridDim.x) {
    const int pg = static_cast<int>(u / kPieces), piece = static_cast<int>(u % kPieces);
    int lo = 0, hi = batch;   // the last b with page_ptr[b] <= pg
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (page_ptr[mid] <= pg) lo = mid;
      else hi = mid;
    }
    const int bid = block_table[static_cast<int64_t>(lo) * max_blocks + (pg - page_ptr[lo])];
    if (bid < 0 || bid >= num_blocks) continue;
    const uint4* src = reinterpret_cast<const uint4*>(
        cache + (static_cast<int64_t>(bid) * kPieces + piece) * kPieceChunks * 16);
    uint4* dst = reinterpret_cast<uint4*>(
        staged + (static_cast<int64_t>(pg) * kPieces + piece) * kPieceChunks * 16);
#pragma unroll
    for (int z = threadIdx.x; z < kPieceChunks; z += kStageThreads) {
      const uint4 w = src[z];
      const uint32_t in[4] = {w.x, w.y, w.z, w.w};
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // two codes -> f16x2 (exact) -> two floats -> bf16x2 (exact)
        const uint32_t h0 = e4m3x2_to_f16x2(static_cast<uint16_t>(in[k]));
        const uint32_t h1 = e4m3x2_to_f16x2(static_cast<uint16_t>(in[k] >> 16));
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
        o[2 * k] = pack_bf16(f0.x, f0.y);
        o[2 * k + 1] = pack_bf16(f1.x, f1.y);
      }
      dst[2 * z] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[2 * z + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

template <bool kFp8>
cudaError_t prefill_tc_smem_optin() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  // the warpgroups' raised register budgets must fit what a CTA is launched
  // with, or the raise would wait for registers that never come
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<kFp8>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * tc::Cfg<kFp8>::kThreads < tc::regs_needed<kFp8>())
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(prefill_tc_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           tc::kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

}  // namespace
}  // namespace hpc

extern "C" int hpc_prefill_plan(const int32_t* query_start, int32_t batch, int32_t* unit_ptr,
                                int32_t* counters, int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(query_start && unit_ptr && counters && status);
  HPC_CHECK_ARG(batch >= 0);
  if (batch > HPC_MAX_BATCH) return HPC_ERR_UNSUPPORTED;
  hpc::prefill_plan_kernel<<<1, hpc::kPfPlanThreads, 0, stream>>>(query_start, batch, unit_ptr,
                                                                  counters, status);
  return HPC_LAUNCH_STATUS();
}

namespace hpc {
namespace {

// hpc_prefill_attn, or with staging set hpc_prefill_attn_staged: the checks,
// the maps and the launches.
int prefill_run(const void* q, int32_t num_tokens, const int32_t* query_start, const void* kv_cache,
                int32_t kv_dtype, const float* kv_scale, int32_t num_blocks,
                const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                int32_t batch, const int32_t* unit_ptr, int32_t* counters, void* out,
                int32_t out_dtype, float sm_scale, void* staging, int32_t staging_pages,
                int32_t* page_ptr, int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(q && query_start && kv_cache && block_table && seq_lens && unit_ptr && counters &&
                out && status);
  HPC_CHECK_ARG(batch >= 0 && num_tokens >= 0 && num_blocks > 0 && max_blocks >= 1 && sm_scale > 0.f);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(kv_cache) & 15) == 0);
  if (out_dtype != HPC_OUT_BF16 && out_dtype != HPC_OUT_FP16 && out_dtype != HPC_OUT_FP32)
    return HPC_ERR_UNSUPPORTED;
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(q) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0);
  if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
  const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
  HPC_CHECK_ARG(!fp8 || kv_scale != nullptr);
  if (batch > HPC_MAX_BATCH || num_blocks > HPC_MAX_NUM_BLOCKS) return HPC_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * kPage >= (int64_t{1} << 31)) return HPC_ERR_UNSUPPORTED;
  const bool staged = fp8 && staging != nullptr;
  if (staged) {
    HPC_CHECK_ARG(page_ptr != nullptr && staging_pages >= 1 &&
                  (reinterpret_cast<uintptr_t>(staging) & 15) == 0);
    if (staging_pages > HPC_MAX_NUM_BLOCKS) return HPC_ERR_UNSUPPORTED;
  }
  if (batch == 0 || num_tokens == 0) return HPC_OK;
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return HPC_ERR_CUDA;
  // the pages the kernel streams: the cache, or its staged BF16 copy
  const void* pages = staged ? staging : kv_cache;
  const bool pages_fp8 = fp8 && !staged;
  const int32_t map_blocks = staged ? staging_pages : num_blocks;
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD),
                              static_cast<cuuint64_t>(map_blocks) * 2 * kHkv * kPage};
  // rows of 128 BF16 (two 64-element boxes per page) or 128 E4M3 codes (one box)
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * (pages_fp8 ? 1 : 2)};
  const cuuint32_t box[2] = {pages_fp8 ? 128u : 64u, static_cast<cuuint32_t>(kPage)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult cr = encode(&map, pages_fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                             2, const_cast<void*>(pages),
                             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return HPC_ERR_INVALID_ARG;
  // q as [tokens][64 heads][128 d]: boxes of 16 tokens x 8 heads x 64 of d
  CUtensorMap q_map;
  const cuuint64_t qdims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(kHq),
                               static_cast<cuuint64_t>(num_tokens)};
  const cuuint64_t qstrides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                  static_cast<cuuint64_t>(kHq) * kD * 2};
  const cuuint32_t qbox[3] = {64, static_cast<cuuint32_t>(kGroup),
                              static_cast<cuuint32_t>(tc::kLaneTokens)};
  const cuuint32_t qestr[3] = {1, 1, 1};
  const CUresult qr = encode(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qdims,
                             qstrides, qbox, qestr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (qr != CUDA_SUCCESS) return HPC_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HPC_ERR_CUDA;
  if (staged) {
    stage_plan_kernel<<<1, kPfPlanThreads, 0, stream>>>(seq_lens, batch, max_blocks, page_ptr, status);
    stage_convert_kernel<<<8 * sms, kStageThreads, 0, stream>>>(
        static_cast<const uint8_t*>(kv_cache), num_blocks, block_table, max_blocks, batch, page_ptr,
        staging_pages, static_cast<uint16_t*>(staging));
    if (cudaPeekAtLastError() != cudaSuccess) return HPC_ERR_CUDA;
  }
  if (pages_fp8) {
    if (prefill_tc_smem_optin<true>() != cudaSuccess) return HPC_ERR_CUDA;
    prefill_tc_kernel<true><<<sms, tc::Cfg<true>::kThreads, tc::kSmemBytes, stream>>>(
        map, q_map, num_tokens, static_cast<const uint8_t*>(kv_cache), kv_scale, query_start,
        seq_lens, batch, block_table, max_blocks, num_blocks, unit_ptr, counters, out, out_dtype,
        sm_scale, status, nullptr, 0);
  } else {
    // BF16 pages: the cache itself (no scales, whatever kv_scale points at),
    // or the staged copy of an E4M3 cache (its scales; the real block table
    // still says which tiles are bad)
    if (prefill_tc_smem_optin<false>() != cudaSuccess) return HPC_ERR_CUDA;
    prefill_tc_kernel<false><<<sms, tc::Cfg<false>::kThreads, tc::kSmemBytes, stream>>>(
        map, q_map, num_tokens, static_cast<const uint8_t*>(pages), staged ? kv_scale : nullptr,
        query_start, seq_lens, batch, block_table, max_blocks, num_blocks, unit_ptr, counters, out,
        out_dtype, sm_scale, status, staged ? page_ptr : nullptr, staged ? staging_pages : 0);
  }
  return HPC_LAUNCH_STATUS();
}

}  // namespace
}  // namespace hpc

extern "C" int hpc_prefill_attn(const void* q, int32_t num_tokens, const int32_t* query_start,
                                const void* kv_cache,
                                int32_t kv_dtype, const float* kv_scale, int32_t num_blocks,
                                const int32_t* block_table, int32_t max_blocks,
                                const int32_t* seq_lens, int32_t batch, const int32_t* unit_ptr,
                                int32_t* counters, void* out, int32_t out_dtype, float sm_scale,
                                int32_t* status, cudaStream_t stream) {
  return hpc::prefill_run(q, num_tokens, query_start, kv_cache, kv_dtype, kv_scale, num_blocks,
                          block_table, max_blocks, seq_lens, batch, unit_ptr, counters, out,
                          out_dtype, sm_scale, nullptr, 0, nullptr, status, stream);
}

extern "C" int hpc_prefill_attn_staged(const void* q, int32_t num_tokens,
                                       const int32_t* query_start, const void* kv_cache,
                                       int32_t kv_dtype, const float* kv_scale, int32_t num_blocks,
                                       const int32_t* block_table, int32_t max_blocks,
                                       const int32_t* seq_lens, int32_t batch,
                                       const int32_t* unit_ptr, int32_t* counters, void* out,
                                       int32_t out_dtype, float sm_scale, void* staging,
                                       int32_t staging_pages, int32_t* page_ptr, int32_t* status,
                                       cudaStream_t stream) {
  if (kv_dtype == HPC_KV_FP8_E4M3) HPC_CHECK_ARG(staging != nullptr);
  return hpc::prefill_run(q, num_tokens, query_start, kv_cache, kv_dtype, kv_scale, num_blocks,
                          block_table, max_blocks, seq_lens, batch, unit_ptr, counters, out,
                          out_dtype, sm_scale, staging, staging_pages, page_ptr, status, stream);
}
