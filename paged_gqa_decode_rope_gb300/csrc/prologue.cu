// Fused decode prologue: RoPE (NeoX half rotation) -> per-head RMSNorm ->
// BF16 q output and K/V write into the paged cache, in one pass.
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper", section "Why does dynamic scheduling matter for attention?" (the
// prologue fuses RoPE rotation, QK-Norm and the KV write into a single kernel
// pass to remove HBM round trips between them); page "[vllm] Introducing the
// HPC-Ops attention backend", "Code analysis" section 2 and "General lessons"
// item 1 (the same fusion, as a custom op writing a caller-provided output).
//
// Layout of the work: grid (9, batch), 8 warps per CTA, one warp per head.
// CTAs x = 0..7 take query heads 8x..8x+7; CTA x = 8 takes the 8 KV heads (K
// with RoPE + norm, V as is).  Lane l holds elements 2l, 2l+1 and 64+2l,
// 64+2l+1 of its head, so each RoPE pair (i, i+64) lives in one lane and the
// row loads are two coalesced 128-byte segments.  A head is ~0.5 KB of
// traffic: the kernel is latency-bound, not bandwidth-bound.
#include "prologue_body.cuh"

namespace hpc {
namespace {

__global__ void rope_table_kernel(double theta, int32_t max_pos, float* __restrict__ cos_sin) {
  const int64_t n = static_cast<int64_t>(max_pos) * (kD / 2);
  const double log_theta = log(theta);
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t pos = e / (kD / 2);
    const int i = static_cast<int>(e % (kD / 2));
    const double inv_freq = exp(-(2.0 * i / kD) * log_theta);
    double s, c;
    sincos(static_cast<double>(pos) * inv_freq, &s, &c);
    cos_sin[pos * kD + i] = static_cast<float>(c);
    cos_sin[pos * kD + kD / 2 + i] = static_cast<float>(s);
  }
}

template <bool kFp8, bool kQ8>
__global__ void __launch_bounds__(256) prologue_kernel(
    const uint16_t* q, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
    const int32_t* __restrict__ positions, const float* __restrict__ cos_sin, int32_t max_pos,
    const uint16_t* __restrict__ q_w, const uint16_t* __restrict__ k_w, float eps,
    uint8_t* __restrict__ kv_cache, int32_t num_blocks, const int64_t* __restrict__ slot_mapping,
    const float* __restrict__ kv_scale, void* q_out, float q_scale,
    int32_t* __restrict__ status) {
  prologue_heads<kFp8, kQ8>(blockIdx.x, blockIdx.y, q, k, v, positions, cos_sin, max_pos, q_w, k_w, eps,
                       kv_cache, num_blocks, slot_mapping, kv_scale, q_out, q_scale, status);
}

}  // namespace
}  // namespace hpc

extern "C" int hpc_rope_cos_sin_cache(double theta, int32_t max_pos, float* cos_sin,
                                      cudaStream_t stream) {
  HPC_CHECK_ARG(cos_sin != nullptr && max_pos > 0 && theta > 0.0);
  const int64_t n = static_cast<int64_t>(max_pos) * (hpc::kD / 2);
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  hpc::rope_table_kernel<<<static_cast<unsigned>(blocks < 65535 * 16 ? blocks : 65535 * 16),
                           threads, 0, stream>>>(theta, max_pos, cos_sin);
  return HPC_LAUNCH_STATUS();
}

extern "C" int hpc_rope_norm_kvwrite_ex(const void* q, const void* k, const void* v,
                                        const int32_t* positions, const float* cos_sin,
                                        int32_t max_pos, const void* q_norm_w,
                                        const void* k_norm_w, float eps, void* kv_cache,
                                        int32_t kv_dtype, int32_t num_blocks,
                                        const int64_t* slot_mapping, const float* kv_scale,
                                        int32_t q_dtype, float q_scale, void* q_out,
                                        int32_t batch, int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(q && k && v && positions && cos_sin && q_norm_w && k_norm_w && kv_cache &&
                slot_mapping && q_out && status);
  HPC_CHECK_ARG(batch >= 0 && max_pos > 0 && num_blocks > 0 && eps >= 0.0f);
  if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
  if (kv_dtype == HPC_KV_FP8_E4M3) HPC_CHECK_ARG(kv_scale != nullptr);
  if (q_dtype != HPC_Q_BF16 && q_dtype != HPC_Q_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
  if (q_dtype == HPC_Q_FP8_E4M3) HPC_CHECK_ARG(q_scale > 0.0f && q_scale < 3.0e38f);
  if (batch == 0) return HPC_OK;
  const dim3 grid(batch, hpc::kGroup + 1);   // tokens on x: any token count of a prefill
  auto* qp = static_cast<const uint16_t*>(q);
  auto* kp = static_cast<const uint16_t*>(k);
  auto* vp = static_cast<const uint16_t*>(v);
  auto* qw = static_cast<const uint16_t*>(q_norm_w);
  auto* kw = static_cast<const uint16_t*>(k_norm_w);
  auto* cache = static_cast<uint8_t*>(kv_cache);
  auto launch = [&](auto kernel) {
    kernel<<<grid, 256, 0, stream>>>(qp, kp, vp, positions, cos_sin, max_pos, qw, kw, eps, cache,
                                     num_blocks, slot_mapping, kv_scale, q_out, q_scale, status);
  };
  const bool q8 = q_dtype == HPC_Q_FP8_E4M3;
  if (kv_dtype == HPC_KV_BF16) {
    if (q8) launch(hpc::prologue_kernel<false, true>);
    else launch(hpc::prologue_kernel<false, false>);
  } else {
    if (q8) launch(hpc::prologue_kernel<true, true>);
    else launch(hpc::prologue_kernel<true, false>);
  }
  return HPC_LAUNCH_STATUS();
}

extern "C" int hpc_rope_norm_kvwrite(const void* q, const void* k, const void* v,
                                     const int32_t* positions, const float* cos_sin,
                                     int32_t max_pos, const void* q_norm_w, const void* k_norm_w,
                                     float eps, void* kv_cache, int32_t kv_dtype,
                                     int32_t num_blocks, const int64_t* slot_mapping,
                                     const float* kv_scale, void* q_out, int32_t batch,
                                     int32_t* status, cudaStream_t stream) {
  return hpc_rope_norm_kvwrite_ex(q, k, v, positions, cos_sin, max_pos, q_norm_w, k_norm_w, eps,
                                  kv_cache, kv_dtype, num_blocks, slot_mapping, kv_scale,
                                  HPC_Q_BF16, 1.0f, q_out, batch, status, stream);
}
