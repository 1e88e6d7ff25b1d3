// Log-sum-exp merge of the split-KV partials into the BF16 output.
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper", section "Why does dynamic scheduling matter for attention?": the
// schedules there are split-KV schedules, so a sequence whose tiles were dealt
// to several compute units has several partial results to combine.  The
// combination is the exact one: with lse_k = log sum exp(s) over split k,
// out = sum_k exp(lse_k - M) O_k / sum_k exp(lse_k - M), M = max_k lse_k.
//
// One CTA per (sequence, kv_head) segment and new token, 256 threads: warp r
// handles query head 8h + r and each lane 4 consecutive elements, so every
// partial row is one coalesced 512-byte read.  Items are combined in item
// order (that is, tile order), which makes the output bit-reproducible.  A
// segment whose every partial is empty (lse = -inf) merges to zeros.  With
// q_len new tokens per sequence the partial of item i for token j is row
// (i*q_len + j)*8 + r, and the output row is (b*q_len + j)*64 + 8h + r.
#include "common.cuh"
#include "internal.h"

namespace hpc {
namespace {

__global__ void __launch_bounds__(256, 4) merge_kernel(const float* __restrict__ partial_o,
                                                    const float* __restrict__ partial_lse,
                                                    const int32_t* __restrict__ seg_ptr,
                                                    int32_t capacity, int32_t q_len,
                                                    void* __restrict__ out, int32_t out_dtype,
                                                    bool skip_single) {
  const int s = blockIdx.x;            // segment = seq * 8 + kv_head
  const int j = blockIdx.y;            // new token
  const int r = threadIdx.x >> 5;      // query head within the group
  const int d = (threadIdx.x & 31) * 4;
  // partial row of item i, output row of this CTA
  auto prow = [&](int i) { return (static_cast<int64_t>(i) * q_len + j) * kGroup + r; };
  const int64_t orow = (static_cast<int64_t>(s / kHkv) * q_len + j) * kHq + (s % kHkv) * kGroup + r;
  int i0 = seg_ptr[s], i1 = seg_ptr[s + 1];
  if (i0 < 0 || i1 < i0 || i1 > capacity) i1 = i0;   // a corrupt plan merges to zeros
  if (skip_single && i1 - i0 == 1) return;            // written by the attention kernel

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i1 - i0 == 1) {
    acc = *reinterpret_cast<const float4*>(partial_o + prow(i0) * kD + d);
  } else if (i1 > i0) {
    // The segment's log-sum-exps of this warp's head are staged in shared
    // memory by one parallel load per chunk of kChunk items, so the maximum
    // comes from shared memory and the weighted sum is one pass of
    // independent partial loads (a long sequence's segment holds tens of
    // items).  Chunks after the first rescale what came before (online).
    constexpr int kChunk = 256;
    __shared__ float lse_s[kGroup][kChunk];
    const int lane = threadIdx.x & 31;
    float M = -INFINITY, wsum = 0.f;
    for (int c0 = i0; c0 < i1; c0 += kChunk) {
      const int cn = min(kChunk, i1 - c0);
      __syncwarp();   // the previous chunk's values are read
      for (int k = lane; k < cn; k += 32) lse_s[r][k] = partial_lse[prow(c0 + k)];
      __syncwarp();
      float Mc = -INFINITY;
      for (int k = 0; k < cn; ++k) Mc = fmaxf(Mc, lse_s[r][k]);
      const float Mn = fmaxf(M, Mc);
      if (Mn == -INFINITY) continue;   // nothing but empty partials so far
      const float sc = M == -INFINITY ? 0.f : expf(M - Mn);
      acc.x *= sc;
      acc.y *= sc;
      acc.z *= sc;
      acc.w *= sc;
      wsum *= sc;
#pragma unroll 8
      for (int k = 0; k < cn; ++k) {
        const float w = expf(lse_s[r][k] - Mn);
        const float4 o = *reinterpret_cast<const float4*>(partial_o + prow(c0 + k) * kD + d);
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
        wsum += w;
      }
      M = Mn;
    }
    if (wsum > 0.f) {
      const float inv = 1.0f / wsum;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
  }
  if (out_dtype == HPC_OUT_FP32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + orow * kD + d) = acc;
  } else {
    uint2 packed;
    packed.x = out_dtype == HPC_OUT_FP16 ? pack_f16(acc.x, acc.y) : pack_bf16(acc.x, acc.y);
    packed.y = out_dtype == HPC_OUT_FP16 ? pack_f16(acc.z, acc.w) : pack_bf16(acc.z, acc.w);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + orow * kD + d) = packed;
  }
}

}  // namespace
}  // namespace hpc

int hpc::launch_merge(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
                      int32_t batch, const hpc_attn_options* opts, void* out, bool skip_single,
                      cudaStream_t stream) {
  HPC_CHECK_ARG(partial_o && partial_lse && plan && plan->seg_ptr && out);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(partial_o) & 15) == 0);   // read 16 bytes at a time
  hpc_attn_options o;
  o.q_len = 1;
  o.q_dtype = HPC_Q_BF16;
  o.q_scale = 1.0f;
  o.out_dtype = HPC_OUT_BF16;
  if (opts != nullptr) o = *opts;
  HPC_CHECK_ARG(batch >= 0 && o.q_len >= 1 && o.q_len <= HPC_MAX_Q_LEN);
  if (o.out_dtype != HPC_OUT_BF16 && o.out_dtype != HPC_OUT_FP16 && o.out_dtype != HPC_OUT_FP32)
    return HPC_ERR_UNSUPPORTED;
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(out) & (o.out_dtype == HPC_OUT_FP32 ? 15 : 7)) == 0);
  if (batch == 0) return HPC_OK;
  if (static_cast<int64_t>(batch) * hpc::kHkv > 0x7fffffff) return HPC_ERR_UNSUPPORTED;
  hpc::merge_kernel<<<dim3(batch * hpc::kHkv, o.q_len), 256, 0, stream>>>(
      partial_o, partial_lse, plan->seg_ptr, plan->capacity, o.q_len, out, o.out_dtype, skip_single);
  return HPC_LAUNCH_STATUS();
}

extern "C" int hpc_merge_ex(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
                            int32_t batch, const hpc_attn_options* opts, void* out,
                            cudaStream_t stream) {
  return hpc::launch_merge(partial_o, partial_lse, plan, batch, opts, out, false, stream);
}

extern "C" int hpc_merge_mt(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
                            int32_t batch, int32_t q_len, void* out, cudaStream_t stream) {
  hpc_attn_options o;
  o.q_len = q_len;
  o.q_dtype = HPC_Q_BF16;
  o.q_scale = 1.0f;
  o.out_dtype = HPC_OUT_BF16;
  return hpc_merge_ex(partial_o, partial_lse, plan, batch, &o, out, stream);
}

extern "C" int hpc_merge(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
                         int32_t batch, void* out, cudaStream_t stream) {
  return hpc_merge_ex(partial_o, partial_lse, plan, batch, nullptr, out, stream);
}
