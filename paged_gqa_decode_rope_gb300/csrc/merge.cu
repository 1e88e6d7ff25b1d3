// Log-sum-exp merge of the split-KV partials into the BF16 output.
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper", section "Why does dynamic scheduling matter for attention?": the
// schedules there are split-KV schedules, so a sequence whose tiles were dealt
// to several compute units has several partial results to combine.  The
// combination is the exact one: with lse_k = log sum exp(s) over split k,
// out = sum_k exp(lse_k - M) O_k / sum_k exp(lse_k - M), M = max_k lse_k.
//
// One CTA per (sequence, kv_head) segment, 256 threads: warp r handles query
// head 8h + r and each lane 4 consecutive elements, so every partial row is
// one coalesced 512-byte read.  Items are combined in item order (that is,
// tile order), which makes the output bit-reproducible.
#include "common.cuh"

namespace hpc {
namespace {

__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ partial_o,
                                                    const float* __restrict__ partial_lse,
                                                    const int32_t* __restrict__ seg_ptr,
                                                    int32_t capacity,
                                                    uint16_t* __restrict__ out) {
  const int s = blockIdx.x;            // segment = seq * 8 + kv_head
  const int r = threadIdx.x >> 5;      // query head within the group
  const int d = (threadIdx.x & 31) * 4;
  int i0 = seg_ptr[s], i1 = seg_ptr[s + 1];
  if (i0 < 0 || i1 < i0 || i1 > capacity) i1 = i0;   // a corrupt plan merges to zeros

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (i1 - i0 == 1) {
    acc = *reinterpret_cast<const float4*>(partial_o + (static_cast<int64_t>(i0) * kGroup + r) * kD + d);
  } else if (i1 > i0) {
    // both loops are unrolled so that several partials are in flight at once
    // (a long sequence's segment holds tens of items)
    float M = -INFINITY;
#pragma unroll 8
    for (int i = i0; i < i1; ++i) M = fmaxf(M, partial_lse[static_cast<int64_t>(i) * kGroup + r]);
    if (M != -INFINITY) {
      float wsum = 0.f;
#pragma unroll 8
      for (int i = i0; i < i1; ++i) {
        const float w = expf(partial_lse[static_cast<int64_t>(i) * kGroup + r] - M);
        const float4 o =
            *reinterpret_cast<const float4*>(partial_o + (static_cast<int64_t>(i) * kGroup + r) * kD + d);
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
        wsum += w;
      }
      const float inv = 1.0f / wsum;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
  }
  uint2 packed;
  packed.x = pack_bf16(acc.x, acc.y);
  packed.y = pack_bf16(acc.z, acc.w);
  // segment s = b*8 + h holds query heads 8h .. 8h+7 of sequence b, i.e. rows
  // s*8 .. s*8+7 of the [batch*64, 128] output
  *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(s) * kGroup + r) * kD + d) = packed;
}

}  // namespace
}  // namespace hpc

extern "C" int hpc_merge(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
                         int32_t batch, void* out, cudaStream_t stream) {
  HPC_CHECK_ARG(partial_o && partial_lse && plan && plan->seg_ptr && out);
  HPC_CHECK_ARG(batch >= 0);
  if (batch == 0) return HPC_OK;
  if (static_cast<int64_t>(batch) * hpc::kHkv > 0x7fffffff) return HPC_ERR_UNSUPPORTED;
  hpc::merge_kernel<<<batch * hpc::kHkv, 256, 0, stream>>>(partial_o, partial_lse, plan->seg_ptr,
                                                          plan->capacity,
                                                          static_cast<uint16_t*>(out));
  return HPC_LAUNCH_STATUS();
}
