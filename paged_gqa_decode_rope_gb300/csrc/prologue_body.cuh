// Device code of the fused decode prologue (RoPE -> per-head RMSNorm -> q
// output, BF16 or E4M3 codes of q / q_scale, and K/V write into the paged
// cache), shared by the standalone prologue kernel and the fused prologue +
// planner kernel.
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper", section "Why does dynamic scheduling matter for attention?" (RoPE
// rotation, QK-Norm and the KV write in a single kernel pass); page "[vllm]
// Introducing the HPC-Ops attention backend", "Code analysis" section 2.
//
// One block of 8 warps handles one sequence b and one head block xblk:
// xblk = 0..7 takes query heads 8*xblk .. 8*xblk+7, xblk = 8 the 8 KV heads
// (K with RoPE + norm, V as is).  Lane l holds elements 2l, 2l+1 and 64+2l,
// 64+2l+1 of its head, so each RoPE pair (i, i+64) lives in one lane.
#pragma once

#include "common.cuh"

namespace hpc {
namespace {

// kQ8: q is stored as E4M3 codes of q / q_scale (RNE, saturating) instead of BF16.
template <bool kFp8, bool kQ8>
__device__ __forceinline__ void prologue_heads(
    int b, int xblk, const uint16_t* q, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, const int32_t* __restrict__ positions,
    const float* __restrict__ cos_sin, int32_t max_pos, const uint16_t* __restrict__ q_w,
    const uint16_t* __restrict__ k_w, float eps, uint8_t* __restrict__ kv_cache,
    int32_t num_blocks, const int64_t* __restrict__ slot_mapping,
    const float* __restrict__ kv_scale, void* q_out, float q_scale, int32_t* __restrict__ status) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool is_kv = xblk == kGroup;   // the 9th block of a sequence

  const int32_t pos = positions[b];
  if (pos < 0 || pos >= max_pos) {
    if (threadIdx.x == 0 && xblk == 0) atomicOr(status, HPC_STATUS_BAD_POSITION);
    return;
  }
  const int d0 = 2 * lane;          // this lane's first-half pair index
  const float2 cs = *reinterpret_cast<const float2*>(cos_sin + static_cast<int64_t>(pos) * kD + d0);
  const float2 sn = *reinterpret_cast<const float2*>(cos_sin + static_cast<int64_t>(pos) * kD + kD / 2 + d0);

  const uint16_t* src;
  const uint16_t* w;
  if (!is_kv) {
    src = q + (static_cast<int64_t>(b) * kHq + xblk * kGroup + warp) * kD;
    w = q_w;
  } else {
    src = k + (static_cast<int64_t>(b) * kHkv + warp) * kD;
    w = k_w;
  }
  const uint32_t xa = *reinterpret_cast<const uint32_t*>(src + d0);
  const uint32_t xb = *reinterpret_cast<const uint32_t*>(src + kD / 2 + d0);
  const float a0 = bf16_lo(xa), a1 = bf16_hi(xa);   // x[2l], x[2l+1]
  const float b0 = bf16_lo(xb), b1 = bf16_hi(xb);   // x[64+2l], x[64+2l+1]

  // RoPE: pair (i, i+64) turns by the table angle of row `pos`.
  const float r0 = a0 * cs.x - b0 * sn.x;
  const float r1 = a1 * cs.y - b1 * sn.y;
  const float r2 = b0 * cs.x + a0 * sn.x;
  const float r3 = b1 * cs.y + a1 * sn.y;

  // RMSNorm over the 128 elements of the head.
  float ss = r0 * r0 + r1 * r1 + r2 * r2 + r3 * r3;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float inv = 1.0f / sqrtf(ss * (1.0f / kD) + eps);
  const uint32_t wa = *reinterpret_cast<const uint32_t*>(w + d0);
  const uint32_t wb = *reinterpret_cast<const uint32_t*>(w + kD / 2 + d0);
  const float y0 = r0 * inv * bf16_lo(wa), y1 = r1 * inv * bf16_hi(wa);
  const float y2 = r2 * inv * bf16_lo(wb), y3 = r3 * inv * bf16_hi(wb);

  if (!is_kv) {
    const int64_t row = static_cast<int64_t>(b) * kHq + xblk * kGroup + warp;
    if constexpr (kQ8) {
      uint8_t* dst = static_cast<uint8_t*>(q_out) + row * kD;
      *reinterpret_cast<uint16_t*>(dst + d0) = f32x2_to_e4m3x2(y0 / q_scale, y1 / q_scale);
      *reinterpret_cast<uint16_t*>(dst + kD / 2 + d0) = f32x2_to_e4m3x2(y2 / q_scale, y3 / q_scale);
    } else {
      uint16_t* dst = static_cast<uint16_t*>(q_out) + row * kD;
      *reinterpret_cast<uint32_t*>(dst + d0) = pack_bf16(y0, y1);
      *reinterpret_cast<uint32_t*>(dst + kD / 2 + d0) = pack_bf16(y2, y3);
    }
    return;
  }

  // K and V of KV head `warp` go to the cache slot of this sequence.
  const int64_t slot = slot_mapping[b];
  if (slot < 0) return;                                   // padding entry
  if (slot >= static_cast<int64_t>(num_blocks) * kPage) {
    if (lane == 0) atomicOr(status, HPC_STATUS_BAD_SLOT);
    return;
  }
  const int64_t blk = slot / kPage;
  const int off = static_cast<int>(slot % kPage);
  const int64_t k_row = ((blk * 2 + 0) * kHkv + warp) * kPage + off;   // [blk][0][h][off]
  const int64_t v_row = ((blk * 2 + 1) * kHkv + warp) * kPage + off;   // [blk][1][h][off]
  const uint16_t* vsrc = v + (static_cast<int64_t>(b) * kHkv + warp) * kD;
  const uint32_t va = *reinterpret_cast<const uint32_t*>(vsrc + d0);
  const uint32_t vb = *reinterpret_cast<const uint32_t*>(vsrc + kD / 2 + d0);

  if constexpr (!kFp8) {
    uint16_t* kc = reinterpret_cast<uint16_t*>(kv_cache);
    *reinterpret_cast<uint32_t*>(kc + k_row * kD + d0) = pack_bf16(y0, y1);
    *reinterpret_cast<uint32_t*>(kc + k_row * kD + kD / 2 + d0) = pack_bf16(y2, y3);
    *reinterpret_cast<uint32_t*>(kc + v_row * kD + d0) = va;
    *reinterpret_cast<uint32_t*>(kc + v_row * kD + kD / 2 + d0) = vb;
  } else {
    const float ks = kv_scale[0], vs = kv_scale[1];
    uint8_t* kc = kv_cache;
    *reinterpret_cast<uint16_t*>(kc + k_row * kD + d0) = f32x2_to_e4m3x2(y0 / ks, y1 / ks);
    *reinterpret_cast<uint16_t*>(kc + k_row * kD + kD / 2 + d0) = f32x2_to_e4m3x2(y2 / ks, y3 / ks);
    *reinterpret_cast<uint16_t*>(kc + v_row * kD + d0) =
        f32x2_to_e4m3x2(bf16_lo(va) / vs, bf16_hi(va) / vs);
    *reinterpret_cast<uint16_t*>(kc + v_row * kD + kD / 2 + d0) =
        f32x2_to_e4m3x2(bf16_lo(vb) / vs, bf16_hi(vb) / vs);
  }
}


}  // namespace
}  // namespace hpc
