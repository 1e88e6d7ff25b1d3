// Split-KV paged GQA decode attention (q_len = 1), sm_103a.
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper": intro of "Two new HPC backends in the vLLM ecosystem" (64 query
// heads, 8 KV heads, head_dim 128) and "Why does dynamic scheduling matter
// for attention?" (split-KV over 64-token tiles dealt to compute units in
// proportion to length; BF16 and FP8).  Page "[vllm] Introducing the HPC-Ops
// attention backend", introduction (FP8 E4M3 models).
//
// Design (GB300-first; the pages give no kernel structure):
//  * Persistent grid, one CTA per SM.  CTA c runs the work items
//    cta_ptr[c] .. cta_ptr[c+1]-1 of the plan.  The path is bound by HBM: each
//    64-token K page and V page of a KV head is read exactly once and serves
//    all 8 query heads of its group.
//  * One producer warp streams pages with TMA (cp.async.bulk.tensor, 128-byte
//    swizzle, L2 evict-first) into a ring of stages guarded by mbarriers; a
//    stage is one tile = the K page + the V page of one (block, kv_head).
//    Block ids are fetched 32 at a time by the whole warp, so the issue loop
//    never waits on a global load per tile.
//  * Two groups of four consumer warps take alternate tiles, so two tiles are
//    in flight through the math at once; inside a group the four warps split
//    the tile's 64 tokens, 16 each.  Every warp keeps its own online-softmax
//    state (running max m, sum l, output O) for the current item; at the end
//    of an item the eight states are merged in shared memory, in a fixed warp
//    order, and written as one partial (O, lse).
//  * Tensor cores at q_len = 1 without padding: S^T[16 tok x 8 heads] =
//    K[16 x 128] . Q^T[128 x 8] (m16n8k16, tokens on M, heads on N), then
//    O^T[128 x 8] += V^T[128 x 16 tok] . P^T[16 x 8] (d on M, heads on N).
//    The softmax runs on the S^T accumulator fragment; movmatrix transposes
//    P^T into the B-operand layout, so P never touches shared memory.
//  * FP8 E4M3 pages are converted to f16 in registers after ldmatrix
//    (exact), q is taken to f16 once per item; the k scale folds into the
//    softmax scale and the v scale into the output.  For FP8 the dot products
//    run over a fixed permutation of d (and the V rows over a permutation of
//    d inside each 16-row tile) that makes each ldmatrix word feed the MMA
//    directly; q uses the same permutation and the epilogue undoes it.
//  * Tokens past the sequence length get p = 0 and their V entries are
//    zeroed in registers (the cache may hold NaN there: 0 * NaN is NaN).
//  * Every wait is bounded (kWaitLimitNs): a stuck pipeline records
//    HPC_STATUS_WAIT_TIMEOUT and winds down, waiting for its own copies.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace hpc {
namespace {

template <bool kFp8>
struct AttnTraits {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kPageBytes = kPage * kD * kElem;      // one K or V page of one KV head
  static constexpr int kBoxBytes = 64 * 128;                  // one 64-row x 128-byte TMA box
  static constexpr int kStageBytes = 2 * kPageBytes;          // K page + V page
  static constexpr int kStages = kFp8 ? 10 : 6;
  static constexpr int kWarpsPerGroup = 4;                    // 16 tokens of a tile each
  static constexpr int kGroups = 2;                           // groups take alternate tiles
  static constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
  static constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + the producer warp
  static constexpr int kOStride = kD + 4;                     // padded row of the merge buffer
  static constexpr int kOffO = kStages * kStageBytes;                 // [warps][8][kOStride]
  static constexpr int kOffM = kOffO + kConsumerWarps * kGroup * kOStride * 4;
  static constexpr int kOffL = kOffM + kConsumerWarps * kGroup * 4;
  static constexpr int kOffBar = kOffL + kConsumerWarps * kGroup * 4;
  static constexpr int kOffOk = kOffBar + 2 * kStages * 8;
  static constexpr int kOffAbort = kOffOk + kStages * 4;
  static constexpr int kSmemUsed = kOffAbort + 16;
  static constexpr int kSmemBytes = kSmemUsed + 1024;         // slack for 1024-byte alignment
  static_assert(kOffBar % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory");
};

struct Item {
  int seq, h, t0, t1, len;
  bool ok;
};

__device__ __forceinline__ Item load_item(const hpc_work_item* items, int i,
                                          const int32_t* seq_lens, int batch, int max_blocks) {
  const int4 w = __ldg(reinterpret_cast<const int4*>(items) + i);
  Item it{w.x, w.y, w.z, w.w, 0, false};
  if (it.seq >= 0 && it.seq < batch && it.h >= 0 && it.h < kHkv) {
    const int L = __ldg(seq_lens + it.seq);
    if (L >= 0 && L <= max_blocks * kPage) {
      const int n = (L + kPage - 1) / kPage;
      if (it.t0 >= 0 && it.t0 < it.t1 && it.t1 <= n) {
        it.ok = true;
        it.len = L;
      }
    }
  }
  return it;
}

template <bool kFp8>
__global__ void __launch_bounds__(AttnTraits<kFp8>::kThreads, 1) decode_attn_kernel(
    const __grid_constant__ CUtensorMap kv_map, const uint16_t* __restrict__ q,
    const float* __restrict__ kv_scale, const int32_t* __restrict__ block_table, int32_t max_blocks,
    int32_t num_blocks, const int32_t* __restrict__ seq_lens, int32_t batch,
    const hpc_work_item* __restrict__ items, const int32_t* __restrict__ cta_ptr, int32_t capacity,
    float* __restrict__ partial_o, float* __restrict__ partial_lse, float sm_scale,
    int32_t* __restrict__ status) {
  using T = AttnTraits<kFp8>;
  constexpr int S = T::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* sm_o = reinterpret_cast<float*>(smem + T::kOffO);
  float* sm_m = reinterpret_cast<float*>(smem + T::kOffM);
  float* sm_l = reinterpret_cast<float*>(smem + T::kOffL);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::kOffBar);
  uint64_t* empty = full + S;
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + T::kOffOk);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int it_begin = cta_ptr[blockIdx.x];
  const int it_end = cta_ptr[blockIdx.x + 1];
  if (it_begin < 0 || it_end < it_begin || it_end > capacity) {
    if (threadIdx.x == 0) atomicOr(status, HPC_STATUS_BAD_PLAN);
    return;
  }
  if (it_begin == it_end) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), T::kWarpsPerGroup);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == T::kConsumerWarps) {
    if (lane == 0) tma_prefetch_desc(&kv_map);
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t stage0 = smem_u32(smem);
    uint32_t g = 0;          // tiles issued so far by this CTA
    bool alive = true;
    for (int i = it_begin; i < it_end && alive; ++i) {
      const Item it = load_item(items, i, seq_lens, batch, max_blocks);
      if (!it.ok) {
        if (lane == 0) atomicOr(status, HPC_STATUS_BAD_PLAN);
        continue;
      }
      const int32_t* bt_row = block_table + static_cast<int64_t>(it.seq) * max_blocks;
      for (int tb = it.t0; tb < it.t1 && alive; tb += 32) {
        const int nt = min(32, it.t1 - tb);
        const int my_bid = lane < nt ? __ldg(bt_row + tb + lane) : 0;
        for (int j = 0; j < nt; ++j) {
          const int bid = __shfl_sync(0xffffffffu, my_bid, j);
          int ok = 1;
          if (lane == 0) {
            const int s = static_cast<int>(g % S);
            const uint32_t use = g / S;
            if (*abort_flag) {
              ok = 0;
            } else if (use > 0 && !mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, status)) {
              *abort_flag = 1;
              ok = 0;
            }
            if (ok) {
              const uint32_t fb = smem_u32(&full[s]);
              if (bid >= 0 && bid < num_blocks) {
                stage_ok[s] = 1;
                mbar_arrive_expect_tx(fb, T::kStageBytes);
                const uint32_t dst = stage0 + s * T::kStageBytes;
                const int yk = ((bid * 2 + 0) * kHkv + it.h) * kPage;   // row of [bid][0][h][0]
                const int yv = yk + kHkv * kPage;                        // row of [bid][1][h][0]
                if constexpr (kFp8) {
                  tma_load_2d(dst, &kv_map, 0, yk, fb, policy);
                  tma_load_2d(dst + T::kPageBytes, &kv_map, 0, yv, fb, policy);
                } else {
                  tma_load_2d(dst, &kv_map, 0, yk, fb, policy);
                  tma_load_2d(dst + T::kBoxBytes, &kv_map, 64, yk, fb, policy);
                  tma_load_2d(dst + T::kPageBytes, &kv_map, 0, yv, fb, policy);
                  tma_load_2d(dst + T::kPageBytes + T::kBoxBytes, &kv_map, 64, yv, fb, policy);
                }
              } else {
                atomicOr(status, HPC_STATUS_BAD_BLOCK);
                stage_ok[s] = 0;
                mbar_arrive(fb);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            alive = false;
            break;
          }
          ++g;
        }
      }
    }
    // After a fault, copies may still be landing in stages nobody will wait
    // on: wait for the last one issued into every stage before exiting.
    if (lane == 0 && *abort_flag) {
      for (uint32_t s = 0; s < static_cast<uint32_t>(S) && s < g; ++s) {
        const uint32_t last = s + S * ((g - 1 - s) / S);
        mbar_wait(smem_u32(&full[s]), (last / S) & 1, status);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const uint32_t grp = warp / T::kWarpsPerGroup;   // this warp's tiles: g % kGroups == grp
  const int wq = warp % T::kWarpsPerGroup;         // token quarter of each tile
  const int r = lane >> 2, c = lane & 3;
  const float k_scale = kFp8 ? kv_scale[0] : 1.f;
  const float v_scale = kFp8 ? kv_scale[1] : 1.f;
  const float scale_log2 = sm_scale * k_scale * 1.4426950408889634f;
  const uint32_t stage0 = smem_u32(smem);
  const int sw = lane & 7;                                        // swizzle of this lane's row
  const int row = 16 * wq + (lane & 7) + ((lane >> 3) & 1) * 8;   // ldmatrix row (token)
  const int hi = lane >> 4;                                        // second 16-byte chunk
  const int vtok_bf16 = 16 * wq + (lane & 7) + hi * 8;             // V^T .trans row (token)
  const int vsel_bf16 = (lane >> 3) & 1;                           // V^T d half
  uint32_t g = 0;
  bool dead = false;

  for (int i = it_begin; i < it_end; ++i) {
    const Item it = load_item(items, i, seq_lens, batch, max_blocks);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2c, 2c+1
    float o[8][4];
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;

    if (it.ok) {
      // B operand Q^T for the 8 query heads of this KV head (head = r)
      uint32_t bq[8][2];
      const uint16_t* qrow = q + (static_cast<int64_t>(it.seq) * kHq + it.h * kGroup + r) * kD;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if constexpr (kFp8) {
          const uint2 x = __ldg(reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c));
          bq[ks][0] = pack_f16(bf16_lo(x.x), bf16_hi(x.x));
          bq[ks][1] = pack_f16(bf16_lo(x.y), bf16_hi(x.y));
        } else {
          bq[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c));
          bq[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * c));
        }
      }

      for (int t = it.t0; t < it.t1; ++t, ++g) {
        if (dead || g % T::kGroups != grp) continue;
        const int s = static_cast<int>(g % S);
        const uint32_t use = g / S;
        bool ok = !*abort_flag && mbar_wait(smem_u32(&full[s]), use & 1, status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) *abort_flag = 1;
          dead = true;
          continue;
        }
        const int nvalid = it.len - t * kPage - 16 * wq;   // valid tokens of my 16
        if (stage_ok[s] && nvalid > 0) {
          const uint32_t kb = stage0 + s * T::kStageBytes;
          const uint32_t vb = kb + T::kPageBytes;

          // S^T = K Q^T  (rows: my 16 tokens, cols: 8 heads); two chains
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (kFp8) {
#pragma unroll
            for (int kp = 0; kp < 4; ++kp) {
              uint32_t r0, r1, r2, r3;
              ldsm_x4(kb + row * 128 + ((((2 * kp + hi) & 7) ^ sw) << 4), r0, r1, r2, r3);
              mma_f16(sa, e4m3x2_to_f16x2(r0 & 0xffff), e4m3x2_to_f16x2(r1 & 0xffff),
                      e4m3x2_to_f16x2(r0 >> 16), e4m3x2_to_f16x2(r1 >> 16), bq[2 * kp][0],
                      bq[2 * kp][1]);
              mma_f16(sb, e4m3x2_to_f16x2(r2 & 0xffff), e4m3x2_to_f16x2(r3 & 0xffff),
                      e4m3x2_to_f16x2(r2 >> 16), e4m3x2_to_f16x2(r3 >> 16), bq[2 * kp + 1][0],
                      bq[2 * kp + 1][1]);
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(kb + (ks >> 2) * T::kBoxBytes + row * 128 + ((((2 * ks + hi) & 7) ^ sw) << 4),
                      a0, a1, a2, a3);
              if (ks & 1) mma_bf16(sb, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
              else        mma_bf16(sa, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
            }
          }
          // fragment: x0 = S[tok r][head 2c], x1 = [r][2c+1], x2 = [r+8][2c], x3 = [r+8][2c+1]
          float x0 = (sa[0] + sb[0]) * scale_log2, x1 = (sa[1] + sb[1]) * scale_log2;
          float x2 = (sa[2] + sb[2]) * scale_log2, x3 = (sa[3] + sb[3]) * scale_log2;
          uint32_t mask01 = 0xffffffffu, mask23 = 0xffffffffu;
          if (nvalid < 16) {
            if (r >= nvalid) x0 = x1 = -INFINITY;
            if (r + 8 >= nvalid) x2 = x3 = -INFINITY;
            mask01 = (2 * c < nvalid ? 0x0000ffffu : 0u) | (2 * c + 1 < nvalid ? 0xffff0000u : 0u);
            mask23 = (2 * c + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * c + 9 < nvalid ? 0xffff0000u : 0u);
          }
          float mt0 = fmaxf(x0, x2), mt1 = fmaxf(x1, x3);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, off));
            mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, off));
          }
          const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
          const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
          const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = exp2f(m0 - ms0), al1 = exp2f(m1 - ms1);
          const float p0 = exp2f(x0 - ms0), p1 = exp2f(x1 - ms1);
          const float p2 = exp2f(x2 - ms0), p3 = exp2f(x3 - ms1);
          l0 = l0 * al0 + (p0 + p2);
          l1 = l1 * al1 + (p1 + p3);
          m0 = mn0;
          m1 = mn1;
#pragma unroll
          for (int mi = 0; mi < 8; ++mi) {
            o[mi][0] *= al0;
            o[mi][1] *= al1;
            o[mi][2] *= al0;
            o[mi][3] *= al1;
          }
          // P^T fragment -> B operand (k = token, n = head) by an 8x8 transpose
          uint32_t pb0, pb1;
          if constexpr (kFp8) {
            pb0 = movmatrix_t(pack_f16(p0, p1));
            pb1 = movmatrix_t(pack_f16(p2, p3));
          } else {
            pb0 = movmatrix_t(pack_bf16(p0, p1));
            pb1 = movmatrix_t(pack_bf16(p2, p3));
          }

          // O^T += V^T P^T  (rows: d, cols: 8 heads)
          if constexpr (kFp8) {
#pragma unroll
            for (int mp = 0; mp < 4; ++mp) {
              uint32_t r0, r1, r2, r3;
              ldsm_x4_t(vb + row * 128 + ((((2 * mp + hi) & 7) ^ sw) << 4), r0, r1, r2, r3);
              // r0: tokens 2c, 2c+1 at d 2r, 2r+1 (bytes t0d0, t0d1, t1d0, t1d1)
              const uint32_t x = prmt(r0, 0, 0x3120), y = prmt(r1, 0, 0x3120);
              const uint32_t z = prmt(r2, 0, 0x3120), w = prmt(r3, 0, 0x3120);
              mma_f16(o[2 * mp], e4m3x2_to_f16x2(x & 0xffff) & mask01,
                      e4m3x2_to_f16x2(x >> 16) & mask01, e4m3x2_to_f16x2(y & 0xffff) & mask23,
                      e4m3x2_to_f16x2(y >> 16) & mask23, pb0, pb1);
              mma_f16(o[2 * mp + 1], e4m3x2_to_f16x2(z & 0xffff) & mask01,
                      e4m3x2_to_f16x2(z >> 16) & mask01, e4m3x2_to_f16x2(w & 0xffff) & mask23,
                      e4m3x2_to_f16x2(w >> 16) & mask23, pb0, pb1);
            }
          } else {
#pragma unroll
            for (int mi = 0; mi < 8; ++mi) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4_t(vb + (mi >> 2) * T::kBoxBytes + vtok_bf16 * 128 +
                            ((((2 * mi + vsel_bf16) & 7) ^ sw) << 4),
                        a0, a1, a2, a3);
              mma_bf16(o[mi], a0 & mask01, a1 & mask01, a2 & mask23, a3 & mask23, pb0, pb1);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      }
    }

    // ---- merge the four warps' states and write the item's partial
    l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
    if (lane < 4) {
      sm_m[warp * kGroup + 2 * c] = m0;
      sm_m[warp * kGroup + 2 * c + 1] = m1;
      sm_l[warp * kGroup + 2 * c] = l0;
      sm_l[warp * kGroup + 2 * c + 1] = l1;
    }
    named_bar_sync(1, 32 * T::kConsumerWarps);
    {
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < T::kConsumerWarps; ++w) {
        M0 = fmaxf(M0, sm_m[w * kGroup + 2 * c]);
        M1 = fmaxf(M1, sm_m[w * kGroup + 2 * c + 1]);
      }
      const float Ms0 = M0 == -INFINITY ? 0.f : M0, Ms1 = M1 == -INFINITY ? 0.f : M1;
      float L0 = 0.f, L1 = 0.f;
#pragma unroll
      for (int w = 0; w < T::kConsumerWarps; ++w) {
        L0 += sm_l[w * kGroup + 2 * c] * exp2f(sm_m[w * kGroup + 2 * c] - Ms0);
        L1 += sm_l[w * kGroup + 2 * c + 1] * exp2f(sm_m[w * kGroup + 2 * c + 1] - Ms1);
      }
      const float f0 = L0 > 0.f ? exp2f(m0 - Ms0) / L0 * v_scale : 0.f;
      const float f1 = L1 > 0.f ? exp2f(m1 - Ms1) / L1 * v_scale : 0.f;
      // this warp's share, scaled to the merged normaliser, into its own slice
      // (summed below in a fixed warp order: the result is bit-reproducible)
      float* o_h0 = sm_o + (warp * kGroup + 2 * c) * T::kOStride;
      float* o_h1 = o_h0 + T::kOStride;
#pragma unroll
      for (int mi = 0; mi < 8; ++mi) {
        // rows of the O^T fragment: d_a for o[mi][0..1], d_b for o[mi][2..3]
        const int d_a = kFp8 ? 16 * mi + 2 * r : 16 * mi + r;
        const int d_b = kFp8 ? d_a + 1 : d_a + 8;
        o_h0[d_a] = f0 * o[mi][0];
        o_h1[d_a] = f1 * o[mi][1];
        o_h0[d_b] = f0 * o[mi][2];
        o_h1[d_b] = f1 * o[mi][3];
      }
    }
    named_bar_sync(1, 32 * T::kConsumerWarps);
    {
      const int ct = threadIdx.x;   // 0 .. 127
      float* dst = partial_o + static_cast<int64_t>(i) * kGroup * kD;
#pragma unroll
      for (int e = ct * 4; e < kGroup * kD; e += 32 * T::kConsumerWarps * 4) {
        const int off = (e >> 7) * T::kOStride + (e & 127);
        float4 acc = *reinterpret_cast<const float4*>(sm_o + off);
#pragma unroll
        for (int w = 1; w < T::kConsumerWarps; ++w) {
          const float4 x = *reinterpret_cast<const float4*>(sm_o + w * kGroup * T::kOStride + off);
          acc.x += x.x;
          acc.y += x.y;
          acc.z += x.z;
          acc.w += x.w;
        }
        *reinterpret_cast<float4*>(dst + e) = acc;
      }
      if (ct < kGroup) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < T::kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * kGroup + ct]);
        float L = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < T::kConsumerWarps; ++w)
            L += sm_l[w * kGroup + ct] * exp2f(sm_m[w * kGroup + ct] - M);
        }
        partial_lse[static_cast<int64_t>(i) * kGroup + ct] =
            L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
      }
    }
    named_bar_sync(1, 32 * T::kConsumerWarps);
  }
}

// ------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

template <bool kFp8>
cudaError_t ensure_smem_attr() {
  // once per device: the dynamic shared memory opt-in is a per-device setting
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(decode_attn_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           AttnTraits<kFp8>::kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

template <bool kFp8>
int launch_attn(const void* q, const void* kv_cache, const float* kv_scale, int32_t num_blocks,
                const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                int32_t batch, const hpc_plan* plan, float* partial_o, float* partial_lse,
                float sm_scale, int32_t* status, cudaStream_t stream) {
  using T = AttnTraits<kFp8>;
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return HPC_ERR_CUDA;
  if (ensure_smem_attr<kFp8>() != cudaSuccess) return HPC_ERR_CUDA;
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD),
                              static_cast<cuuint64_t>(num_blocks) * 2 * kHkv * kPage};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * T::kElem};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / T::kElem), static_cast<cuuint32_t>(kPage)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult cr = encode(&map,
                             kFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                             2, const_cast<void*>(kv_cache), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return HPC_ERR_INVALID_ARG;
  decode_attn_kernel<kFp8><<<plan->num_ctas, T::kThreads, T::kSmemBytes, stream>>>(
      map, static_cast<const uint16_t*>(q), kv_scale, block_table, max_blocks, num_blocks, seq_lens,
      batch, plan->items, plan->cta_ptr, plan->capacity, partial_o, partial_lse, sm_scale, status);
  return HPC_LAUNCH_STATUS();
}

}  // namespace
}  // namespace hpc

extern "C" int hpc_decode_attn(const void* q, const void* kv_cache, int32_t kv_dtype,
                               const float* kv_scale, int32_t num_blocks,
                               const int32_t* block_table, int32_t max_blocks,
                               const int32_t* seq_lens, int32_t batch, const hpc_plan* plan,
                               float* partial_o, float* partial_lse, float sm_scale,
                               int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(q && kv_cache && block_table && seq_lens && plan && partial_o && partial_lse &&
                status && plan->items && plan->cta_ptr);
  HPC_CHECK_ARG(num_blocks > 0 && max_blocks >= 1 && batch >= 0 && plan->num_ctas >= 1 &&
                plan->capacity >= 0);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(kv_cache) & 15) == 0);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(plan->items) & 15) == 0);
  if (num_blocks > HPC_MAX_NUM_BLOCKS) return HPC_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * hpc::kPage >= (int64_t{1} << 31)) return HPC_ERR_UNSUPPORTED;
  if (plan->num_ctas > 0x7fffffff - 1) return HPC_ERR_UNSUPPORTED;
  if (kv_dtype == HPC_KV_BF16)
    return hpc::launch_attn<false>(q, kv_cache, kv_scale, num_blocks, block_table, max_blocks,
                                   seq_lens, batch, plan, partial_o, partial_lse, sm_scale, status,
                                   stream);
  if (kv_dtype == HPC_KV_FP8_E4M3) {
    HPC_CHECK_ARG(kv_scale != nullptr);
    return hpc::launch_attn<true>(q, kv_cache, kv_scale, num_blocks, block_table, max_blocks,
                                  seq_lens, batch, plan, partial_o, partial_lse, sm_scale, status,
                                  stream);
  }
  return HPC_ERR_UNSUPPORTED;
}

extern "C" int hpc_decode_num_ctas(int32_t kv_dtype, int32_t* num_ctas) {
  HPC_CHECK_ARG(num_ctas != nullptr);
  if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HPC_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HPC_ERR_CUDA;
  *num_ctas = sms;   // one resident CTA per SM (the stage ring takes ~200 KB)
  return HPC_OK;
}
