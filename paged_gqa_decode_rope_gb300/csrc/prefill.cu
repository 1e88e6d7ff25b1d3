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
// Design (GB300-first; the pages give no kernel structure):
//  * A work unit is (sequence, kv_head, block of 16 new tokens): its 16 x 8
//    query rows share every K/V page of the KV head, so a page read from HBM
//    (or L2, for the other token blocks of the sequence) serves 128 rows.
//    Units are dealt at run time from one atomic counter to a persistent
//    grid; within a sequence the blocks with the most keys come first.
//  * One producer warp streams the unit's visible pages with TMA into a ring
//    of stages (the decode kernel's tensor map: 64-row x 128-byte boxes,
//    128-byte swizzle); eight consumer warps, one per query head of the
//    group, each own the unit's 16 tokens of their head.
//  * S = Q K^T and O += P V on mma.sync m16n8k16 (tokens on M): Q's A
//    fragments stay in registers for the unit, K's B fragments come from
//    ldmatrix and V's from ldmatrix.trans, and the S accumulators become P's
//    A fragments in registers (the accumulator and A layouts coincide).
//  * Keys past a token's position get p = 0; V entries past the sequence
//    length are zeroed in registers (the cache may hold NaN there).
//  * Every wait is bounded (kWaitLimitNs), as in the decode kernel.
#include "attn_kernel.cuh"
#include "plan_body.cuh"
#include "prefill_tc.cuh"

namespace hpc {
namespace {

constexpr int kPfWarps = 8;                       // consumer warps: one per query head of the group
constexpr int kPfThreads = 32 * (kPfWarps + 1);   // + the producer warp
constexpr int kPfStages = 4;
constexpr int kPfRing = 2;                        // units queued ahead
constexpr int kPfBoxBytes = 64 * 128;
constexpr int kPfPageBytes = kPage * kD * 2;      // BF16 page of one KV head
constexpr int kPfStageBytes = 2 * kPfPageBytes;
constexpr int kPfOffBar = kPfStages * kPfStageBytes;
constexpr int kPfNumBars = 2 * kPfStages + 2 * kPfRing;
constexpr int kPfOffRing = kPfOffBar + kPfNumBars * 8;
constexpr int kPfOffOk = kPfOffRing + kPfRing * 4 * 4;     // per stage: 1 = data landed
constexpr int kPfOffAbort = kPfOffOk + kPfStages * 4;
constexpr int kPfSmemBytes = kPfOffAbort + 16 + 1024;   // + slack for 1024-byte alignment
constexpr int kPfTokens = 16;                           // new tokens per unit

// Two consecutive output elements (index even) in the caller's output type.
__device__ __forceinline__ void store_out2(void* out, int64_t idx, float a, float b,
                                           int32_t out_dtype) {
  if (out_dtype == HPC_OUT_FP32) {
    *reinterpret_cast<float2*>(static_cast<float*>(out) + idx) = make_float2(a, b);
  } else {
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(out) + idx) =
        out_dtype == HPC_OUT_FP16 ? pack_f16(a, b) : pack_bf16(a, b);
  }
}

// Units of every sequence (8 kv heads x token blocks) and their prefix;
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
    local += kHkv * ((n + kPfTokens - 1) / kPfTokens);
  }
  int total;
  int run = cta_exclusive_scan<kPfPlanThreads>(local, warp_sums, &total);
  for (int b = b0; b < b1; ++b) {
    unit_ptr[b] = run;
    const int n = query_start[b + 1] - query_start[b];
    if (n > 0) run += kHkv * ((n + kPfTokens - 1) / kPfTokens);
  }
  if (threadIdx.x == 0) {
    unit_ptr[batch] = total;
    counters[0] = 0;   // next unit
    counters[1] = 0;   // CTAs done
  }
}

__global__ void __launch_bounds__(kPfThreads, 1) prefill_attn_kernel(
    const __grid_constant__ CUtensorMap kv_map, const uint16_t* __restrict__ q,
    const int32_t* __restrict__ query_start, const int32_t* __restrict__ seq_lens, int32_t batch,
    const int32_t* __restrict__ block_table, int32_t max_blocks, int32_t num_blocks,
    const int32_t* __restrict__ unit_ptr, int32_t* counters, void* __restrict__ out,
    int32_t out_dtype, float sm_scale, int32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPfOffBar);
  uint64_t* empty = full + kPfStages;
  uint64_t* unit_full = empty + kPfStages;
  uint64_t* unit_empty = unit_full + kPfRing;
  volatile int* ring = reinterpret_cast<volatile int*>(smem + kPfOffRing);
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + kPfOffOk);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kPfOffAbort);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kPfWarps);
    }
    for (int r = 0; r < kPfRing; ++r) {
      mbar_init(smem_u32(&unit_full[r]), 1);
      mbar_init(smem_u32(&unit_empty[r]), kPfWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kPfWarps && lane == 0) tma_prefetch_desc(&kv_map);
  __syncthreads();
  const int total_units = unit_ptr[batch];

  // ------------------------------------------------------------ producer
  if (warp == kPfWarps) {
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t stage0 = smem_u32(smem);
    uint32_t g = 0, n_pushed = 0;
    bool alive = true;
    while (alive) {
      int u = 0;
      if (lane == 0) u = atomicAdd(&counters[0], 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      int b = -1, h = 0, qb = 0, ntiles = 0;
      if (u < total_units) {
        // the sequence of unit u: the last b with unit_ptr[b] <= u (32-ary search)
        int lo = 0, hi = batch;
        while (hi - lo > 1) {
          const int step = (hi - lo + 31) / 32;
          const int idx = lo + lane * step;
          const bool le = idx < hi && unit_ptr[idx] <= u;
          const uint32_t m = __ballot_sync(0xffffffffu, le);
          const int k = 31 - __clz(m);   // lane 0 always qualifies (unit_ptr[lo] <= u)
          lo += k * step;
          hi = min(hi, lo + step);
        }
        b = lo;
        const int j = u - unit_ptr[b];
        const int qs = query_start[b], qlen = query_start[b + 1] - qs, L = seq_lens[b];
        const int nqb = (qlen + kPfTokens - 1) / kPfTokens;
        h = j % kHkv;
        qb = nqb - 1 - j / kHkv;               // the blocks with the most keys first
        if (qlen < 1 || L < qlen || L > max_blocks * kPage || qb < 0) {
          if (lane == 0) atomicOr(status, HPC_STATUS_BAD_SEQ_LEN);
          ntiles = -1;
        } else {
          const int last = min(kPfTokens, qlen - qb * kPfTokens) - 1;   // last row of the block
          const int last_pos = L - qlen + qb * kPfTokens + last;
          ntiles = last_pos / kPage + 1;
        }
      }
      // hand the unit (or the end mark, b = -1) to the consumers
      int ok = 1;
      if (lane == 0) {
        const int r = static_cast<int>(n_pushed % kPfRing);
        const uint32_t use = n_pushed / kPfRing;
        if (*abort_flag) {
          ok = 0;
        } else if (use > 0 && !mbar_wait(smem_u32(&unit_empty[r]), (use - 1) & 1, status)) {
          *abort_flag = 1;
          ok = 0;
        }
        if (ok) {
          volatile int* slot = ring + r * 4;
          slot[0] = b;
          slot[1] = h;
          slot[2] = qb;
          slot[3] = ntiles;
          mbar_arrive(smem_u32(&unit_full[r]));
        }
      }
      ++n_pushed;
      if (!__shfl_sync(0xffffffffu, ok, 0) || b < 0) break;
      for (int tb = 0; tb < ntiles && alive; tb += 32) {
        const int t = tb + lane;
        const int bids = t < ntiles ? block_table[static_cast<int64_t>(b) * max_blocks + t] : 0;
        for (int jj = 0; jj < min(32, ntiles - tb) && alive; ++jj) {
          const int bid = __shfl_sync(0xffffffffu, bids, jj);
          int tok = 1;
          if (lane == 0) {
            const int s = static_cast<int>(g % kPfStages);
            const uint32_t use = g / kPfStages;
            if (*abort_flag) {
              tok = 0;
            } else if (use > 0 && !mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, status)) {
              *abort_flag = 1;
              tok = 0;
            }
            if (tok) {
              const uint32_t fb = smem_u32(&full[s]);
              if (bid >= 0 && bid < num_blocks) {
                stage_ok[s] = 1;
                mbar_arrive_expect_tx(fb, kPfStageBytes);
                const uint32_t dst = stage0 + s * kPfStageBytes;
                const int yk = ((bid * 2 + 0) * kHkv + h) * kPage;
                const int yv = yk + kHkv * kPage;
                tma_load_2d(dst, &kv_map, 0, yk, fb, policy);
                tma_load_2d(dst + kPfBoxBytes, &kv_map, 64, yk, fb, policy);
                tma_load_2d(dst + kPfPageBytes, &kv_map, 0, yv, fb, policy);
                tma_load_2d(dst + kPfPageBytes + kPfBoxBytes, &kv_map, 64, yv, fb, policy);
              } else {
                // a bad block id: the stage arrives without data and the
                // consumers skip the tile
                atomicOr(status, HPC_STATUS_BAD_BLOCK);
                stage_ok[s] = 0;
                mbar_arrive(fb);
              }
            }
          }
          alive = __shfl_sync(0xffffffffu, tok, 0) != 0;
          ++g;
        }
      }
    }
    if (lane == 0) {
      if (atomicAdd(&counters[1], 1) == static_cast<int>(gridDim.x) - 1) {
        counters[0] = 0;   // the last CTA resets the counters: the plan can run again
        counters[1] = 0;
      }
      if (*abort_flag) {   // wait for copies still landing in stages nobody waits on
        for (uint32_t s = 0; s < static_cast<uint32_t>(kPfStages) && s < g; ++s) {
          const uint32_t last = s + kPfStages * ((g - 1 - s) / kPfStages);
          mbar_wait(smem_u32(&full[s]), (last / kPfStages) & 1, status);
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int r8 = lane >> 2, c = lane & 3;   // fragment row (token) and column pair
  const float scale_log2 = sm_scale * 1.4426950408889634f;
  const uint32_t stage0 = smem_u32(smem);
  uint32_t g = 0;
  bool dead = false;
  for (uint32_t n = 0; !dead; ++n) {
    const int rslot = static_cast<int>(n % kPfRing);
    bool ok = !*abort_flag && mbar_wait(smem_u32(&unit_full[rslot]), (n / kPfRing) & 1, status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) *abort_flag = 1;
      break;
    }
    const volatile int* slot = ring + rslot * 4;
    const int b = slot[0], h = slot[1], qb = slot[2], ntiles = slot[3];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&unit_empty[rslot]));
    if (b < 0) break;
    if (ntiles <= 0) continue;

    const int qs = query_start[b], qlen = query_start[b + 1] - qs, L = seq_lens[b];
    const int head = h * kGroup + warp;
    // rows r8 and r8 + 8 of the block: new tokens i0, i1 at positions p0, p1
    const int i0 = qb * kPfTokens + r8, i1 = i0 + 8;
    const bool v0 = i0 < qlen, v1 = i1 < qlen;
    const int p0 = L - qlen + i0, p1 = L - qlen + i1;
    // Q's A fragments for the 8 k-steps of d (zeros for rows past the chunk)
    uint32_t qa[8][4];
    {
      const uint16_t* q0 = q + (static_cast<int64_t>(qs + i0) * kHq + head) * kD;
      const uint16_t* q1 = q + (static_cast<int64_t>(qs + i1) * kHq + head) * kD;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + 16 * ks + 2 * c) : 0u;
        qa[ks][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + 16 * ks + 2 * c) : 0u;
        qa[ks][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + 16 * ks + 8 + 2 * c) : 0u;
        qa[ks][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + 16 * ks + 8 + 2 * c) : 0u;
      }
    }
    float o[16][4];
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows r8, r8 + 8

    for (int t = 0; t < ntiles; ++t, ++g) {
      if (dead) continue;
      const int s = static_cast<int>(g % kPfStages);
      bool tok = !*abort_flag && mbar_wait(smem_u32(&full[s]), (g / kPfStages) & 1, status);
      tok = __all_sync(0xffffffffu, tok);
      if (!tok) {
        if (lane == 0) *abort_flag = 1;
        dead = true;
        continue;
      }
      if (!stage_ok[s]) {   // a tile without data (bad block id): skipped
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        continue;
      }
      const uint32_t kb = stage0 + s * kPfStageBytes;
      const uint32_t vb = kb + kPfPageBytes;
      const int key0 = t * kPage;
      const int mi = lane >> 3, lr = lane & 7;   // ldmatrix: matrix and row of this lane's address

      // S = Q K^T: n-block nb = keys key0 + 8nb .. +7
      float sfr[8][4];
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) sfr[nb][0] = sfr[nb][1] = sfr[nb][2] = sfr[nb][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {   // n-blocks 2np, 2np + 1
          const int key = 8 * (2 * np + (mi >> 1)) + lr;
          const int chunk = 2 * ks + (mi & 1);
          uint32_t b0a, b1a, b0b, b1b;
          ldsm_x4(kb + (chunk >> 3) * kPfBoxBytes + key * 128 + (((chunk & 7) ^ (key & 7)) << 4),
                  b0a, b1a, b0b, b1b);
          mma_bf16(sfr[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0a, b1a);
          mma_bf16(sfr[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0b, b1b);
        }
      }
      // scale, mask (keys past the row's position), row maxima
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
        const int k0 = key0 + 8 * nb + 2 * c;
        sfr[nb][0] = (v0 && k0 <= p0) ? sfr[nb][0] * scale_log2 : -INFINITY;
        sfr[nb][1] = (v0 && k0 + 1 <= p0) ? sfr[nb][1] * scale_log2 : -INFINITY;
        sfr[nb][2] = (v1 && k0 <= p1) ? sfr[nb][2] * scale_log2 : -INFINITY;
        sfr[nb][3] = (v1 && k0 + 1 <= p1) ? sfr[nb][3] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(sfr[nb][0], sfr[nb][1]));
        mx1 = fmaxf(mx1, fmaxf(sfr[nb][2], sfr[nb][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2_ftz(m0 - ms0), al1 = exp2_ftz(m1 - ms1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
        sfr[nb][0] = exp2_ftz(sfr[nb][0] - ms0);   // from here on sfr holds p
        sfr[nb][1] = exp2_ftz(sfr[nb][1] - ms0);
        sfr[nb][2] = exp2_ftz(sfr[nb][2] - ms1);
        sfr[nb][3] = exp2_ftz(sfr[nb][3] - ms1);
        ps0 += sfr[nb][0] + sfr[nb][1];
        ps1 += sfr[nb][2] + sfr[nb][3];
      }
      l0 = l0 * al0 + ps0;   // this lane's share of the row sums
      l1 = l1 * al1 + ps1;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        o[nd][0] *= al0;
        o[nd][1] *= al0;
        o[nd][2] *= al1;
        o[nd][3] *= al1;
      }
      // O += P V; k-step ks2 = keys key0 + 16 ks2 .. +15; V rows past the
      // sequence length are zeroed (0 * NaN would poison the sum)
#pragma unroll
      for (int ks2 = 0; ks2 < 4; ++ks2) {
        const uint32_t pa0 = pack_bf16(sfr[2 * ks2][0], sfr[2 * ks2][1]);
        const uint32_t pa1 = pack_bf16(sfr[2 * ks2][2], sfr[2 * ks2][3]);
        const uint32_t pa2 = pack_bf16(sfr[2 * ks2 + 1][0], sfr[2 * ks2 + 1][1]);
        const uint32_t pa3 = pack_bf16(sfr[2 * ks2 + 1][2], sfr[2 * ks2 + 1][3]);
        const int kk = key0 + 16 * ks2;
        const bool tail = kk + 16 > L;
        const uint32_t mlo = (kk + 2 * c < L ? 0x0000ffffu : 0u) | (kk + 2 * c + 1 < L ? 0xffff0000u : 0u);
        const uint32_t mhi =
            (kk + 8 + 2 * c < L ? 0x0000ffffu : 0u) | (kk + 8 + 2 * c + 1 < L ? 0xffff0000u : 0u);
#pragma unroll
        for (int np = 0; np < 8; ++np) {   // d chunks 2np, 2np + 1
          const int key = 16 * ks2 + (mi & 1) * 8 + lr;
          const int chunk = 2 * np + (mi >> 1);
          uint32_t b0a, b1a, b0b, b1b;
          ldsm_x4_t(vb + (chunk >> 3) * kPfBoxBytes + key * 128 + (((chunk & 7) ^ (key & 7)) << 4),
                    b0a, b1a, b0b, b1b);
          if (tail) {
            b0a &= mlo;
            b1a &= mhi;
            b0b &= mlo;
            b1b &= mhi;
          }
          mma_bf16(o[2 * np], pa0, pa1, pa2, pa3, b0a, b1a);
          mma_bf16(o[2 * np + 1], pa0, pa1, pa2, pa3, b0b, b1b);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    if (dead) break;
    // rows of the block: O / l, written as the caller's type
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const int64_t row0 = (static_cast<int64_t>(qs + i0) * kHq + head) * kD;
    const int64_t row1 = (static_cast<int64_t>(qs + i1) * kHq + head) * kD;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      if (v0) store_out2(out, row0 + 8 * nd + 2 * c, o[nd][0] * inv0, o[nd][1] * inv0, out_dtype);
      if (v1) store_out2(out, row1 + 8 * nd + 2 * c, o[nd][2] * inv1, o[nd][3] * inv1, out_dtype);
    }
  }
}

template <typename Kernel>
cudaError_t smem_optin_once(Kernel kernel, int bytes, bool (&done)[64]) {
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

cudaError_t prefill_smem_optin() {
  static bool done[64] = {};
  return smem_optin_once(prefill_attn_kernel, kPfSmemBytes, done);
}

cudaError_t prefill_tc_smem_optin() {
  static bool done[64] = {};
  return smem_optin_once(prefill_tc_kernel, tc::kSmemBytes, done);
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

extern "C" int hpc_prefill_attn(const void* q, const int32_t* query_start, const void* kv_cache,
                                int32_t kv_dtype, const float* kv_scale, int32_t num_blocks,
                                const int32_t* block_table, int32_t max_blocks,
                                const int32_t* seq_lens, int32_t batch, const int32_t* unit_ptr,
                                int32_t* counters, void* out, int32_t out_dtype, float sm_scale,
                                int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(q && query_start && kv_cache && block_table && seq_lens && unit_ptr && counters &&
                out && status);
  HPC_CHECK_ARG(batch >= 0 && num_blocks > 0 && max_blocks >= 1);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(kv_cache) & 15) == 0);
  if (out_dtype != HPC_OUT_BF16 && out_dtype != HPC_OUT_FP16 && out_dtype != HPC_OUT_FP32)
    return HPC_ERR_UNSUPPORTED;
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(q) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0);
  (void)kv_scale;
  if (kv_dtype != HPC_KV_BF16) return HPC_ERR_UNSUPPORTED;   // an E4M3 cache: not yet
  if (batch > HPC_MAX_BATCH || num_blocks > HPC_MAX_NUM_BLOCKS) return HPC_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * hpc::kPage >= (int64_t{1} << 31)) return HPC_ERR_UNSUPPORTED;
  if (batch == 0) return HPC_OK;
  auto encode = hpc::tensor_map_encoder();
  if (encode == nullptr) return HPC_ERR_CUDA;
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(hpc::kD),
                              static_cast<cuuint64_t>(num_blocks) * 2 * hpc::kHkv * hpc::kPage};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(hpc::kD) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(hpc::kPage)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult cr = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_cache),
                             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return HPC_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HPC_ERR_CUDA;
  if (hpc::prefill_tc_smem_optin() != cudaSuccess) return HPC_ERR_CUDA;
  hpc::prefill_tc_kernel<<<sms, hpc::tc::kThreads, hpc::tc::kSmemBytes, stream>>>(
      map, static_cast<const uint16_t*>(q), query_start, seq_lens, batch, block_table, max_blocks,
      num_blocks, unit_ptr, counters, out, out_dtype, sm_scale, status);
  return HPC_LAUNCH_STATUS();
}
