// Prefill attention on the 5th-generation tensor cores (tcgen05): the work
// unit of prefill.cu (sequence, kv_head, 16 new tokens) as one 128-row tile,
// row r = 8 * token + query head of the group.
//
// Source: as prefill.cu (prefill, decode and mixed batches over the paged
// cache; 64 query heads, 8 KV heads, head_dim 128).
//
// Per unit and 64-key tile (warp roles):
//  * producer warp: claims units, hands them on through a ring, and streams
//    the visible K and V pages by TMA into a 3-stage ring (128-byte swizzle);
//  * MMA warp (one elected lane issues): S = Q K^T into one of two TMEM
//    buffers (M 128, N 64 keys, K 128 as 8 K-major steps), then, once the
//    softmax has written P, O += P V (A = P K-major, B = V MN-major, two
//    N = 64 halves of d), O resident in TMEM for the whole unit;
//  * softmax warpgroup (4 warps, thread = row): loads its S row from TMEM,
//    masks by position, keeps the running maximum until it grows by more
//    than 2^8 (only then rescales its O row in TMEM), writes P as BF16 into
//    shared memory, zeroes V rows past the sequence length, and at the end
//    divides its O row by the row sum and stores it.
// Every mbarrier wait is bounded; on a timeout the CTA winds down, and the
// TMEM it holds is freed before it exits.
#pragma once

#include "common.cuh"

namespace hpc {
namespace {
namespace tc {

constexpr int kThreads = 192;          // warps 0-3 softmax, 4 producer, 5 MMA
constexpr int kWarpProd = 4;
constexpr int kWarpMma = 5;
constexpr int kStages = 3;
constexpr int kBox = 64 * 128;                      // one 64-row x 128-byte TMA box
constexpr int kPage = 2 * kBox;                     // BF16 page of one KV head (128 d)
constexpr int kStageBytes = 2 * kPage;              // K page + V page
constexpr int kOffQ = kStages * kStageBytes;        // Q: 2 halves of d x 128 rows x 128 B
constexpr int kQBytes = 2 * 128 * 128;
constexpr int kOffP = kOffQ + kQBytes;              // P: 2 buffers x 128 rows x 64 keys (BF16)
constexpr int kPBytes = 128 * 128;
constexpr int kOffBar = kOffP + 2 * kPBytes;
// mbarriers (index of the first of each kind)
constexpr int kBarFull = 0;        // [3] stage landed (TMA)
constexpr int kBarEmpty = 3;       // [3] stage consumed (the tile's P V done)
constexpr int kBarSFull = 6;       // [2] S buffer written (tcgen05.commit)
constexpr int kBarSFree = 8;       // [2] S buffer read (128 softmax threads)
constexpr int kBarPFull = 10;      // [2] P buffer written (128 softmax threads)
constexpr int kBarPFree = 12;      // [2] P buffer read (the P V done)
constexpr int kBarODone = 14;      // every P V done, in order
constexpr int kBarOFinal = 15;     // a unit's last P V done
constexpr int kBarOFree = 16;      // a unit's O read out (128 softmax threads)
constexpr int kBarQReady = 17;     // a unit's Q written (128 softmax threads)
constexpr int kBarUnitFull = 18;   // [2] unit descriptor handed on
constexpr int kBarUnitEmpty = 20;  // [2] unit descriptor read (MMA warp + 4 softmax warps)
constexpr int kBarDrain = 22;      // every tcgen05 op of the MMA warp done (at exit)
constexpr int kNumBars = 23;
constexpr int kOffRing = kOffBar + kNumBars * 8;
constexpr int kOffOk = kOffRing + 2 * 4 * 4;
constexpr int kOffMisc = kOffOk + kStages * 4;      // [0] abort flag, [1] TMEM address
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = 256;                 // S0 0..63, S1 64..127, O 128..255
constexpr int kTokens = 16;
constexpr float kRescaleLog2 = 8.0f;                // rescale O only when the max grows by > 2^8

}  // namespace tc

// Eight consecutive output elements (index a multiple of 8) in the caller's type.
__device__ __forceinline__ void store_out8(void* out, int64_t idx, const float (&v)[8],
                                           int32_t out_dtype) {
  if (out_dtype == HPC_OUT_FP32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
    o[0] = make_float4(v[0], v[1], v[2], v[3]);
    o[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    const bool h = out_dtype == HPC_OUT_FP16;
    uint4 p;
    p.x = h ? pack_f16(v[0], v[1]) : pack_bf16(v[0], v[1]);
    p.y = h ? pack_f16(v[2], v[3]) : pack_bf16(v[2], v[3]);
    p.z = h ? pack_f16(v[4], v[5]) : pack_bf16(v[4], v[5]);
    p.w = h ? pack_f16(v[6], v[7]) : pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + idx) = p;
  }
}

__global__ void __launch_bounds__(tc::kThreads, 1) prefill_tc_kernel(
    const __grid_constant__ CUtensorMap kv_map, const uint16_t* __restrict__ q,
    const int32_t* __restrict__ query_start, const int32_t* __restrict__ seq_lens, int32_t batch,
    const int32_t* __restrict__ block_table, int32_t max_blocks, int32_t num_blocks,
    const int32_t* __restrict__ unit_ptr, int32_t* counters, void* __restrict__ out,
    int32_t out_dtype, float sm_scale, int32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + tc::kOffBar);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  volatile int* ring = reinterpret_cast<volatile int*>(smem + tc::kOffRing);
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + tc::kOffOk);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + tc::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + tc::kOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < tc::kStages; ++s) {
      mbar_init(bar(tc::kBarFull + s), 1);
      mbar_init(bar(tc::kBarEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(tc::kBarSFull + i), 1);
      mbar_init(bar(tc::kBarSFree + i), 128);
      mbar_init(bar(tc::kBarPFull + i), 128);
      mbar_init(bar(tc::kBarPFree + i), 1);
      mbar_init(bar(tc::kBarUnitFull + i), 1);
      mbar_init(bar(tc::kBarUnitEmpty + i), 5);
    }
    mbar_init(bar(tc::kBarODone), 1);
    mbar_init(bar(tc::kBarOFinal), 1);
    mbar_init(bar(tc::kBarOFree), 128);
    mbar_init(bar(tc::kBarQReady), 128);
    mbar_init(bar(tc::kBarDrain), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == tc::kWarpMma) tmem_alloc(smem_u32(tmem_slot), tc::kTmemCols);
  if (warp == tc::kWarpProd && lane == 0) tma_prefetch_desc(&kv_map);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total_units = unit_ptr[batch];

  // a bounded wait by the whole warp; false (and the abort flag set) on a timeout
  auto wait_all = [&](int b, uint32_t parity) -> bool {
    bool ok = !*abort_flag && mbar_wait(bar(b), parity, status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) *abort_flag = 1;
    return ok;
  };

  if (warp == tc::kWarpProd) {
    // ---------------------------------------------------------- producer
    const uint64_t policy = l2_evict_first_policy();
    uint32_t g = 0, n_pushed = 0;   // tiles issued, units handed on
    bool alive = true;
    while (alive) {
      int u = 0;
      if (lane == 0) u = atomicAdd(&counters[0], 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      int b = -1, h = 0, qb = 0, ntiles = 0;
      if (u < total_units) {
        int lo = 0, hi = batch;   // the last b with unit_ptr[b] <= u (32-ary search)
        while (hi - lo > 1) {
          const int step = (hi - lo + 31) / 32;
          const int idx = lo + lane * step;
          const bool le = idx < hi && unit_ptr[idx] <= u;
          const uint32_t m = __ballot_sync(0xffffffffu, le);
          lo += (31 - __clz(m)) * step;
          hi = min(hi, lo + step);
        }
        b = lo;
        const int j = u - unit_ptr[b];
        const int qs = query_start[b], qlen = query_start[b + 1] - qs, L = seq_lens[b];
        const int nqb = (qlen + tc::kTokens - 1) / tc::kTokens;
        h = j % kHkv;
        qb = nqb - 1 - j / kHkv;   // the blocks with the most keys first
        if (qlen < 1 || L < qlen || L > max_blocks * kPage || qb < 0) {
          if (lane == 0) atomicOr(status, HPC_STATUS_BAD_SEQ_LEN);
          ntiles = -1;
        } else {
          const int last = min(tc::kTokens, qlen - qb * tc::kTokens) - 1;
          ntiles = (L - qlen + qb * tc::kTokens + last) / kPage + 1;
        }
      }
      int ok = 1;
      if (lane == 0) {
        const int r = static_cast<int>(n_pushed & 1);
        const uint32_t use = n_pushed >> 1;
        if (*abort_flag) {
          ok = 0;
        } else if (use > 0 && !mbar_wait(bar(tc::kBarUnitEmpty + r), (use - 1) & 1, status)) {
          *abort_flag = 1;
          ok = 0;
        }
        if (ok) {
          volatile int* slot = ring + r * 4;
          slot[0] = b;
          slot[1] = h;
          slot[2] = qb;
          slot[3] = ntiles;
          mbar_arrive(bar(tc::kBarUnitFull + r));
        }
      }
      ++n_pushed;
      if (!__shfl_sync(0xffffffffu, ok, 0) || b < 0) break;
      for (int tb = 0; tb < ntiles && alive; tb += 32) {
        const int t = tb + lane;
        const int bids = t < ntiles ? block_table[static_cast<int64_t>(b) * max_blocks + t] : 0;
        for (int jj = 0; jj < min(32, ntiles - tb) && alive; ++jj) {
          int bid = __shfl_sync(0xffffffffu, bids, jj);
          int tok = 1;
          if (lane == 0) {
            const int s = static_cast<int>(g % tc::kStages);
            const uint32_t use = g / tc::kStages;
            if (*abort_flag) {
              tok = 0;
            } else if (use > 0 && !mbar_wait(bar(tc::kBarEmpty + s), (use - 1) & 1, status)) {
              *abort_flag = 1;
              tok = 0;
            }
            if (tok) {
              // a bad block id loads block 0 in its place and marks the
              // stage: the softmax masks its keys and zeroes its V rows
              const bool good = bid >= 0 && bid < num_blocks;
              if (!good) {
                atomicOr(status, HPC_STATUS_BAD_BLOCK);
                bid = 0;
              }
              stage_ok[s] = good ? 1 : 0;
              const uint32_t fb = bar(tc::kBarFull + s);
              mbar_arrive_expect_tx(fb, tc::kStageBytes);
              const uint32_t dst = base + s * tc::kStageBytes;
              const int yk = ((bid * 2 + 0) * kHkv + h) * kPage;
              const int yv = yk + kHkv * kPage;
              tma_load_2d(dst, &kv_map, 0, yk, fb, policy);
              tma_load_2d(dst + tc::kBox, &kv_map, 64, yk, fb, policy);
              tma_load_2d(dst + tc::kPage, &kv_map, 0, yv, fb, policy);
              tma_load_2d(dst + tc::kPage + tc::kBox, &kv_map, 64, yv, fb, policy);
            }
          }
          alive = __shfl_sync(0xffffffffu, tok, 0) != 0;
          if (alive) ++g;
        }
      }
    }
    if (lane == 0) {
      if (atomicAdd(&counters[1], 1) == static_cast<int>(gridDim.x) - 1) {
        counters[0] = 0;   // the last CTA resets the counters: the plan can run again
        counters[1] = 0;
      }
      if (*abort_flag) {   // copies still landing in stages nobody waits on
        for (uint32_t s = 0; s < static_cast<uint32_t>(tc::kStages) && s < g; ++s) {
          const uint32_t last = s + tc::kStages * ((g - 1 - s) / tc::kStages);
          mbar_wait(bar(tc::kBarFull + s), (last / tc::kStages) & 1, status);
        }
      }
    }
  } else if (warp == tc::kWarpMma) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdescS = umma_idesc_bf16(128, 64, false);
    constexpr uint32_t kIdescO = umma_idesc_bf16(128, 64, true);
    uint32_t G = 0, U = 0, V = 0;   // tiles, unit descriptors read, units with tiles
    bool dead = false;
    // O (+)= P V of global tile gp; the unit's first overwrites O, its last
    // also signals the readout
    auto issue_pv = [&](uint32_t gp, bool first, bool last) {
      if (dead || !wait_all(tc::kBarPFull + (gp & 1), (gp >> 1) & 1) ||
          (first && V > 0 && !wait_all(tc::kBarOFree, (V - 1) & 1))) {
        dead = true;
        return;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t pb = base + tc::kOffP + (gp & 1) * tc::kPBytes;
        const uint32_t vb = base + (gp % tc::kStages) * tc::kStageBytes + tc::kPage;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {        // 16 keys per step
#pragma unroll
          for (int dh = 0; dh < 2; ++dh)        // halves of d, N = 64 each
            umma_bf16_ss(tmem + 128 + 64 * dh, umma_smem_desc(pb + 32 * ks, 1024, 1024),
                         umma_smem_desc(vb + dh * tc::kBox + ks * 2048, 1024, 1024), kIdescO,
                         !(first && ks == 0));
        }
        umma_commit(bar(tc::kBarPFree + (gp & 1)));
        umma_commit(bar(tc::kBarEmpty + gp % tc::kStages));
        umma_commit(bar(tc::kBarODone));
        if (last) umma_commit(bar(tc::kBarOFinal));
      }
      __syncwarp();
    };
    while (!dead) {
      const int r = static_cast<int>(U & 1);
      if (!wait_all(tc::kBarUnitFull + r, (U >> 1) & 1)) break;
      const int b = ring[r * 4 + 0], ntiles = ring[r * 4 + 3];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(tc::kBarUnitEmpty + r));
      ++U;
      if (b < 0) break;
      if (ntiles <= 0) continue;
      if (!wait_all(tc::kBarQReady, V & 1)) break;
      const uint32_t n = static_cast<uint32_t>(ntiles);
      for (uint32_t t = 0; t < n && !dead; ++t) {
        const uint32_t g = G + t;
        if (!wait_all(tc::kBarFull + g % tc::kStages, (g / tc::kStages) & 1) ||
            (g >= 2 && !wait_all(tc::kBarSFree + (g & 1), ((g - 2) >> 1) & 1))) {
          dead = true;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t qa = base + tc::kOffQ;
          const uint32_t kb = base + (g % tc::kStages) * tc::kStageBytes;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {       // 16 of d per step
            const uint32_t off = (ks >> 2) * tc::kBox * 2 + (ks & 3) * 32;
            const uint32_t koff = (ks >> 2) * tc::kBox + (ks & 3) * 32;
            umma_bf16_ss(tmem + 64 * (g & 1), umma_smem_desc(qa + off, 1024, 1024),
                         umma_smem_desc(kb + koff, 1024, 1024), kIdescS, ks > 0);
          }
          umma_commit(bar(tc::kBarSFull + (g & 1)));
        }
        __syncwarp();
        if (t >= 1) issue_pv(g - 1, t == 1, false);
      }
      if (dead) break;
      issue_pv(G + n - 1, n == 1, true);
      G += n;
      ++V;
    }
    // every tcgen05 op issued here has completed before TMEM is freed
    if (lane == 0) {
      umma_commit(bar(tc::kBarDrain));
      mbar_wait(bar(tc::kBarDrain), 0, status);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- softmax warpgroup
    const int row = threadIdx.x;                       // 0 .. 127: 8 * token + head
    const int tok = row >> 3, hl = row & 7;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const float scale_log2 = sm_scale * 1.4426950408889634f;
    uint32_t G = 0, U = 0, V = 0;
    bool dead = false;
    while (!dead) {
      const int r = static_cast<int>(U & 1);
      if (!wait_all(tc::kBarUnitFull + r, (U >> 1) & 1)) break;
      const int b = ring[r * 4 + 0], h = ring[r * 4 + 1], qb = ring[r * 4 + 2],
                ntiles = ring[r * 4 + 3];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(tc::kBarUnitEmpty + r));
      ++U;
      if (b < 0) break;
      if (ntiles <= 0) continue;
      const int qs = query_start[b], qlen = query_start[b + 1] - qs, L = seq_lens[b];
      const int i = qb * tc::kTokens + tok;
      const bool valid = i < qlen;
      const int pos = L - qlen + i;
      const int head = h * kGroup + hl;
      // this row of Q into the swizzled tile (zeros past the chunk); the
      // previous unit's S products, the last readers of the tile, are done
      {
        const uint4* src =
            reinterpret_cast<const uint4*>(q + (static_cast<int64_t>(qs + i) * kHq + head) * kD);
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const uint4 v = valid ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
          const int half = ch >> 3, c8 = ch & 7;
          *reinterpret_cast<uint4*>(smem + tc::kOffQ + half * 2 * tc::kBox + row * 128 +
                                    ((c8 ^ (row & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(tc::kBarQReady));
      float m_used = -INFINITY, l = 0.f;
      const uint32_t n = static_cast<uint32_t>(ntiles);
      for (uint32_t t = 0; t < n; ++t) {
        const uint32_t g = G + t;
        const int s = static_cast<int>(g % tc::kStages);
        if (!wait_all(tc::kBarSFull + (g & 1), (g >> 1) & 1) ||
            !wait_all(tc::kBarFull + s, (g / tc::kStages) & 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64(tmem + lane_addr + 64 * (g & 1), sr);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(tc::kBarSFree + (g & 1)));
        const bool tile_ok = stage_ok[s] != 0;
        const int key0 = static_cast<int>(t) * kPage;
        float mx = -INFINITY;
        float x[64];
#pragma unroll
        for (int jk = 0; jk < 64; ++jk) {
          x[jk] = (valid && tile_ok && key0 + jk <= pos) ? __uint_as_float(sr[jk]) * scale_log2
                                                          : -INFINITY;
          mx = fmaxf(mx, x[jk]);
        }
        // the running maximum moves only when it grows by more than 2^8
        // (weights stay <= 2^8); the row's O is then rescaled in TMEM
        const bool grow = mx > m_used + tc::kRescaleLog2;
        const float alpha = grow ? exp2_ftz(m_used - mx) : 1.f;   // 0 while m_used = -inf
        if (grow) {
          l *= alpha;
          m_used = mx;
        }
        if (t > 0 && __any_sync(0xffffffffu, grow)) {
          // the previous tile's P V must be in O before it is rescaled
          if (!wait_all(tc::kBarODone, (g - 1) & 1)) {
            dead = true;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t ov[64];
            tmem_ld64(tmem + lane_addr + 128 + 64 * half, ov);
            tmem_wait_ld();
#pragma unroll
            for (int jk = 0; jk < 64; ++jk) ov[jk] = __float_as_uint(__uint_as_float(ov[jk]) * alpha);
            tmem_st64(tmem + lane_addr + 128 + 64 * half, ov);
          }
          tmem_wait_st();
        }
        const float ms = m_used == -INFINITY ? 0.f : m_used;
        float ps = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int jk = 0; jk < 32; ++jk) {
          const float p0 = exp2_ftz(x[2 * jk] - ms), p1 = exp2_ftz(x[2 * jk + 1] - ms);
          ps += p0 + p1;
          pk[jk] = pack_bf16(p0, p1);
        }
        l += ps;
        // P row into its buffer once the P V two tiles back has read it
        if (g >= 2 && !wait_all(tc::kBarPFree + (g & 1), ((g - 2) >> 1) & 1)) {
          dead = true;
          break;
        }
        uint8_t* prow = smem + tc::kOffP + (g & 1) * tc::kPBytes + row * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          *reinterpret_cast<uint4*>(prow + ((c8 ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
        // V rows past the sequence length (the cache may hold NaN there) or
        // of a bad tile become zeros: 0 * NaN would poison O
        const int keep = tile_ok ? max(0, min(64, L - key0)) : 0;
        if (keep < 64) {
          uint8_t* vst = smem + s * tc::kStageBytes + tc::kPage;
          const int nz = (64 - keep) * 16;   // 16-byte chunks: rows x 2 boxes x 8
          for (int z = row; z < nz; z += 128) {
            const int vr = keep + (z >> 4), box = (z >> 3) & 1, c8 = z & 7;
            *reinterpret_cast<uint4*>(vst + box * tc::kBox + vr * 128 + (c8 << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(tc::kBarPFull + (g & 1)));
      }
      if (dead) break;
      // the row of O once the unit's last P V is done: divide by the row sum, store
      if (!wait_all(tc::kBarOFinal, V & 1)) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow = (static_cast<int64_t>(qs + i) * kHq + head) * kD;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t ov[64];
        tmem_ld64(tmem + lane_addr + 128 + 64 * half, ov);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int jk = 0; jk < 64; jk += 8) {
            float v8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v8[e] = __uint_as_float(ov[jk + e]) * inv;
            store_out8(out, orow + 64 * half + jk, v8, out_dtype);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(tc::kBarOFree));
      G += n;
      ++V;
    }
  }
  // every warp is done with TMEM: free it
  tc_fence_before();
  __syncthreads();
  if (warp == tc::kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, tc::kTmemCols);
  }
}

}  // namespace
}  // namespace hpc
