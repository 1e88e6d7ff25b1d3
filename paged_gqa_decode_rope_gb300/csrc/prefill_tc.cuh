// Prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Source: page "[vllm] Introducing the HPC-Ops attention backend" (the
// backend serves prefill, decode and mixed batches); page "vLLM and Tencent
// Hunyuan upstream two HPC backends for NVIDIA Hopper", intro of "Two new HPC
// backends in the vLLM ecosystem" (64 query heads, 8 KV heads, head_dim 128,
// paged KV in 64-token blocks).  Each new token attends to its history and
// the new tokens up to itself.
//
// A work unit is (sequence, kv_head, 32 new tokens): two 128-row tiles
// ("lanes"), row r = 8 * token + query head of the group, tokens 0..15 in
// lane 0 and 16..31 in lane 1.  Both lanes read the same K/V pages, which one
// producer warp streams by TMA into a ring of stages (64-row x 128-byte
// boxes, 128-byte swizzle).  Per 64-key tile and lane:
//  * S = Q K^T (M 128, N 64, K 128: eight K-major steps, both operands in
//    shared memory) into one of the lane's two TMEM score buffers; a Q
//    loader warp loads each lane's Q tile by TMA (a 3-D map over [tokens,
//    heads, d]) as soon as the lane's last Q K^T of the previous unit is done;
//  * its softmax warpgroup (thread = row) loads the row of S, masks it by
//    position, keeps the running maximum until it grows by more than 2^8
//    (only then rescaling the row of O in TMEM), and writes P as BF16 pairs
//    back over the scores;
//  * O += P V (M 128, N 128 = d, K 64: four steps, A = P read from TMEM, B =
//    V MN-major in shared memory), O resident in TMEM for the whole unit.
// Each lane has its own MMA warp, so one lane's softmax runs overlap the
// other lane's products and one warp's barrier waits never idle the tensor
// core.  V rows past the sequence length (or of a tile whose
// block id is bad) are zeroed before any P V reads them: the cache may hold
// NaN there.  Every mbarrier wait is bounded; on a timeout the CTA winds
// down, lets its copies and products finish, and frees its TMEM.
//
// E4M3 caches (kFp8): no TMA ring of codes.  A converter warpgroup reads
// each tile's codes straight from the cache (the page two tiles on
// prefetched into L2), writes them as F16 (every E4M3 value is an F16 value)
// into the ring the MMA warps read, and turns each lane's BF16 Q tile into
// F16 in place (exact for |q| in [2^-14, 65504]); both products then run on
// F16 operands.  The K
// scale joins the softmax scale and the V scale the final division, so the
// result is the attention over the dequantised cache.
#pragma once

#include "common.cuh"

namespace hpc {
namespace {
namespace tc {

// warps 0-3: softmax of lane 0, 4-7: of lane 1, 8: K/V producer, 9: MMA of
// lane 0, 10: Q loader, 11: MMA of lane 1, 12-15 (E4M3 caches): converter.
// The third (and fourth) warpgroup lend registers to the softmax warpgroups.
constexpr int kWarpProd = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpQ = 10;
constexpr int kWarpMma1 = 11;
constexpr int kWarpConv0 = 12;
constexpr int kBox = 64 * 128;                      // one 64-row x 128-byte TMA box
constexpr int kPage = 2 * kBox;                     // BF16 page of one KV head (d = 128)
constexpr int kTileBytes = 2 * kPage;               // K + V of one tile as the MMA reads them
constexpr int kQBytes = 2 * 128 * 128;              // per lane: 2 halves of d x 128 rows x 128 B
constexpr int kOffBar = 208 * 1024;                 // after the rings and Q of either layout

template <bool kFp8>
struct Cfg;
template <>
struct Cfg<false> {   // BF16 cache: the MMA reads the TMA ring itself
  static constexpr int kThreads = 384;
  static constexpr int kPStages = 4;                // producer ring (TMA)
  static constexpr int kPStageBytes = 2 * kPage;    // K page + V page
  static constexpr int kMStages = kPStages;         // tiles the MMA side holds
  static constexpr int kOffM = 0;
  static constexpr int kOffQ = kMStages * kTileBytes;
  static constexpr uint32_t kRegsSoftmax = 200, kRegsMid = 104, kRegsConv = 0;
  static constexpr int kUnitReaders = 11;           // 2 MMA, Q loader, 8 softmax warps
};
template <>
struct Cfg<true> {    // E4M3 cache: the converter reads the codes itself into F16 tiles
  static constexpr int kThreads = 512;
  static constexpr int kPStages = 4;                // (no TMA ring: the producer loads no tile)
  static constexpr int kPStageBytes = 0;
  static constexpr int kMStages = 4;
  static constexpr int kOffM = 0;
  static constexpr int kOffQ = kOffM + kMStages * kTileBytes;
  static constexpr uint32_t kRegsSoftmax = 176, kRegsMid = 64, kRegsConv = 96;
  static constexpr int kUnitReaders = 15;           // + the 4 converter warps
};
static_assert(Cfg<false>::kOffQ + 2 * kQBytes <= kOffBar, "BF16 layout overlaps the barriers");
static_assert(Cfg<true>::kOffQ + 2 * kQBytes <= kOffBar, "E4M3 layout overlaps the barriers");
static_assert(Cfg<false>::kPStages <= 4 && Cfg<true>::kPStages <= 4 && Cfg<true>::kMStages <= 4,
              "barrier and flag arrays hold four stages");

template <bool kFp8>
constexpr int regs_needed() {   // per CTA, for the warpgroups' raised budgets
  return 256 * Cfg<kFp8>::kRegsSoftmax + 128 * Cfg<kFp8>::kRegsMid + 128 * Cfg<kFp8>::kRegsConv;
}

// mbarriers (index of the first of each kind; [l] per lane, [l][i] per lane and buffer)
constexpr int kBarRawFull = 0;     // [4] BF16: producer stage landed (TMA)
                                   // (4 .. 7 unused)
constexpr int kBarMFull = 8;       // [4] E4M3: F16 tile written (128 converter threads)
constexpr int kBarTEmpty = 12;     // [2][4] the lane's P V of the tile the MMA side holds done
                                   //     (a lane without the tile commits for it at its unit end)
constexpr int kBarSFull = 20;      // [2][2] scores written
constexpr int kBarPFull = 24;      // [2][2] P written over the scores (128 softmax threads)
constexpr int kBarOFinal = 28;     // [2] the lane's last P V of a unit done
constexpr int kBarOFree = 30;      // [2] the lane's O read out (128 softmax threads)
constexpr int kBarQFull = 32;      // [2] the lane's Q tile landed (TMA)
constexpr int kBarQReady = 34;     // [2] E4M3: the lane's Q tile turned into F16 (128 threads)
constexpr int kBarQFree = 36;      // [2] the lane's last Q K^T of a unit done
constexpr int kBarUnitFull = 38;   // [2] unit descriptor handed on
constexpr int kBarUnitEmpty = 40;  // [2] unit descriptor read (every warp that follows units)
constexpr int kBarDrain = 42;      // [2] every product of the lane's MMA warp done (at exit)
constexpr int kNumBars = 44;
constexpr int kRingInts = 8;       // b, h, pair, ntiles lane 0, ntiles lane 1
constexpr int kOffRing = kOffBar + kNumBars * 8;
constexpr int kOffOk = kOffRing + 2 * kRingInts * 4;   // [4] producer stages, [2] F16 tiles
constexpr int kOffMisc = kOffOk + 8 * 4;            // [0] abort flag, [1] TMEM address
// [8 softmax warps][32 rows][64 bytes]: one 32-column chunk of a warp's O rows
// in a 16-bit output type, on its way to global memory
constexpr int kEpiWarpBytes = 32 * 64;
constexpr int kOffEpi = (kOffMisc + 16 + 127) / 128 * 128;
constexpr int kSmemBytes = kOffEpi + 8 * kEpiWarpBytes + 1024;   // + slack for the 1024-byte alignment
static_assert(kSmemBytes <= 227 * 1024, "the prefill layout exceeds a CTA's shared memory");
constexpr uint32_t kTmemCols = 512;                 // lane l: S 256l + {0, 64}, O 256l + 128
constexpr int kLaneTokens = 16;
constexpr int kUnitTokens = 32;
constexpr float kRescaleLog2 = 8.0f;                // rescale O only when the max grows by > 2^8

// tiles of a lane of a unit: 0 without new tokens, else those its last token sees
__device__ __forceinline__ int lane_tiles(int qlen, int L, int first_token) {
  const int cnt = min(kLaneTokens, qlen - first_token);
  return cnt > 0 ? (L - qlen + first_token + cnt - 1) / hpc::kPage + 1 : 0;
}

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

// The chains below are executed by a whole converged MMA warp (one per
// lane): the descriptors stay warp-uniform and one elected thread issues
// every product of a chain back to back from one asm block (issued one by one
// from a single diverged thread, each product costs the issuer far more than
// the tensor core's time for it).

// S = Q K^T of one lane for one tile: eight K-major steps (16 of d each; Q
// halves of d 16 KB apart, K halves 8 KB, a step 32 bytes along a row) into
// d, a commit on s_full, and on q_free too if it was the lane's last tile of
// the unit (its Q tile may then be replaced).
__device__ __forceinline__ void umma_qk_lane(uint32_t d, uint64_t q, uint64_t k, uint32_t idesc,
                                             uint32_t s_full, bool last, uint32_t q_free) {
#define HPC_QK_STEP(QO, KO) \
  "add.s64 a, %1, " QO ";\n\tadd.s64 b, %2, " KO ";\n\t" \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
  asm volatile(
      "{\n\t.reg .pred e, f, pf, pt;\n\t.reg .b64 a, b;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.and.b32 f, %5, 0, e;\n\t"
      "setp.ne.b32 pf, %5, %5;\n\tsetp.eq.b32 pt, %5, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      HPC_QK_STEP("2", "2") HPC_QK_STEP("4", "4") HPC_QK_STEP("6", "6")
      HPC_QK_STEP("1024", "512") HPC_QK_STEP("1026", "514") HPC_QK_STEP("1028", "516")
      HPC_QK_STEP("1030", "518")
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t"
      "@f tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
      ::"r"(d), "l"(q), "l"(k), "r"(idesc), "r"(s_full), "r"(last ? 1u : 0u), "r"(q_free)
      : "memory");
#undef HPC_QK_STEP
}

template <bool kFp8>
__global__ void __launch_bounds__(tc::Cfg<kFp8>::kThreads, 1) prefill_tc_kernel(
    const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
    int32_t num_tokens, const uint8_t* __restrict__ kv_codes, const float* __restrict__ kv_scale,
    const int32_t* __restrict__ query_start, const int32_t* __restrict__ seq_lens, int32_t batch,
    const int32_t* __restrict__ block_table, int32_t max_blocks, int32_t num_blocks,
    const int32_t* __restrict__ unit_ptr, int32_t* counters, void* __restrict__ out,
    int32_t out_dtype, float sm_scale, int32_t* __restrict__ status,
    const int32_t* __restrict__ page_ptr, int32_t staged_pages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + tc::kOffBar);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  volatile int* ring = reinterpret_cast<volatile int*>(smem + tc::kOffRing);
  using C = tc::Cfg<kFp8>;
  // per producer stage and per tile the MMA side holds: 1 = a good block
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + tc::kOffOk);
  volatile int* tile_ok_of = kFp8 ? stage_ok + 4 : stage_ok;
  // the MMA side's ring: the TMA stages themselves, or the F16 tiles
  constexpr int kBarTileFull = kFp8 ? tc::kBarMFull : tc::kBarRawFull;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + tc::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + tc::kOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kPStages; ++s) mbar_init(bar(tc::kBarRawFull + s), 1);
    for (int c = 0; c < C::kMStages; ++c) {
      mbar_init(bar(tc::kBarMFull + c), 128);
      mbar_init(bar(tc::kBarTEmpty + c), 1);
      mbar_init(bar(tc::kBarTEmpty + 4 + c), 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(tc::kBarSFull + i), 1);
      mbar_init(bar(tc::kBarPFull + i), 128);
    }
    for (int l = 0; l < 2; ++l) {
      mbar_init(bar(tc::kBarDrain + l), 1);
      mbar_init(bar(tc::kBarOFinal + l), 1);
      mbar_init(bar(tc::kBarOFree + l), 128);
      mbar_init(bar(tc::kBarQFull + l), 1);
      mbar_init(bar(tc::kBarQReady + l), 128);
      mbar_init(bar(tc::kBarQFree + l), 1);
      mbar_init(bar(tc::kBarUnitFull + l), 1);
      mbar_init(bar(tc::kBarUnitEmpty + l), C::kUnitReaders);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == tc::kWarpMma) tmem_alloc(smem_u32(tmem_slot), tc::kTmemCols);   // both lanes' columns
  if (warp == tc::kWarpProd && lane == 0) {
    tma_prefetch_desc(&kv_map);
    tma_prefetch_desc(&q_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total_units = unit_ptr[batch];

  // a bounded wait by the whole warp; false (and the abort flag set) on a
  // timeout.  Fast path: the phase is already complete for every lane.
  auto wait_all = [&](int b, uint32_t parity) -> bool {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar(b), parity))) return true;
    bool ok = !*abort_flag && mbar_wait(bar(b), parity, status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) *abort_flag = 1;
    return ok;
  };
  // the next unit descriptor (slot u & 1), handed back once read
  struct Unit {
    int b, h, pair, nt[2];
  };
  auto read_unit = [&](uint32_t u, Unit& d) -> bool {
    const int r = static_cast<int>(u & 1);
    if (!wait_all(tc::kBarUnitFull + r, (u >> 1) & 1)) return false;
    const volatile int* slot = ring + r * tc::kRingInts;
    d.b = slot[0];
    d.h = slot[1];
    d.pair = slot[2];
    d.nt[0] = slot[3];
    d.nt[1] = slot[4];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(tc::kBarUnitEmpty + r));
    return true;
  };

  if (warp == tc::kWarpProd) {
    // ---------------------------------------------------------- producer
    regs_dec<C::kRegsMid>();
    // every pair of new tokens of a sequence reads the KV head's pages again
    const uint64_t policy = l2_evict_last_policy();
    uint32_t g = 0, n_pushed = 0;   // stream tiles issued, units handed on
    bool alive = true;
    while (alive) {
      int u = 0;
      if (lane == 0) u = atomicAdd(&counters[0], 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      int b = -1, h = 0, pair = 0, nt0 = 0, nt1 = 0;
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
        const int npair = (qlen + tc::kUnitTokens - 1) / tc::kUnitTokens;
        h = j % kHkv;
        pair = npair - 1 - j / kHkv;   // the pairs with the most keys first
        if (qlen < 1 || L < qlen || L > max_blocks * kPage || pair < 0 || qs < 0 ||
            qs + qlen > num_tokens) {
          if (lane == 0) atomicOr(status, HPC_STATUS_BAD_SEQ_LEN);
          nt0 = nt1 = -1;
        } else {
          nt0 = tc::lane_tiles(qlen, L, pair * tc::kUnitTokens);
          nt1 = tc::lane_tiles(qlen, L, pair * tc::kUnitTokens + tc::kLaneTokens);
          // staged pages: sequence b's pages are staged pages page_ptr[b] ..
          if (page_ptr != nullptr && page_ptr[b + 1] > staged_pages) {
            if (lane == 0) atomicOr(status, HPC_STATUS_PLAN_OVERFLOW);
            nt0 = nt1 = -1;
          }
        }
      }
      const int ntiles = max(nt0, nt1);
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
          volatile int* slot = ring + r * tc::kRingInts;
          slot[0] = b;
          slot[1] = h;
          slot[2] = pair;
          slot[3] = nt0;
          slot[4] = nt1;
          mbar_arrive(bar(tc::kBarUnitFull + r));
        }
      }
      ++n_pushed;
      if (!__shfl_sync(0xffffffffu, ok, 0) || b < 0) break;
      // the unit's tiles by TMA, BF16 caches only (for E4M3 caches the
      // converter reads the pages itself)
      for (int tb = 0; !kFp8 && tb < ntiles && alive; tb += 32) {
        const int t = tb + lane;
        const int bids = t < ntiles ? block_table[static_cast<int64_t>(b) * max_blocks + t] : 0;
        const int page0 = page_ptr != nullptr ? page_ptr[b] + tb : 0;   // staged page of tile tb
        for (int jj = 0; jj < min(32, ntiles - tb) && alive; ++jj) {
          const int bid = __shfl_sync(0xffffffffu, bids, jj);
          const bool good = bid >= 0 && bid < num_blocks;
          const int s = static_cast<int>(g % C::kPStages);
          int tok = 1;
          if (lane == 0) {
            const uint32_t use = g / C::kPStages;
            if (*abort_flag) {
              tok = 0;
            } else if (use > 0) {
              const uint32_t par = (use - 1) & 1;
              // the MMA side reads the stage itself; both lanes release it
              const bool freed = mbar_wait(bar(tc::kBarTEmpty + s), par, status) &&
                                 mbar_wait(bar(tc::kBarTEmpty + 4 + s), par, status);
              if (!freed) {
                *abort_flag = 1;
                tok = 0;
              }
            }
            if (tok && good) {
              stage_ok[s] = 1;
              const uint32_t fb = bar(tc::kBarRawFull + s);
              mbar_arrive_expect_tx(fb, C::kPStageBytes);
              const uint32_t dst = base + s * C::kPStageBytes;
              // the cache's block, or (staged) the staged copy of the sequence's page
              const int yb = page_ptr != nullptr ? page0 + jj : bid;
              const int yk = ((yb * 2 + 0) * kHkv + h) * kPage;
              const int yv = yk + kHkv * kPage;
              // two 64-row x 64-element boxes per page
              tma_load_2d(dst, &kv_map, 0, yk, fb, policy);
              tma_load_2d(dst + tc::kBox, &kv_map, 64, yk, fb, policy);
              tma_load_2d(dst + tc::kPage, &kv_map, 0, yv, fb, policy);
              tma_load_2d(dst + tc::kPage + tc::kBox, &kv_map, 64, yv, fb, policy);
            }
          }
          tok = __shfl_sync(0xffffffffu, tok, 0);
          if (tok && !good) {
            // a bad block id: no copy; the stage is marked (its keys are
            // masked, its V rows zeroed) and the status set
            uint4* vst = reinterpret_cast<uint4*>(smem + s * C::kPStageBytes + tc::kPage);
            for (int z = lane; z < tc::kPage / 16; z += 32) vst[z] = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              atomicOr(status, HPC_STATUS_BAD_BLOCK);
              stage_ok[s] = 0;
              mbar_arrive(bar(tc::kBarRawFull + s));
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
      // the last copy issued into every stage has landed before this warp
      // leaves, on every path: after an abort seen by another warp once this
      // one had finished issuing, nobody else waits on those stages
      {
        for (uint32_t s = 0; s < static_cast<uint32_t>(C::kPStages) && s < g; ++s) {
          const uint32_t last = s + C::kPStages * ((g - 1 - s) / C::kPStages);
          mbar_wait(bar(tc::kBarRawFull + s), (last / C::kPStages) & 1, status);
        }
      }
    }
  } else if (warp == tc::kWarpMma || warp == tc::kWarpMma1) {
    // ---------------------------------------------------------- MMA issuers
    // One warp per lane: while one waits on its lane's barriers, the products
    // the other has issued keep the tensor core busy.  The whole warp runs the
    // loop (descriptors warp-uniform); one elected thread issues each chain
    // and each commit.
    regs_dec<C::kRegsMid>();
    const int l = warp == tc::kWarpMma ? 0 : 1;
    constexpr uint32_t kIdescS = kFp8 ? umma_idesc_f16(128, 64, false) : umma_idesc_bf16(128, 64, false);
    constexpr uint32_t kIdescO = kFp8 ? umma_idesc_f16(128, 128, true) : umma_idesc_bf16(128, 128, true);
    // descriptors of the first step of each operand; a step adds a constant
    const uint64_t desc_q = umma_smem_desc(base + C::kOffQ + l * tc::kQBytes, 1024, 1024);
    const uint64_t desc_k = umma_smem_desc(base + C::kOffM, 1024, 1024);
    const uint64_t desc_v = umma_smem_desc(base + C::kOffM + tc::kPage, tc::kBox, 1024);
    constexpr uint64_t kStageStep = tc::kTileBytes >> 4;
    const uint32_t tl = tmem + 256 * l;   // the lane's columns: S 0 / 64, O 128
    constexpr int kBarQ = kFp8 ? tc::kBarQReady : tc::kBarQFull;   // Q as the MMA reads it
    uint32_t G = 0, U = 0, Gl = 0, Vl = 0;   // stream tiles, units read, lane tiles, lane units
    bool dead = false;
    Unit d;
    // O += P V of the lane's tile jj of the unit (ntl tiles); then its share
    // of the stage's release
    auto issue_pv = [&](int jj, int ntl) {
      const uint32_t g = G + jj, gl = Gl + jj, st = g % C::kMStages;
      if (dead || !wait_all(tc::kBarPFull + 2 * l + (gl & 1), (gl >> 1) & 1) ||
          (jj == 0 && Vl > 0 && !wait_all(tc::kBarOFree + l, (Vl - 1) & 1))) {
        dead = true;
        return;
      }
      tc_fence_after();
      umma_pv_lane(tl + 128, tl + 64 * (gl & 1), desc_v + st * kStageStep, kIdescO, jj != 0,
                   jj == ntl - 1, bar(tc::kBarOFinal + l), bar(tc::kBarTEmpty + 4 * l + st));
    };
    while (!dead) {
      if (!read_unit(U, d)) break;
      ++U;
      if (d.b < 0) break;
      const int nt = max(d.nt[0], d.nt[1]);
      if (nt <= 0) continue;
      const int ntl = l ? d.nt[1] : d.nt[0];
      const int L = seq_lens[d.b];
      if (ntl > 0 && !wait_all(kBarQ + l, Vl & 1)) break;
      for (int j = 0; j < ntl && !dead; ++j) {
        const uint32_t g = G + j, gl = Gl + j;
        const uint32_t st = g % C::kMStages;
        if (!wait_all(kBarTileFull + st, (g / C::kMStages) & 1)) {
          dead = true;
          break;
        }
        // V rows past the sequence length (the cache may hold NaN there) ->
        // zeros before this lane's P V of the tile reads them; only the page
        // of the sequence's last key has such rows.  Both lanes' warps write
        // the same zeros, each before its own P V (the converter does it for
        // E4M3 caches).
        const int keep = L - 64 * j;
        if (!kFp8 && keep < 64) {
          uint4* vst = reinterpret_cast<uint4*>(smem + st * tc::kTileBytes + tc::kPage);
          for (int z = keep * 8 + lane; z < 64 * 8; z += 32) {   // rows keep..63, both boxes
            vst[z] = make_uint4(0u, 0u, 0u, 0u);
            vst[tc::kBox / 16 + z] = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        umma_qk_lane(tl + 64 * (gl & 1), desc_q, desc_k + st * kStageStep, kIdescS,
                     bar(tc::kBarSFull + 2 * l + (gl & 1)), j == ntl - 1, bar(tc::kBarQFree + l));
        if (j >= 1) issue_pv(j - 1, ntl);
      }
      if (dead) break;
      if (ntl > 0) issue_pv(ntl - 1, ntl);
      if (dead) break;
      // the release of the tiles this lane has none in: commits, so they
      // arrive after the lane's earlier ones on the same barrier, each once
      // its tile has landed (an earlier commit would complete a phase the
      // producer has not waited for yet)
      for (int j = max(ntl, 0); j < nt && !dead; ++j) {
        const uint32_t g = G + j, st = g % C::kMStages;
        if (!wait_all(kBarTileFull + st, (g / C::kMStages) & 1)) {
          dead = true;
          break;
        }
        umma_commit_elect(bar(tc::kBarTEmpty + 4 * l + st));
      }
      if (dead) break;
      G += nt;
      if (ntl > 0) {
        Gl += ntl;
        ++Vl;
      }
    }
    // every product issued here has completed before TMEM is freed
    umma_commit_elect(bar(tc::kBarDrain + l));
    mbar_wait(bar(tc::kBarDrain + l), 0, status);
    __syncwarp();
  } else if (warp < 8) {
    // ---------------------------------------------------------- softmax warpgroups
    regs_inc<C::kRegsSoftmax>();
    const int l = warp >> 2;                           // lane (tile) of the unit
    const int row = threadIdx.x & 127;                 // 8 * token + head
    const int tok = row >> 3, hl = row & 7;
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 256 * l;
    // E4M3: scores of the codes times the K scale, outputs times the V scale
    // (also for BF16 pages staged from an E4M3 cache: the host passes the scales then)
    const float scale_log2 =
        sm_scale * 1.4426950408889634f * (kFp8 || kv_scale != nullptr ? kv_scale[0] : 1.f);
    const float v_scale = kFp8 || kv_scale != nullptr ? kv_scale[1] : 1.f;
    uint32_t G = 0, U = 0, Gl = 0, Vl = 0;
    bool dead = false;
    Unit d;
    while (!dead) {
      if (!read_unit(U, d)) break;
      ++U;
      if (d.b < 0) break;
      const int nt = max(d.nt[0], d.nt[1]);
      if (nt <= 0) continue;
      const int ntl = l ? d.nt[1] : d.nt[0];
      if (ntl <= 0) {
        G += nt;
        continue;
      }
      const int qs = query_start[d.b], qlen = query_start[d.b + 1] - qs, L = seq_lens[d.b];
      const int i = d.pair * tc::kUnitTokens + l * tc::kLaneTokens + tok;
      const bool valid = i < qlen;
      const int pos = L - qlen + i;
      const int head = d.h * kGroup + hl;
      float m_used = -INFINITY, lsum = 0.f;
      for (int j = 0; j < ntl; ++j) {
        const uint32_t g = G + j, gl = Gl + j;
        const int s = static_cast<int>(g % C::kMStages);
        if (!wait_all(tc::kBarSFull + 2 * l + (gl & 1), (gl >> 1) & 1) ||
            !wait_all(kBarTileFull + s, (g / C::kMStages) & 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64(trow + 64 * (gl & 1), sr);
        tmem_wait_ld();
        const bool tile_ok = tile_ok_of[s] != 0;
        const int key0 = j * kPage;
        // keys of this tile the row sees: 0 .. lim (none for lim < 0); only
        // the tiles on a row's diagonal (or a bad tile) need the mask, which
        // sets the other scores to -inf in place (a copy of the row would
        // cost a move per score on the unmasked tiles)
        const int lim = (valid && tile_ok) ? min(63, pos - key0) : -1;
        if (!__all_sync(0xffffffffu, lim == 63)) {
#pragma unroll
          for (int jk = 0; jk < 64; ++jk)
            if (jk > lim) sr[jk] = 0xff800000u;
        }
        // the row maximum of the raw scores, three-input maxima in 8
        // independent chains (each started from a pair); the scale is
        // positive, so it commutes with the maximum
        float m8[8];
#pragma unroll
        for (int jk = 0; jk < 64; jk += 2) {
          const int c = (jk >> 1) & 7;
          const float a = __uint_as_float(sr[jk]), b = __uint_as_float(sr[jk + 1]);
          m8[c] = jk < 16 ? fmaxf(a, b) : max3f(m8[c], a, b);
        }
        const float mx =
            max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) *
            scale_log2;
        // the running maximum moves only when it grows by more than 2^8
        // (weights stay <= 2^8); the row's O is then rescaled in TMEM
        const bool grow = mx > m_used + tc::kRescaleLog2;
        const float alpha = grow ? exp2_ftz(m_used - mx) : 1.f;   // 0 while m_used = -inf
        if (grow) {
          lsum *= alpha;
          m_used = mx;
        }
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // the previous tile's P V must be in O before it is rescaled: the
          // lane's tile-empty barrier of that tile completes with it
          if (!wait_all(tc::kBarTEmpty + 4 * l + (g - 1) % C::kMStages,
                        ((g - 1) / C::kMStages) & 1)) {
            dead = true;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int qc = 0; qc < 4; ++qc) {
            uint32_t ov[32];
            tmem_ld32(trow + 128 + 32 * qc, ov);
            tmem_wait_ld();
#pragma unroll
            for (int jk = 0; jk < 32; ++jk) ov[jk] = __float_as_uint(__uint_as_float(ov[jk]) * alpha);
            tmem_st32(trow + 128 + 32 * qc, ov);
          }
        }
        // p = 2^(s * scale - m) as one FMA and one exponential, packed as
        // BF16 (F16 for E4M3 caches) pairs over the scores; the row sum in 4
        // independent chains
        {
          const float nms = m_used == -INFINITY ? 0.f : -m_used;
          const uint64_t scale2 = f32x2(scale_log2, scale_log2), nms2 = f32x2(nms, nms);
          uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};   // pairs of row sums
          uint32_t pk[32];
#pragma unroll
          for (int jk = 0; jk < 32; ++jk) {
            float a0, a1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[2 * jk]), __uint_as_float(sr[2 * jk + 1])),
                                  scale2, nms2),
                        a0, a1);
            const float p0 = exp2_ftz(a0), p1 = exp2_ftz(a1);
            ps2[jk & 3] = add_f32x2(ps2[jk & 3], f32x2(p0, p1));
            pk[jk] = kFp8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
          }
          tmem_st32(trow + 64 * (gl & 1), pk);
          float s0, s1;
          f32x2_split(add_f32x2(add_f32x2(ps2[0], ps2[1]), add_f32x2(ps2[2], ps2[3])), s0, s1);
          lsum += s0 + s1;
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(tc::kBarPFull + 2 * l + (gl & 1)));
      }
      if (dead) break;
      // the row of O once the lane's last P V is done: divide by the row sum, store
      if (!wait_all(tc::kBarOFinal + l, Vl & 1)) break;
      tc_fence_after();
      const float inv = lsum > 0.f ? v_scale / lsum : 0.f;
      const int64_t orow = (static_cast<int64_t>(qs + i) * kHq + head) * kD;
      if (out_dtype == HPC_OUT_FP32) {
#pragma unroll
        for (int qc = 0; qc < 4; ++qc) {
          uint32_t ov[32];
          tmem_ld32(trow + 128 + 32 * qc, ov);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int jk = 0; jk < 32; jk += 8) {
              float v8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v8[e] = __uint_as_float(ov[jk + e]) * inv;
              store_out8(out, orow + 32 * qc + jk, v8, out_dtype);
            }
          }
        }
      } else {
        // 16-bit outputs: each 32-column chunk of the warp's 32 rows goes
        // through shared memory, so that a store instruction writes 64
        // contiguous bytes of each of 8 rows (a thread's own row, stored 16
        // bytes at a time, would make every store 32 separate requests on
        // this chain).  The 16-byte pieces of row r are rotated by (r / 2) % 4:
        // both the row-wise writes and the piece-wise reads are free of bank
        // conflicts.
        const bool h16 = out_dtype == HPC_OUT_FP16;
        uint8_t* ebuf = smem + tc::kOffEpi + warp * tc::kEpiWarpBytes;
        const int rr0 = lane >> 2, pp = lane & 3;   // read side: rows 8 s + rr0, piece pp
#pragma unroll
        for (int qc = 0; qc < 4; ++qc) {
          uint32_t ov[32];
          tmem_ld32(trow + 128 + 32 * qc, ov);
          tmem_wait_ld();
#pragma unroll
          for (int pc = 0; pc < 4; ++pc) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float a = __uint_as_float(ov[8 * pc + 2 * k]) * inv;
              const float b = __uint_as_float(ov[8 * pc + 2 * k + 1]) * inv;
              w[k] = h16 ? pack_f16(a, b) : pack_bf16(a, b);
            }
            *reinterpret_cast<uint4*>(ebuf + lane * 64 + 16 * (pc ^ ((lane >> 1) & 3))) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
#pragma unroll
          for (int st = 0; st < 4; ++st) {
            const int rr = 8 * st + rr0;                         // the warp's row read here
            const int rrow = (warp & 3) * 32 + rr;               // its row of the lane's tile
            const int ri = d.pair * tc::kUnitTokens + l * tc::kLaneTokens + (rrow >> 3);
            const uint4 v = *reinterpret_cast<const uint4*>(ebuf + rr * 64 + 16 * (pp ^ ((rr >> 1) & 3)));
            if (ri < qlen) {
              const int64_t o = (static_cast<int64_t>(qs + ri) * kHq + d.h * kGroup + (rrow & 7)) * kD +
                                32 * qc + 8 * pp;
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + o) = v;
            }
          }
          __syncwarp();   // the chunk is read before the next one is written
        }
      }
      tc_fence_before();
      mbar_arrive(bar(tc::kBarOFree + l));
      G += nt;
      Gl += ntl;
      ++Vl;
    }
  } else if (warp == tc::kWarpQ) {
    // ---------------------------------------------------------- Q loader
    // Each lane's Q tile, [16 tokens][8 heads][64 of d] boxes (two halves of
    // d), is loaded once the lane's last Q K^T of the previous unit is done.
    regs_dec<C::kRegsMid>();
    const uint64_t policy = l2_evict_first_policy();   // Q is read once
    uint32_t U = 0, vq0 = 0, vq1 = 0;
    Unit d;
    while (true) {
      if (!read_unit(U, d)) break;
      ++U;
      if (d.b < 0) break;
      if (max(d.nt[0], d.nt[1]) <= 0) continue;
      const int tok0 = query_start[d.b] + d.pair * tc::kUnitTokens;
      bool ok = true;
#pragma unroll
      for (int l = 0; l < 2; ++l) {
        if ((l ? d.nt[1] : d.nt[0]) <= 0) continue;
        uint32_t& vq = l ? vq1 : vq0;
        if (vq > 0 && !wait_all(tc::kBarQFree + l, (vq - 1) & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t qb = bar(tc::kBarQFull + l);
          const uint32_t dst = base + C::kOffQ + l * tc::kQBytes;
          const int t = tok0 + l * tc::kLaneTokens;
          mbar_arrive_expect_tx(qb, tc::kQBytes);
          tma_load_3d(dst, &q_map, 0, d.h * kGroup, t, qb, policy);
          tma_load_3d(dst + 2 * tc::kBox, &q_map, 64, d.h * kGroup, t, qb, policy);
        }
        ++vq;
      }
      if (!ok) break;
    }
    // the last Q copy of each lane has landed before this warp leaves (on
    // every path: the MMA side may have stopped waiting on an abort)
    if (lane == 0) {
      if (vq0 > 0) mbar_wait(bar(tc::kBarQFull + 0), (vq0 - 1) & 1, status);
      if (vq1 > 0) mbar_wait(bar(tc::kBarQFull + 1), (vq1 - 1) & 1, status);
    }
    __syncwarp();
  } else if (kFp8 && warp >= tc::kWarpConv0) {
    // ---------------------------------------------------------- converter (E4M3)
    // Per unit: each lane's Q tile BF16 -> F16 in place (thread = row), then
    // each tile's K and V codes, read from the cache (global memory, the
    // page two tiles on prefetched into L2), -> F16 into the MMA side's
    // ring, in the layout a BF16 stage has (two 64-column boxes per page,
    // 128-byte swizzle); V rows past the sequence length, or of a bad block
    // (status set), -> 0.
    regs_dec<C::kRegsConv>();
    const int t = static_cast<int>(threadIdx.x) - 32 * tc::kWarpConv0;   // 0 .. 127
    uint32_t G = 0, U = 0, vq0 = 0, vq1 = 0;
    bool dead = false;
    Unit d;
    while (!dead) {
      if (!read_unit(U, d)) break;
      ++U;
      if (d.b < 0) break;
      const int nt = max(d.nt[0], d.nt[1]);
      if (nt <= 0) continue;
      const int L = seq_lens[d.b];
#pragma unroll
      for (int l = 0; l < 2; ++l) {
        if (dead || (l ? d.nt[1] : d.nt[0]) <= 0) continue;
        uint32_t& vq = l ? vq1 : vq0;
        if (!wait_all(tc::kBarQFull + l, vq & 1)) {
          dead = true;
          break;
        }
        uint8_t* qrow = smem + C::kOffQ + l * tc::kQBytes + t * 128;
        // 8 BF16 -> 8 F16 per 16-byte chunk, in place; the chunk order is
        // rotated by the row, so the eight rows of a quarter-warp touch eight
        // different 16-byte bank groups at every step
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int cc = (c & 8) | ((c ^ t) & 7);
          uint4* p = reinterpret_cast<uint4*>(qrow + (cc >> 3) * 2 * tc::kBox + (cc & 7) * 16);
          uint4 w = *p;
          w.x = pack_f16(bf16_lo(w.x), bf16_hi(w.x));
          w.y = pack_f16(bf16_lo(w.y), bf16_hi(w.y));
          w.z = pack_f16(bf16_lo(w.z), bf16_hi(w.z));
          w.w = pack_f16(bf16_lo(w.w), bf16_hi(w.w));
          *p = w;
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(tc::kBarQReady + l));
        ++vq;
      }
      // the unit's pages, read here straight from the cache: row r of a page
      // is 128 codes at r * 128; this thread's 16-byte chunks z = t + 128 k
      const int64_t bt = static_cast<int64_t>(d.b) * max_blocks;
      auto page = [&](int bid, int kv) {
        return kv_codes + ((static_cast<int64_t>(bid) * 2 + kv) * kHkv + d.h) * (kPage * kD);
      };
      for (int j = 0; j < nt && !dead; ++j) {
        const uint32_t g = G + j;
        const int c = static_cast<int>(g % C::kMStages);
        // the page two tiles on into L2 (one 128-byte line per thread)
        if (j + 2 < nt) {
          const int bid2 = block_table[bt + j + 2];
          if (bid2 >= 0 && bid2 < num_blocks)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(page(bid2, t >> 6) + (t & 63) * 128));
        }
        const int bid = block_table[bt + j];
        const bool ok = bid >= 0 && bid < num_blocks;
        if (!ok && t == 0) atomicOr(status, HPC_STATUS_BAD_BLOCK);
        const int keep = ok ? max(0, min(64, L - 64 * j)) : 0;
        uint4 kw[4], vw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int z = t + 128 * k;
          kw[k] = ok ? *reinterpret_cast<const uint4*>(page(bid, 0) + z * 16) : make_uint4(0u, 0u, 0u, 0u);
          vw[k] = (z >> 3) < keep ? *reinterpret_cast<const uint4*>(page(bid, 1) + z * 16)
                                  : make_uint4(0u, 0u, 0u, 0u);
        }
        if (g >= static_cast<uint32_t>(C::kMStages) &&
            (!wait_all(tc::kBarTEmpty + c, ((g - C::kMStages) / C::kMStages) & 1) ||
             !wait_all(tc::kBarTEmpty + 4 + c, ((g - C::kMStages) / C::kMStages) & 1))) {
          dead = true;
          break;
        }
        uint8_t* dst = smem + C::kOffM + c * tc::kTileBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // 16 codes of row r (d = 16 lc .. 16 lc + 15) -> half lc / 4 of d,
          // logical chunks 2 (lc % 4) and the next, swizzled by the row.  The
          // lanes of the second half store their odd chunk first, so the eight
          // lanes of a row (a quarter-warp) write eight different 16-byte bank
          // groups with each store
          const int z = t + 128 * k, r = z >> 3, lc = z & 7;
          const int hd = lc >> 2, dl = (lc & 3) * 2 + hd;
          const int o0 = hd * tc::kBox + r * 128 + ((dl ^ (r & 7)) << 4);
          const int o1 = hd * tc::kBox + r * 128 + (((dl ^ 1) ^ (r & 7)) << 4);
          const uint4 wk = kw[k], wv = vw[k];
          const uint4 w = hd ? make_uint4(wk.z, wk.w, wk.x, wk.y) : wk;
          const uint4 v = hd ? make_uint4(wv.z, wv.w, wv.x, wv.y) : wv;
          *reinterpret_cast<uint4*>(dst + o0) =
              make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w.x)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.x >> 16)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.y)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.y >> 16)));
          *reinterpret_cast<uint4*>(dst + o1) =
              make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w.z)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.z >> 16)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.w)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(w.w >> 16)));
          *reinterpret_cast<uint4*>(dst + tc::kPage + o0) =
              make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(v.x)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(v.x >> 16)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(v.y)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(v.y >> 16)));
          *reinterpret_cast<uint4*>(dst + tc::kPage + o1) =
              make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(v.z)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(v.z >> 16)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(v.w)),
                         e4m3x2_to_f16x2(static_cast<uint16_t>(v.w >> 16)));
        }
        if (t == 0) tile_ok_of[c] = ok ? 1 : 0;
        fence_proxy_async_smem();
        mbar_arrive(bar(tc::kBarMFull + c));
      }
      G += nt;
    }
  } else {
    regs_dec<C::kRegsMid>();   // the idle warp of the third warpgroup
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
