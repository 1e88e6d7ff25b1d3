#pragma once
// Split-KV paged GQA decode attention, sm_103a: one new token per sequence
// (decode) or q_len = 2..4 new tokens (multi-token decode, causal among the
// new tokens).
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper": intro of "Two new HPC backends in the vLLM ecosystem" (64 query
// heads, 8 KV heads, head_dim 128; the multi-token-prediction layer of the
// model) and "Why does dynamic scheduling matter for attention?" (split-KV
// over 64-token tiles dealt to compute units in proportion to length; BF16
// and FP8).  Page "[vllm] Introducing the HPC-Ops attention backend",
// introduction (FP8 E4M3 models).
//
// Design (GB300-first; the pages give no kernel structure):
//  * Persistent grid, one CTA per SM, each CTA hosting kGroups work queues.
//    Queue k of CTA b runs the plan's range b * kGroups + k: its home items,
//    then pooled chunks it claims.  The path is bound by HBM: each 64-token K
//    page and V page of a KV head is read exactly once and serves all 8 query
//    heads of its group (and all new tokens of its sequence).
//  * A queue has one producer warp that streams pages with TMA
//    (cp.async.bulk.tensor, 128-byte swizzle, L2 evict-first) into its own
//    ring of stages guarded by mbarriers; a stage is one tile = the K page +
//    the V page of one (block, kv_head).  Block ids are fetched 32 at a time
//    by the whole warp, so the issue loop never waits on a global load per
//    tile.  Its four consumer warps run whole work items; one queue's
//    epilogue and merge overlap the other queues' streaming.
//  * Inside a queue the warps split the tile: with kQ tokens per query
//    layout, 4 / kQ warps serve each query and each covers 16 * kQ tokens.
//    Every warp keeps its own online-softmax state (running max m, sum l,
//    output O) for the current item; at the end of an item the states of a
//    query's warps are merged in shared memory, in a fixed warp order, and
//    written as one partial (O, lse) per query.
//  * Tensor cores without padding: S^T[16 tok x 8 heads] = K[16 x 128] .
//    Q^T[128 x 8] (m16n8k16, tokens on M, heads on N), then O^T[128 x 8] +=
//    V^T[128 x 16 tok] . P^T[16 x 8] (d on M, heads on N).  The softmax runs
//    on the S^T accumulator fragment; movmatrix transposes P^T into the
//    B-operand layout, so P never touches shared memory.
//  * FP8 E4M3 pages are converted to f16 in registers after ldmatrix
//    (exact), q is taken to f16 once per item; the k scale folds into the
//    softmax scale and the v scale into the output.  For FP8 the dot products
//    run over a fixed permutation of d (and the V rows over a permutation of
//    d inside each 16-row tile) that makes each ldmatrix word feed the MMA
//    directly; q uses the same permutation and the epilogue undoes it.
//  * With an E4M3 q (kQ8; E4M3 caches only) Q K^T runs as E4M3 x E4M3
//    products (m16n8k32) on the codes themselves, q_scale joining the
//    softmax scale; P V stays f16.
//  * With the merge fused in (out set), a segment of one item is written to
//    the output directly; the queue that finishes the last item of a longer
//    segment (a per-segment arrival counter, one acquire-release atomic)
//    merges its partials in item order, so the result does not depend on
//    which queue merges.  A queue merging after its own last item lands the
//    partials in its idle stages by cp.async first.
//  * Tokens past a query's last visible key get p = 0 and their V entries
//    are zeroed in registers (the cache may hold NaN there: 0 * NaN is NaN).
//  * The 4-token layout (q_len 3, 4; and q_len 2 with an E4M3 q on an E4M3
//    cache, where the rows of the third and fourth tokens stay empty) runs
//    the tensor-core form (kTC): its
//    q_len x 8 query rows are one M = 128 tcgen05 operand, so per 64-token
//    tile a single Q K^T (N 64) into tensor memory, a softmax warp with one
//    row per thread, and one P V (N 128, P read from tensor memory) serve
//    all new tokens; an MMA warp per queue issues the products of two tiles
//    in flight, whichever is ready first.  Over E4M3 pages Q K^T runs on
//    E4M3 products (kind::f8f6f4) directly on the landed K codes, a BF16 q
//    split per row into two E4M3 terms under a power-of-two row scale (exact
//    for every element within 2^10 of the row's largest); two converter
//    warps widen only the V page to F16, in place.  A segment of one item is
//    written to the output directly; the other items' partials are combined
//    by the merge pass after the kernel.
//  * Every wait is bounded (kWaitLimitNs): a stuck pipeline records
//    HPC_STATUS_WAIT_TIMEOUT and winds down, waiting for its own copies.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace hpc {
namespace {

// kTC: the tensor-core form of the 4-token layout: per queue one MMA warp
// issuing tcgen05 products into tensor memory, one softmax warp and (E4M3
// pages) two converter warps; the Q tiles sit ahead of the stage rings.
template <bool kFp8, bool kTC = false>
struct AttnTraits {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kPageBytes = kPage * kD * kElem;      // one K or V page of one KV head
  static constexpr int kBoxBytes = 64 * 128;                  // one 64-row x 128-byte TMA box
  static constexpr int kTmaStageBytes = 2 * kPageBytes;       // K page + V page as loaded
  // a stage of the tensor-core form holds the tile as the products read it:
  // BF16 K and V pages, or over E4M3 pages the K page of codes as it landed
  // (Q K^T runs on E4M3 products) and the V page widened to F16 in place
  static constexpr int kF16Page = kPage * kD * 2;
  // (over E4M3 pages: the K page as landed, then V widened in place, 24 KB)
  static constexpr int kStageBytes = kTC ? (kFp8 ? kPageBytes + kF16Page : 2 * kF16Page) : kTmaStageBytes;
  // A CTA hosts kGroups independent work queues.  A queue has its own producer
  // warp, stage ring, item ring and 4 consumer warps, and runs whole work
  // items, so one queue's epilogue and merge overlap the other queues'
  // streaming.  FP8 tiles carry a longer per-tile chain (the conversions) at
  // half the bytes, so FP8 keeps three queues in flight.
  static constexpr int kGroups = (kFp8 && !kTC) ? 3 : 2;
  static constexpr int kGroupStages = (kTC && kFp8) ? 4 : 3;   // stage ring of one queue
  // tiles per queue pulled into L2 while a programmatic dependent launch
  // waits for the plan (about 29 MB in all on a 152-SM part)
  static constexpr int kL2PrefetchTiles = kFp8 ? 4 : 3;
  static constexpr int kStages = kGroups * kGroupStages;
  static constexpr int kWarpsPerGroup = 4;                    // 16 tokens of a tile each
  static constexpr int kConsumerWarps = kGroups * kWarpsPerGroup;
  static constexpr int kGroupThreads = 32 * kWarpsPerGroup;
  static constexpr int kThreads = 32 * (kConsumerWarps + kGroups);   // + a producer warp per queue
  static constexpr int kOStride = kD + 4;                     // padded row of the merge buffer
  // tensor-core form: per queue a 16 KB Q tile of 64 rows (BF16 pages: two
  // 64-column halves; E4M3 pages: the rows' leading E4M3 terms, then their
  // remainders, 128 codes a row); the M = 128 operand's rows past 64 read
  // whatever follows, which the products ignore, and the tiles sit ahead of
  // the rings so that those rows stay in bounds
  static constexpr int kQtBytes = 16384;
  static constexpr int kOffQt = 0;
  static constexpr int kOffStages = kTC ? kGroups * kQtBytes : 0;
  static constexpr int kSliceWarps = kTC ? 0 : kConsumerWarps;   // merge slices (the mma.sync form)
  static constexpr int kOffO = kOffStages + kStages * kStageBytes;    // [warps][8][kOStride]
  static constexpr int kOffM = kOffO + kSliceWarps * kGroup * kOStride * 4;
  static constexpr int kOffL = kOffM + kSliceWarps * kGroup * 4;
  static constexpr int kOffBar = kOffL + kSliceWarps * kGroup * 4;
  static constexpr int kItemRing = 2;                         // items queued ahead, per queue
  // barriers of one queue: full[SG], empty[SG], item_full[R], item_empty[R], consumer barrier,
  // and for the tensor-core form s_full[2], p_full[2], q_full, q_free, o_final, o_free, drain,
  // and over E4M3 pages conv_v[SG] (the stage's V widened to F16)
  static constexpr int kTcBars = kTC ? 9 + (kFp8 ? kGroupStages : 0) : 0;
  static constexpr int kGroupBars = 2 * kGroupStages + 2 * kItemRing + 1 + kTcBars;
  static constexpr int kOffOk = kOffBar + kGroups * kGroupBars * 8;
  static constexpr int kOffRing = kOffOk + kStages * 4;
  static constexpr int kRingInts = 8;                         // idx, seq, h, t0, t1, len
  // flags: the CTA's abort flag, one merge flag per queue, the TMEM address
  static constexpr int kOffFlags = kOffRing + kGroups * kItemRing * kRingInts * 4;
  static constexpr int kSmemUsed = kOffFlags + 4 * (2 + kGroups);
  static constexpr int kSmemBytes = kSmemUsed + 1024;         // slack for 1024-byte alignment
  static_assert(kOffBar % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory");
};

struct Item {
  int seq, h, t0, t1, len;
  bool ok;
};

// The item (w = {seq, kv_head, tile_begin, tile_end}) checked against the
// batch, with `len` the length of its sequence (-1 if the sequence id is bad).
__device__ __forceinline__ Item make_item(int4 w, int len, int batch, int max_blocks) {
  Item it{w.x, w.y, w.z, w.w, 0, false};
  if (it.seq >= 0 && it.seq < batch && it.h >= 0 && it.h < kHkv && len >= 0 &&
      len <= max_blocks * kPage) {
    const int n = (len + kPage - 1) / kPage;
    if (it.t0 >= 0 && it.t0 < it.t1 && it.t1 <= n) {
      it.ok = true;
      it.len = len;
    }
  }
  return it;
}

// Diagnostic record of one CTA: [start ns, end ns, SM id] (globaltimer).
__device__ __forceinline__ void record_cta_clock(unsigned long long* cta_clock,
                                                 unsigned long long t_start) {
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  cta_clock[3 * blockIdx.x + 0] = t_start;
  cta_clock[3 * blockIdx.x + 1] = globaltimer_ns();
  cta_clock[3 * blockIdx.x + 2] = smid;
}

// Tiles of a sequence length (0 for a length out of range).
__device__ __forceinline__ int tiles_of_len(int L, int max_blocks) {
  return (L > 0 && L <= max_blocks * kPage) ? (L + kPage - 1) / kPage : 0;
}

// The first `ntiles` tiles of work queue vq under the length-proportional
// plan, pulled into L2 by one warp.  The plan gives queue vq the flat tiles
// (in (sequence, kv_head, tile) order) from vq * q, with q = ceil(T /
// queues), or at least the common tile count when every sequence has the
// same one and there are no more segments than queues; this is worked out
// here from the lengths and the block table alone.  Only tiles of the
// sequence holding the queue's first tile are taken.  A prefetch only warms
// L2: a guess that misses the plan (another min_tiles, say) costs
// bandwidth, never correctness, and L2 stays coherent with later writes.
template <bool kFp8>
__device__ void l2_prefetch_queue_start(const CUtensorMap* map, const int32_t* seq_lens, int batch,
                                        const int32_t* block_table, int max_blocks, int num_blocks,
                                        int vq, int num_queues, int ntiles) {
  const int lane = threadIdx.x & 31;
  const int n0 = batch > 0 ? tiles_of_len(seq_lens[0], max_blocks) : 0;
  int tot = 0;
  bool same = true;
  for (int b = lane; b < batch; b += 32) {
    const int n = tiles_of_len(seq_lens[b], max_blocks);
    tot += n;
    same = same && n == n0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  same = __all_sync(0xffffffffu, same);
  const int64_t T = int64_t{kHkv} * tot;
  if (T == 0 || num_queues < 1) return;
  int64_t q = (T + num_queues - 1) / num_queues;
  if (same && static_cast<int64_t>(batch) * kHkv <= num_queues && n0 > q) q = n0;
  const int64_t f0 = static_cast<int64_t>(vq) * q;
  if (f0 >= T) return;
  const int64_t fend = min(T, f0 + q);
  // the sequence whose segments hold flat tile f0, 32 sequences at a time
  int64_t base = 0;   // tiles of the sequences before the chunk
  int bsel = -1, nsel = 0;
  int64_t start = 0;  // flat tile of sequence bsel's first segment
  for (int cb = 0; cb < batch && bsel < 0; cb += 32) {
    const int b = cb + lane;
    const int n = b < batch ? tiles_of_len(seq_lens[b], max_blocks) : 0;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned m = __ballot_sync(0xffffffffu, b < batch && kHkv * (base + incl) > f0);
    if (m != 0u) {
      const int src = __ffs(m) - 1;
      bsel = cb + src;
      nsel = __shfl_sync(0xffffffffu, n, src);
      start = kHkv * (base + __shfl_sync(0xffffffffu, incl, src) - nsel);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (bsel < 0 || nsel <= 0) return;
  const int64_t r = f0 - start + lane;   // lane's tile within the sequence's segments
  if (lane < ntiles && f0 + lane < fend && r < int64_t{kHkv} * nsel) {
    const int h = static_cast<int>(r / nsel), t = static_cast<int>(r % nsel);
    const int bid = block_table[static_cast<int64_t>(bsel) * max_blocks + t];
    if (bid >= 0 && bid < num_blocks) {
      const int yk = ((bid * 2 + 0) * kHkv + h) * kPage;   // row of [bid][0][h][0]
      const int yv = yk + kHkv * kPage;                     // row of [bid][1][h][0]
      tma_prefetch_l2_2d(map, 0, yk);
      tma_prefetch_l2_2d(map, 0, yv);
      if constexpr (!kFp8) {
        tma_prefetch_l2_2d(map, 64, yk);
        tma_prefetch_l2_2d(map, 64, yv);
      }
    }
  }
}

// O^T += V^T P^T for one warp's 16 tokens (rows: d, cols: 8 heads).  With
// kMask, V entries of tokens past the length are zeroed first (mask01 covers
// the fragment's tokens 2c, 2c+1; mask23 tokens 2c+8, 2c+9).
template <bool kFp8, bool kMask>
__device__ __forceinline__ void pv_tile(uint32_t vb, int row, int vtok_bf16, int vsel_bf16, int hi,
                                        int sw, uint32_t pb0, uint32_t pb1, uint32_t mask01,
                                        uint32_t mask23, float (&o)[8][4]) {
  if constexpr (kFp8) {
#pragma unroll
    for (int mp = 0; mp < 4; ++mp) {
      uint32_t r0, r1, r2, r3;
      ldsm_x4_t(vb + row * 128 + ((((2 * mp + hi) & 7) ^ sw) << 4), r0, r1, r2, r3);
      // r0: tokens 2c, 2c+1 at d 2r, 2r+1 (bytes t0d0, t0d1, t1d0, t1d1); the
      // byte shuffle pairs the two tokens of one d for each f16x2
      const uint32_t x = prmt(r0, 0, 0x3120), y = prmt(r1, 0, 0x3120);
      const uint32_t z = prmt(r2, 0, 0x3120), w = prmt(r3, 0, 0x3120);
      uint32_t a[8] = {e4m3x2_to_f16x2(x & 0xffff), e4m3x2_to_f16x2(x >> 16),
                       e4m3x2_to_f16x2(y & 0xffff), e4m3x2_to_f16x2(y >> 16),
                       e4m3x2_to_f16x2(z & 0xffff), e4m3x2_to_f16x2(z >> 16),
                       e4m3x2_to_f16x2(w & 0xffff), e4m3x2_to_f16x2(w >> 16)};
      if constexpr (kMask) {
        a[0] &= mask01; a[1] &= mask01; a[2] &= mask23; a[3] &= mask23;
        a[4] &= mask01; a[5] &= mask01; a[6] &= mask23; a[7] &= mask23;
      }
      mma_f16(o[2 * mp], a[0], a[1], a[2], a[3], pb0, pb1);
      mma_f16(o[2 * mp + 1], a[4], a[5], a[6], a[7], pb0, pb1);
    }
  } else {
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vb + (mi >> 2) * (64 * 128) + vtok_bf16 * 128 + ((((2 * mi + vsel_bf16) & 7) ^ sw) << 4),
                a0, a1, a2, a3);
      if constexpr (kMask) {
        a0 &= mask01; a1 &= mask01; a2 &= mask23; a3 &= mask23;
      }
      mma_bf16(o[mi], a0, a1, a2, a3, pb0, pb1);
    }
  }
}

// S = Q K^T of one queue for one tile (tensor-core form): eight K-major steps
// of 16 d, the second 64-column halves of both operands 8 KB on; a commit on
// s_full, and on q_free too after the item's last tile (its Q tile may then
// be replaced).  Run by the whole converged MMA warp; one elected thread
// issues the chain.
__device__ __forceinline__ void umma_qk_tile(uint32_t d, uint64_t q, uint64_t k, uint32_t idesc,
                                             uint32_t s_full, bool last, uint32_t q_free) {
#define HPC_DQK_STEP(O) \
  "add.s64 a, %1, " O ";\n\tadd.s64 b, %2, " O ";\n\t" \
  "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
  asm volatile(
      "{\n\t.reg .pred e, f, pf, pt;\n\t.reg .b64 a, b;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.and.b32 f, %5, 0, e;\n\t"
      "setp.ne.b32 pf, %5, %5;\n\tsetp.eq.b32 pt, %5, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      HPC_DQK_STEP("2") HPC_DQK_STEP("4") HPC_DQK_STEP("6")
      HPC_DQK_STEP("512") HPC_DQK_STEP("514") HPC_DQK_STEP("516") HPC_DQK_STEP("518")
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t"
      "@f tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
      ::"r"(d), "l"(q), "l"(k), "r"(idesc), "r"(s_full), "r"(last ? 1u : 0u), "r"(q_free)
      : "memory");
#undef HPC_DQK_STEP
}

// One 128-code row of an E4M3 page (128-byte swizzled, as TMA lands it),
// read into registers (zeros when !live), and written back as 128 F16 values
// in two 128-byte swizzled rows, d 0..63 and 64..127 (the layout of a 16-bit
// stage).
__device__ __forceinline__ void load_e4m3_row(const uint8_t* raw, int r, bool live, uint4 (&w)[8]) {
  const int sw = r & 7;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    w[c] = live ? *reinterpret_cast<const uint4*>(raw + ((c ^ sw) << 4)) : make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void store_f16_row(const uint4 (&w)[8], uint8_t* lo_row, uint8_t* hi_row, int r) {
  const int sw = r & 7;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint8_t* dst = c < 4 ? lo_row : hi_row;
    const int c0 = (2 * c) & 7, c1 = (2 * c + 1) & 7;   // 16-byte F16 chunks of codes 16c ..
    *reinterpret_cast<uint4*>(dst + ((c0 ^ sw) << 4)) =
        make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w[c].x)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(w[c].x >> 16)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(w[c].y)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(w[c].y >> 16)));
    *reinterpret_cast<uint4*>(dst + ((c1 ^ sw) << 4)) =
        make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(w[c].z)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(w[c].z >> 16)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(w[c].w)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(w[c].w >> 16)));
  }
}

// Four consecutive output elements (index a multiple of 4) in the caller's
// output type.
__device__ __forceinline__ void store_out4(void* out, int64_t idx, float a, float b, float c,
                                           float d, int32_t out_dtype) {
  if (out_dtype == HPC_OUT_FP32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = make_float4(a, b, c, d);
  } else {
    uint2 p;
    p.x = out_dtype == HPC_OUT_FP16 ? pack_f16(a, b) : pack_bf16(a, b);
    p.y = out_dtype == HPC_OUT_FP16 ? pack_f16(c, d) : pack_bf16(c, d);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) = p;
  }
}

// kQ: query layout, 1 (decode), 2 or 4 new tokens per sequence (q_len = 3
// runs the 4-token layout with the fourth query's warp idle).  kQ8: q is E4M3
// codes (FP8 cache only) and QK^T runs as E4M3 x E4M3 products.
template <bool kFp8, int kQ, bool kQ8, bool kTC = false>
__global__ void __launch_bounds__(AttnTraits<kFp8, kTC>::kThreads, 1) decode_attn_kernel(
    // q, the plan arrays and the cache may be written by the kernel this one
    // is a programmatic dependent of: they are read with plain (coherent)
    // loads, never as restrict/read-only data, so that no load of them can be
    // hoisted above the grid-dependency wait
    const __grid_constant__ CUtensorMap kv_map, const void* q, float q_scale,
    const float* __restrict__ kv_scale, const int32_t* __restrict__ block_table, int32_t max_blocks,
    int32_t num_blocks, const int32_t* __restrict__ seq_lens, int32_t batch, int32_t q_len,
    const hpc_work_item* items, const int32_t* cta_ptr, const int32_t* home_end, int32_t* pool,
    int32_t capacity, int32_t num_queues, float* __restrict__ partial_o,
    float* __restrict__ partial_lse,
    float sm_scale, int32_t* __restrict__ status, unsigned long long* __restrict__ cta_clock,
    const int32_t* seg_ptr, int32_t* seg_done, void* __restrict__ out, int32_t out_dtype,
    int32_t l2_prefetch_tiles) {
  using T = AttnTraits<kFp8, kTC>;
  static_assert(kQ == 1 || kQ == 2 || kQ == 4, "query layouts of 1, 2 or 4 tokens");
  static_assert(!kTC || T::kGroups == 2, "tensor-core form: two queues");
  static_assert(kFp8 || !kQ8, "an E4M3 q needs an E4M3 cache");
  constexpr int kWq = T::kWarpsPerGroup / kQ;   // warps per query
  constexpr int kMB = kQ;                       // 16-token blocks per warp and tile
  constexpr int G = T::kGroups;
  constexpr int SG = T::kGroupStages;
  constexpr int R = T::kItemRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* sm_o = reinterpret_cast<float*>(smem + T::kOffO);
  float* sm_m = reinterpret_cast<float*>(smem + T::kOffM);
  float* sm_l = reinterpret_cast<float*>(smem + T::kOffL);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::kOffFlags);
  const bool fuse = out != nullptr;   // merge the partials in this kernel

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // warps 0 .. 4G-1 consume (queue k: warps 4k .. 4k+3); warp 4G + k produces for queue k
  const bool is_producer = warp >= T::kConsumerWarps;
  const int grp = is_producer ? warp - T::kConsumerWarps : warp / T::kWarpsPerGroup;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::kOffBar) + grp * T::kGroupBars;
  uint64_t* empty = full + SG;
  uint64_t* item_full = empty + SG;
  uint64_t* item_empty = item_full + R;
  uint64_t* cons_bar = item_empty + R;
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + T::kOffOk) + grp * SG;
  volatile int* ring = reinterpret_cast<volatile int*>(smem + T::kOffRing) + grp * R * T::kRingInts;
  volatile int* merge_flag = abort_flag + 1 + grp;
  const uint32_t stage_base =
      smem_u32(smem) + T::kOffStages + grp * SG * T::kStageBytes;   // this queue's stages

  const unsigned long long t_start = cta_clock != nullptr ? globaltimer_ns() : 0ull;
  if (threadIdx.x == 0) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::kOffBar);
    for (int k = 0; k < G; ++k) {
      uint64_t* b = bars + k * T::kGroupBars;
      for (int st = 0; st < SG; ++st) {
        mbar_init(smem_u32(&b[st]), 1);                           // full
        // empty: the consumer warps, or the commit of the tile's P V
        mbar_init(smem_u32(&b[SG + st]), kTC ? 1 : T::kWarpsPerGroup);
      }
      for (int r = 0; r < R; ++r) {
        mbar_init(smem_u32(&b[2 * SG + r]), 1);                   // item_full
        // item_empty: every reading warp (tensor-core form: the MMA and softmax
        // warps, and over E4M3 pages the two converter warps)
        mbar_init(smem_u32(&b[2 * SG + R + r]), kTC ? (kFp8 ? 4 : 2) : T::kWarpsPerGroup);
      }
      mbar_init(smem_u32(&b[2 * SG + 2 * R]), T::kGroupThreads);  // the queue's consumer barrier
      for (int x = 0; x < T::kTcBars; ++x)   // conv_v: one arrival per converter warp
        mbar_init(smem_u32(&b[2 * SG + 2 * R + 1 + x]), x >= 9 ? 2 : 1);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == T::kConsumerWarps && lane == 0) tma_prefetch_desc(&kv_map);
  // As a programmatic dependent of the step's prologue + planner launch the
  // CTAs are resident while the plan is made: each producer warp uses that
  // wait to pull its queue's first tiles into L2.
  if (l2_prefetch_tiles > 0 && is_producer)
    l2_prefetch_queue_start<kFp8>(&kv_map, seq_lens, batch, block_table, max_blocks, num_blocks,
                                  static_cast<int>(blockIdx.x) * G + grp, num_queues,
                                  l2_prefetch_tiles);
  // everything above is independent of the previous kernel on the stream;
  // from here on the plan, q and the cache are read
  pdl_wait();

  // The pool counters are pool[0] (next claim) and pool[1] (queues done
  // claiming); the last queue to finish claiming resets both, so the same
  // plan can be run again.  Every queue of the grid takes part in the pool.
  const int queues_in_grid = static_cast<int>(gridDim.x) * G;
  auto finish_claims = [&]() {
    if (atomicAdd(&pool[1], 1) == queues_in_grid - 1) {
      pool[0] = 0;
      pool[1] = 0;
    }
  };

  // every thread checks the ranges of all the CTA's queues, so that the CTA
  // leaves as a whole on a bad plan; queues past num_queues have no home part
  const int pool_len = pool[2];
  bool bad_range = pool_len < 0 || pool_len > capacity;
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int vq = static_cast<int>(blockIdx.x) * G + k;
    if (vq < num_queues) {
      const int b0 = cta_ptr[vq], b1 = home_end[vq];
      bad_range = bad_range || b0 < 0 || b1 < b0 || b1 > capacity;
    }
  }
  if (bad_range) {
    if (threadIdx.x == 0) {
      atomicOr(status, HPC_STATUS_BAD_PLAN);
      for (int k = 0; k < G; ++k) finish_claims();
      if (cta_clock != nullptr) record_cta_clock(cta_clock, t_start);
    }
    return;
  }
  const int vq = static_cast<int>(blockIdx.x) * G + grp;   // this warp's queue
  const int home_begin = vq < num_queues ? cta_ptr[vq] : 0;
  const int home_stop = vq < num_queues ? home_end[vq] : 0;

  // tensor-core form: 512 TMEM columns, 256 per queue (scores 0 / 64, O 128),
  // allocated by warp 3, freed by it after every warp's final barrier
  constexpr int kTmemWarp = 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + T::kOffFlags) + 1 + G;
  if constexpr (kTC) {
    if (warp == kTmemWarp) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (kTC) tc_fence_after();

  // ------------------------------------------------------------ producer
  // The producer does not wait on a global load in its issue loop: the home
  // items' descriptors and lengths arrive 32 at a time (one per lane), the
  // block ids of the next 32 tiles are fetched while the current 32 are
  // issued (across item boundaries), and a pool claim is made when an item
  // starts and resolved during its last chunk.
  if (is_producer) {
    const uint64_t policy = l2_evict_first_policy();
    const int4* items4 = reinterpret_cast<const int4*>(items);
    uint32_t g = 0;          // tiles issued so far into this queue's ring
    uint32_t n_pushed = 0;   // items handed to the consumers so far
    bool claiming = true;    // the pool is not known to be empty yet
    bool alive = true;
    int ticket = -1;         // lane 0: an unresolved pool claim (its counter value)

    // Home items in the order: the first, the last, then the others.  A
    // range's first and last items are the pieces of segments it shares with
    // the ranges before and after it, which run them first as well; so those
    // segments' merges come early instead of at the end of the launch.
    const int home_n = home_stop - home_begin;
    auto home_index = [&](int p) {   // the item at position p of that order
      return home_n >= 3 && p >= 1 ? (p == 1 ? home_stop - 1 : home_begin + p - 1) : home_begin + p;
    };
    // home items, 32 at a time: lane j holds the item at position
    // hb_next - home_begin - hb_cnt + j
    int hb_next = home_begin, hb_cnt = 0, hb_pos = 0;
    int4 hw = make_int4(-1, -1, 0, 0);
    int hlen = -1;
    auto load_home_batch = [&]() {
      hb_cnt = min(32, home_stop - hb_next);
      hb_pos = 0;
      hw = make_int4(-1, -1, 0, 0);
      hlen = -1;
      if (lane < hb_cnt) {
        hw = items4[home_index(hb_next - home_begin + lane)];
        hlen = (hw.x >= 0 && hw.x < batch) ? __ldg(seq_lens + hw.x) : -1;
      }
      hb_next += hb_cnt;
    };
    // start a pool claim (lane 0) once the home part is used up
    auto start_claim = [&]() {
      if (lane == 0 && claiming && ticket < 0 && hb_pos == hb_cnt && hb_next == home_stop)
        ticket = atomicAdd(&pool[0], 1);
    };
    // next item: {index, descriptor, length}; index -1 when nothing is left
    struct Next {
      int idx;
      int4 w;
      int len;
    };
    auto next_item = [&]() -> Next {
      while (true) {
        if (hb_pos == hb_cnt && hb_next < home_stop) load_home_batch();
        if (hb_pos < hb_cnt) {
          Next n;
          n.idx = home_index(hb_next - hb_cnt + hb_pos - home_begin);
          n.w.x = __shfl_sync(0xffffffffu, hw.x, hb_pos);
          n.w.y = __shfl_sync(0xffffffffu, hw.y, hb_pos);
          n.w.z = __shfl_sync(0xffffffffu, hw.z, hb_pos);
          n.w.w = __shfl_sync(0xffffffffu, hw.w, hb_pos);
          n.len = __shfl_sync(0xffffffffu, hlen, hb_pos);
          ++hb_pos;
          return n;
        }
        if (!claiming) return Next{-1, make_int4(-1, -1, 0, 0), -1};
        start_claim();
        const int k = __shfl_sync(0xffffffffu, ticket, 0);
        if (lane == 0) ticket = -1;
        if (k < pool_len) {
          const int idx = pool[3 + k];
          if (idx < 0 || idx >= capacity) {
            if (lane == 0) atomicOr(status, HPC_STATUS_BAD_PLAN);
            continue;
          }
          Next n;
          n.idx = idx;
          n.w = items4[idx];
          n.len = (n.w.x >= 0 && n.w.x < batch) ? __ldg(seq_lens + n.w.x) : -1;
          return n;
        }
        claiming = false;
        if (lane == 0) finish_claims();
        return Next{-1, make_int4(-1, -1, 0, 0), -1};
      }
    };
    // block ids of tiles tb .. tb+31 of an item (lane j: tile tb + j)
    auto fetch_bids = [&](const Item& it, int tb) -> int {
      const int t = tb + lane;
      return (it.ok && t < it.t1) ? __ldg(block_table + static_cast<int64_t>(it.seq) * max_blocks + t)
                                  : 0;
    };
    // hand an item's descriptor (or the end mark) to the consumers
    auto push_item = [&](int idx, const Item& it) -> bool {
      int ok = 1;
      if (lane == 0) {
        const int r = static_cast<int>(n_pushed % R);
        const uint32_t use = n_pushed / R;
        if (*abort_flag) {
          ok = 0;
        } else if (use > 0 && !mbar_wait(smem_u32(&item_empty[r]), (use - 1) & 1, status)) {
          *abort_flag = 1;
          ok = 0;
        }
        if (ok) {
          volatile int* slot = ring + r * T::kRingInts;
          slot[0] = idx;
          slot[1] = it.seq;
          slot[2] = it.h;
          slot[3] = it.t0;
          slot[4] = it.t1;
          slot[5] = it.ok ? it.len : -1;
          mbar_arrive(smem_u32(&item_full[r]));
        }
      }
      ++n_pushed;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    // one stage: a tile (data, block id bid), or a slot without data
    auto issue = [&](int bid, int h, bool data) -> bool {
      int tok = 1;
      if (lane == 0) {
        const int s = static_cast<int>(g % SG);
        const uint32_t use = g / SG;
        if (*abort_flag) {
          tok = 0;
        } else if (use > 0 && !mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, status)) {
          *abort_flag = 1;
          tok = 0;
        }
        if (tok) {
          const uint32_t fb = smem_u32(&full[s]);
          if (data && bid >= 0 && bid < num_blocks) {
            stage_ok[s] = 1;
            mbar_arrive_expect_tx(fb, T::kTmaStageBytes);
            const uint32_t dst = stage_base + s * T::kStageBytes;
            const int yk = ((bid * 2 + 0) * kHkv + h) * kPage;   // row of [bid][0][h][0]
            const int yv = yk + kHkv * kPage;                     // row of [bid][1][h][0]
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
            if (data) atomicOr(status, HPC_STATUS_BAD_BLOCK);
            stage_ok[s] = 0;
            mbar_arrive(fb);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, tok, 0)) return false;
      ++g;
      return true;
    };

    Next cur = next_item();
    Item it = make_item(cur.w, cur.len, batch, max_blocks);
    int cur_bids = fetch_bids(it, it.t0);
    while (alive) {
      if (!push_item(cur.idx, it)) break;
      if (cur.idx < 0) break;
      if (!it.ok) {
        if (lane == 0) atomicOr(status, HPC_STATUS_BAD_PLAN);
      } else {
        start_claim();
      }
      Next nxt{-1, make_int4(-1, -1, 0, 0), -1};
      Item nit{-1, -1, 0, 0, 0, false};
      int nxt_bids = 0;
      bool have_next = false;
      for (int tb = it.t0; it.ok && tb < it.t1 && alive; tb += 32) {
        const int nt = min(32, it.t1 - tb);
        int pre = 0;
        if (tb + 32 < it.t1) {
          pre = fetch_bids(it, tb + 32);              // the next chunk of this item
        } else {
          nxt = next_item();                          // the next item and its first chunk
          nit = make_item(nxt.w, nxt.len, batch, max_blocks);
          nxt_bids = fetch_bids(nit, nit.t0);
          have_next = true;
        }
        for (int j = 0; j < nt && alive; ++j)
          alive = issue(__shfl_sync(0xffffffffu, cur_bids, j), it.h, true);
        cur_bids = pre;
      }
      if (!alive) break;
      if (!have_next) {
        nxt = next_item();
        nit = make_item(nxt.w, nxt.len, batch, max_blocks);
        nxt_bids = fetch_bids(nit, nit.t0);
      }
      cur = nxt;
      it = nit;
      cur_bids = nxt_bids;
    }
    if (claiming && lane == 0) finish_claims();   // stopped early by a fault
    // Wait for the last copy issued into every stage before this warp exits,
    // on every path: a queue that stops on a fault (its own, or the abort of
    // another queue of the CTA, seen after this producer finished issuing)
    // leaves copies landing in stages nobody else waits on, and the CTA must
    // not end while a copy still targets its shared memory.
    if (lane == 0) {
      for (uint32_t s = 0; s < static_cast<uint32_t>(SG) && s < g; ++s) {
        const uint32_t last = s + SG * ((g - 1 - s) / SG);
        mbar_wait(smem_u32(&full[s]), (last / SG) & 1, status);
      }
    }
    if constexpr (kTC) {
      __syncwarp();
      named_bar_sync(2, T::kThreads);   // every warp done; TMEM is freed after this
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int wq = warp % T::kWarpsPerGroup;         // warp within the queue
  const int gt = threadIdx.x - grp * T::kGroupThreads;   // thread index within the queue
  const int qj = wq / kWq;                          // this warp's query (new token)
  const int tok0 = (wq % kWq) * 16 * kMB;           // its first token of every tile
  const int r = lane >> 2, c = lane & 3;
  const float k_scale = kFp8 ? kv_scale[0] : 1.f;
  const float v_scale = kFp8 ? kv_scale[1] : 1.f;
  const float scale_log2 = sm_scale * k_scale * (kQ8 ? q_scale : 1.f) * 1.4426950408889634f;
  const int sw = lane & 7;                                        // swizzle of this lane's row
  const int row = tok0 + (lane & 7) + ((lane >> 3) & 1) * 8;      // ldmatrix row (token), block 0
  const int hi = lane >> 4;                                        // second 16-byte chunk
  const int vtok_bf16 = tok0 + (lane & 7) + hi * 8;                // V^T .trans row (token), block 0
  const int vsel_bf16 = (lane >> 3) & 1;                           // V^T d half
  uint32_t g = 0;
  uint32_t bar_phase = 0;
  bool dead = false;

  // the queue's consumer threads meet; bounded, so a stuck peer ends in a timeout
  auto cons_sync = [&]() -> bool {
    mbar_arrive(smem_u32(cons_bar));
    bool ok = !*abort_flag && mbar_wait(smem_u32(cons_bar), bar_phase & 1, status);
    ++bar_phase;
    ok = __all_sync(0xffffffffu, ok);   // the same answer for the whole warp
    if (!ok && lane == 0) *abort_flag = 1;
    return ok;
  };

  // with the merge fused in, the rows of empty sequences (no items) are
  // zeroed here, the segments spread over the CTAs of the grid
  if (fuse) {
    for (int sg = blockIdx.x; sg < batch * kHkv; sg += gridDim.x) {
      if (seg_ptr[sg + 1] != seg_ptr[sg]) continue;
      const int sb = sg / kHkv, sh = sg % kHkv;
      for (int ej = threadIdx.x * 4; ej < q_len * kGroup * kD; ej += 32 * T::kConsumerWarps * 4) {
        const int j = ej / (kGroup * kD), e = ej - j * kGroup * kD;
        store_out4(out, ((static_cast<int64_t>(sb) * q_len + j) * kHq + sh * kGroup) * kD + e, 0.f, 0.f,
                   0.f, 0.f, out_dtype);
      }
    }
  }

  // An item descriptor from the producer's ring (slot n % R), handed back as
  // soon as it is read; false after an abort.
  struct Desc {
    int i;
    Item it;
  };
  auto fetch_desc = [&](uint32_t n, Desc& d) -> bool {
    const int rslot = static_cast<int>(n % R);
    bool ok = !*abort_flag && mbar_wait(smem_u32(&item_full[rslot]), (n / R) & 1, status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) *abort_flag = 1;
      return false;
    }
    const volatile int* slot = ring + rslot * T::kRingInts;
    d.i = slot[0];
    d.it = Item{slot[1], slot[2], slot[3], slot[4], slot[5], slot[5] >= 0};
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&item_empty[rslot]));
    return true;
  };
  if constexpr (kTC) {
    // ---------------------------------------------------- tensor-core form
    // Multi-token decode on the 5th-generation tensor cores.
    // The item's q_len x 8 query rows (row 8 t + head, zeros for t >= q_len)
    // are rows 32 k .. 32 k + 31 of queue k's M = 128 Q tile, so that queue
    // k's softmax warp is the one whose TMEM lanes those rows are (warp w
    // reaches lanes 32 (w % 4) ..): warp 0 for queue 0, warp 5 for queue 1.
    // Per 64-key tile: S = Q K^T (N 64) into one of two score buffers; the
    // softmax warp (thread = row) masks each row at its token's position,
    // keeps a running maximum that moves only when it grows by more than
    // 2^8 (then O is rescaled in TMEM), and writes P as BF16 pairs over the
    // scores; O += P V (N 128, P from TMEM, V MN-major), O in TMEM for the
    // item.  The item's partial (O / l and lse per row) goes to the partial
    // buffers; a merge pass combines the items of every segment.
    uint64_t* tb = full + 2 * SG + 2 * R + 1;   // this queue's tensor-core barriers
    const uint32_t b_sfull = smem_u32(&tb[0]), b_pfull = smem_u32(&tb[2]);
    const uint32_t b_qfull = smem_u32(&tb[4]), b_qfree = smem_u32(&tb[5]);
    const uint32_t b_ofinal = smem_u32(&tb[6]), b_ofree = smem_u32(&tb[7]);
    const uint32_t b_drain = smem_u32(&tb[8]);
    const uint32_t tmem = *tmem_slot;
    const uint32_t tq = tmem + 256u * static_cast<uint32_t>(grp);   // the queue's columns
    uint8_t* qtile = smem + T::kOffQt + grp * T::kQtBytes;
    auto wait_warp = [&](uint32_t bar, uint32_t parity) -> bool {
      bool ok = !*abort_flag && mbar_wait(bar, parity, status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0) *abort_flag = 1;
      return ok;
    };

    if (wq == 2) {
      // ------------------------------------------------ MMA warp of the queue
      constexpr uint32_t kIdescS = kFp8 ? umma_idesc_e4m3(128, 64) : umma_idesc_bf16(128, 64, false);
      constexpr uint32_t kIdescO = kFp8 ? umma_idesc_f16(128, 128, true) : umma_idesc_bf16(128, 128, true);
      constexpr uint64_t kStageStep = T::kStageBytes >> 4;
      // V: the stage's second part (E4M3 pages: after the 8 KB K page of codes)
      constexpr uint32_t kOffV = kFp8 ? T::kPageBytes : T::kF16Page;
      const uint64_t desc_q = umma_smem_desc(smem_u32(qtile), 1024, 1024);
      const uint64_t desc_k = umma_smem_desc(stage_base, 1024, 1024);
      const uint64_t desc_v = umma_smem_desc(stage_base + kOffV, T::kBoxBytes, 1024);
      uint32_t gl = 0, nq = 0;   // tiles and items of the queue so far
      bool stop = false;
      for (uint32_t n = 0; !stop; ++n) {
        Desc d;
        if (!fetch_desc(n, d) || d.i < 0) break;
        if (!d.it.ok) continue;
        const int nt = d.it.t1 - d.it.t0;
        if (!wait_warp(b_qfull, nq & 1)) break;
        tc_fence_after();
        // Issue Q K^T of tile jq once its K is in place (at most two ahead of
        // P V: two score buffers) and P V of tile jp once its P is written,
        // whichever is ready first, so that neither waits on the other's tile.
        int jq = 0, jp = 0;
        unsigned long long idle_since = 0ull;
        while (jp < nt) {
          bool did = false;
          if (jp < jq) {
            const uint32_t gg = g + jp, st = gg % SG, pb = (gl + jp) & 1u;
            bool ready = mbar_test_wait(b_pfull + 8u * pb, ((gl + jp) >> 1) & 1u);
            if (kFp8) ready = ready && mbar_test_wait(smem_u32(&tb[9 + st]), (gg / SG) & 1);
            if (jp == 0 && nq > 0) ready = ready && mbar_test_wait(b_ofree, (nq - 1) & 1);
            if (__all_sync(0xffffffffu, ready)) {
              tc_fence_after();
              umma_pv_lane(tq + 128, tq + 64u * pb, desc_v + st * kStageStep, kIdescO, jp != 0,
                           jp == nt - 1, b_ofinal, smem_u32(&empty[st]));
              ++jp;
              did = true;
            }
          }
          if (jq < nt && jq - jp < 2) {
            const uint32_t gg = g + jq, st = gg % SG;
            // Q K^T reads K as landed (E4M3 codes, or BF16)
            const bool ready = mbar_test_wait(smem_u32(&full[st]), (gg / SG) & 1);
            if (__all_sync(0xffffffffu, ready)) {
              // V rows the products must not see (the cache may hold NaN
              // there): past the length on the sequence's last tile, all of a
              // bad block's (the converter zeroes them for E4M3 pages)
              const int keep = stage_ok[st] ? min(kPage, d.it.len - (d.it.t0 + jq) * kPage) : 0;
              if (!kFp8 && keep < kPage) {
                uint4* v0 = reinterpret_cast<uint4*>(smem + (stage_base - smem_u32(smem)) +
                                                     st * T::kStageBytes + T::kF16Page);
                uint4* v1 = v0 + T::kBoxBytes / 16;
                for (int z = keep * 8 + lane; z < kPage * 8; z += 32) {
                  v0[z] = make_uint4(0u, 0u, 0u, 0u);
                  v1[z] = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
              }
              tc_fence_after();
              if constexpr (kFp8)
                umma_qk_e4m3(tq + 64u * ((gl + jq) & 1u), desc_q, desc_k + st * kStageStep, kIdescS,
                             b_sfull + 8u * ((gl + jq) & 1u), jq == nt - 1, b_qfree, !kQ8,
                             (T::kQtBytes / 2) >> 4);
              else
                umma_qk_tile(tq + 64u * ((gl + jq) & 1u), desc_q, desc_k + st * kStageStep, kIdescS,
                             b_sfull + 8u * ((gl + jq) & 1u), jq == nt - 1, b_qfree);
              ++jq;
              did = true;
            }
          }
          if (did) {
            idle_since = 0ull;
            continue;
          }
          // nothing ready: bounded like every other wait of the kernel
          if (poll_give_up(idle_since, abort_flag, status, kWaitLimitNs)) {
            stop = true;
            break;
          }
        }
        if (stop) break;
        g += nt;
        gl += nt;
        ++nq;
      }
      // every product issued here has completed before TMEM is freed
      umma_commit_elect(b_drain);
      mbar_wait(b_drain, 0, status);
      __syncwarp();
    } else if (wq == grp) {
      // ------------------------------------------------ softmax warp of the queue
      const int rr = lane, row = 32 * grp + rr;   // row of the Q tile = TMEM lane
      const int tok = rr >> 3, hl = rr & 7;
      const uint32_t trow = tq + (static_cast<uint32_t>(32 * grp) << 16);
      uint32_t gl = 0, nq = 0;
      bool stop = false;
      for (uint32_t n = 0; !stop; ++n) {
        Desc d;
        if (!fetch_desc(n, d) || d.i < 0) break;
        const Item it = d.it;
        const bool valid = tok < q_len;
        const int64_t prow = (static_cast<int64_t>(d.i) * q_len + tok) * kGroup + hl;
        // With the output given, a segment of one item is written to it
        // directly (the merge pass after the kernel leaves such segments
        // alone); other items write their partial.
        const bool seg_known = it.seq >= 0 && it.seq < batch && it.h >= 0 && it.h < kHkv;
        const int seg = seg_known ? it.seq * kHkv + it.h : 0;
        const bool direct = fuse && seg_known && seg_ptr[seg + 1] - seg_ptr[seg] == 1;
        const int64_t orow = ((static_cast<int64_t>(it.seq) * q_len + tok) * kHq + it.h * kGroup + hl) * kD;
        if (!it.ok) {   // no products: an empty partial, or zeros
          if (valid) {
            if (direct) {
              for (int e = 0; e < kD; e += 4) store_out4(out, orow + e, 0.f, 0.f, 0.f, 0.f, out_dtype);
            } else {
              for (int e = 0; e < kD; e += 4)
                *reinterpret_cast<float4*>(partial_o + prow * kD + e) = make_float4(0.f, 0.f, 0.f, 0.f);
              partial_lse[prow] = -INFINITY;
            }
          }
          continue;
        }
        const int nt = it.t1 - it.t0;
        // the item's Q rows, once the previous item's last Q K^T has read the tile
        if (nq > 0 && !wait_warp(b_qfree, (nq - 1) & 1)) break;
        // this row's factor from raw scores to log2 units (over E4M3 pages with
        // a BF16 q: divided by the row's power-of-two scale)
        float c_row = scale_log2;
        {
          const int64_t qr = (static_cast<int64_t>(it.seq) * q_len + (valid ? tok : 0)) * kHq +
                             it.h * kGroup + hl;
          if constexpr (!kFp8) {
            // one row: 16 chunks of 8 BF16 values, d 0..63 then 64..127
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
              uint4 v = make_uint4(0u, 0u, 0u, 0u);
              if (valid) v = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(q) + qr * kD)[ch];
              const int half = ch >> 3, c8 = ch & 7;
              *reinterpret_cast<uint4*>(qtile + half * (T::kQtBytes / 2) + (row >> 3) * 1024 +
                                        (row & 7) * 128 + ((c8 ^ (row & 7)) << 4)) = v;
            }
          } else if constexpr (kQ8) {
            // one row of 128 codes: 8 chunks of 16
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              uint4 v = make_uint4(0u, 0u, 0u, 0u);
              if (valid) v = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(q) + qr * kD)[ch];
              *reinterpret_cast<uint4*>(qtile + (row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4)) = v;
            }
          } else {
            // q = 2^-se (hi + lo): hi the row-scaled q rounded to E4M3, lo the
            // remainder rounded to E4M3, exact for every element within 2^10
            // of the row's largest; se puts the row's largest in [2^7, 2^8).
            // Leading terms in the tile's first 8 KB, remainders in its second.
            uint4 w[16];
            float amax = 0.f;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
              w[ch] = valid ? reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(q) + qr * kD)[ch]
                            : make_uint4(0u, 0u, 0u, 0u);
              amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(w[ch].x)), fabsf(bf16_hi(w[ch].x))),
                                       fmaxf(fabsf(bf16_lo(w[ch].y)), fabsf(bf16_hi(w[ch].y)))));
              amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(w[ch].z)), fabsf(bf16_hi(w[ch].z))),
                                       fmaxf(fabsf(bf16_lo(w[ch].w)), fabsf(bf16_hi(w[ch].w)))));
            }
            const int e2 = amax > 0.f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127 : 0;
            const int se = 7 - max(e2, -119);   // in [-120, 126]
            const float sc = __uint_as_float(static_cast<uint32_t>(127 + se) << 23);
            c_row = scale_log2 * __uint_as_float(static_cast<uint32_t>(127 - se) << 23);
            // codes of 4 values (a 32-bit word), leading term and remainder
            auto split4 = [&](uint32_t u0, uint32_t u1, uint32_t& hi, uint32_t& lo) {
              const float a0 = bf16_lo(u0) * sc, a1 = bf16_hi(u0) * sc;
              const float a2 = bf16_lo(u1) * sc, a3 = bf16_hi(u1) * sc;
              const uint16_t h01 = f32x2_to_e4m3x2(a0, a1), h23 = f32x2_to_e4m3x2(a2, a3);
              uint32_t f01 = e4m3x2_to_f16x2(h01), f23 = e4m3x2_to_f16x2(h23);
              const float2 d01 = __half22float2(*reinterpret_cast<__half2*>(&f01));
              const float2 d23 = __half22float2(*reinterpret_cast<__half2*>(&f23));
              const uint16_t l01 = f32x2_to_e4m3x2(a0 - d01.x, a1 - d01.y);
              const uint16_t l23 = f32x2_to_e4m3x2(a2 - d23.x, a3 - d23.y);
              hi = static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16);
              lo = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
            };
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {   // 16 codes: BF16 chunks 2ch, 2ch+1
              uint4 hi, lo;
              split4(w[2 * ch].x, w[2 * ch].y, hi.x, lo.x);
              split4(w[2 * ch].z, w[2 * ch].w, hi.y, lo.y);
              split4(w[2 * ch + 1].x, w[2 * ch + 1].y, hi.z, lo.z);
              split4(w[2 * ch + 1].z, w[2 * ch + 1].w, hi.w, lo.w);
              const int off = (row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4);
              *reinterpret_cast<uint4*>(qtile + off) = hi;
              *reinterpret_cast<uint4*>(qtile + T::kQtBytes / 2 + off) = lo;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_qfull);
        }
        const int pos = it.len - q_len + tok;   // the row's token position
        float m_used = -INFINITY, lsum = 0.f;
        for (int j = 0; j < nt; ++j) {
          const uint32_t gg = g + j, st = gg % SG, b = (gl + j) & 1u;
          if (!wait_warp(b_sfull + 8u * b, ((gl + j) >> 1) & 1u)) {
            stop = true;
            break;
          }
          tc_fence_after();
          uint32_t sr[64];
          tmem_ld64(trow + 64u * b, sr);
          tmem_wait_ld();
          const int key0 = (it.t0 + j) * kPage;
          const int lim = (valid && stage_ok[st]) ? min(kPage - 1, pos - key0) : -1;
          // the mask sets the scores past lim to -inf in place (a copy of
          // the row would cost a move per score on the unmasked tiles)
          if (!__all_sync(0xffffffffu, lim == kPage - 1)) {
#pragma unroll
            for (int k = 0; k < 64; ++k)
              if (k > lim) sr[k] = 0xff800000u;
          }
          auto x = [&](int k) { return __uint_as_float(sr[k]); };
          // the row maximum in 8 independent chains of three-input maxima,
          // each started from a pair; the scale is positive, so it commutes
          // with the maximum
          float m8[8];
#pragma unroll
          for (int k = 0; k < 64; k += 2) {
            const int c = (k >> 1) & 7;
            m8[c] = k < 16 ? fmaxf(x(k), x(k + 1)) : max3f(m8[c], x(k), x(k + 1));
          }
          const float mx =
              max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * c_row;
          // the running maximum moves only when it grows by more than 2^8
          // (weights stay <= 2^8); the row's O is then rescaled in TMEM
          const bool grow = mx > m_used + 8.f;
          const float alpha = grow ? exp2_ftz(m_used - mx) : 1.f;   // 0 while m_used = -inf
          if (grow) {
            lsum *= alpha;
            m_used = mx;
          }
          if (j > 0 && __any_sync(0xffffffffu, grow)) {
            // the previous tile's P V must be in O before it is rescaled: its
            // stage's empty barrier completes with it
            const uint32_t gp = gg - 1;
            if (!wait_warp(smem_u32(&empty[gp % SG]), (gp / SG) & 1)) {
              stop = true;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int qc = 0; qc < 4; ++qc) {
              uint32_t ov[32];
              tmem_ld32(trow + 128 + 32 * qc, ov);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
              tmem_st32(trow + 128 + 32 * qc, ov);
            }
          }
          // p = 2^(s scale - m): one packed FMA per pair and an exponential
          // each; the row sum in 4 independent chains of packed adds
          const float nms = m_used == -INFINITY ? 0.f : -m_used;
          const uint64_t scale2 = f32x2(c_row, c_row), nms2 = f32x2(nms, nms);
          uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};
          uint32_t pk[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            float a0, a1;
            f32x2_split(fma_f32x2(f32x2(x(2 * k), x(2 * k + 1)), scale2, nms2), a0, a1);
            const float p0 = exp2_ftz(a0), p1 = exp2_ftz(a1);
            ps2[k & 3] = add_f32x2(ps2[k & 3], f32x2(p0, p1));
            pk[k] = kFp8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
          }
          float s0, s1;
          f32x2_split(add_f32x2(add_f32x2(ps2[0], ps2[1]), add_f32x2(ps2[2], ps2[3])), s0, s1);
          lsum += s0 + s1;
          tmem_st32(trow + 64u * b, pk);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_pfull + 8u * b);
        }
        if (stop) break;
        // the item's partial once its last P V is done: this row of O
        if (!wait_warp(b_ofinal, nq & 1)) break;
        tc_fence_after();
        const float inv = lsum > 0.f ? v_scale / lsum : 0.f;
#pragma unroll
        for (int qc = 0; qc < 4; ++qc) {
          uint32_t ov[32];
          tmem_ld32(trow + 128 + 32 * qc, ov);
          tmem_wait_ld();
          if (valid && direct) {
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              store_out4(out, orow + 32 * qc + k, __uint_as_float(ov[k]) * inv,
                         __uint_as_float(ov[k + 1]) * inv, __uint_as_float(ov[k + 2]) * inv,
                         __uint_as_float(ov[k + 3]) * inv, out_dtype);
          } else if (valid) {
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              *reinterpret_cast<float4*>(partial_o + prow * kD + 32 * qc + k) =
                  make_float4(__uint_as_float(ov[k]) * inv, __uint_as_float(ov[k + 1]) * inv,
                              __uint_as_float(ov[k + 2]) * inv, __uint_as_float(ov[k + 3]) * inv);
          }
        }
        if (valid && !direct)
          partial_lse[prow] = lsum > 0.f ? (m_used + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_ofree);
        g += nt;
        gl += nt;
        ++nq;
      }
    }
    if constexpr (kFp8) {
      if (wq != 2 && wq != grp) {
        // -------------------------------------------- converter warps of the queue
        // Each landed tile's V page is widened to F16 in its own stage (Q K^T
        // reads the K codes as they landed): thread ct reads raw V row ct and
        // writes F16 row ct, d 0..63 over the raw row itself and d 64..127
        // into the stage's last 8 KB (zeros past the length or on a bad
        // block).  A thread's output shares bytes only with its own raw row,
        // read before, so the widening needs no barrier.
        const int ct = (wq == 3 ? 32 : 0) + lane;
        bool stop = false;
        for (uint32_t n = 0; !stop; ++n) {
          Desc d;
          if (!fetch_desc(n, d) || d.i < 0) break;
          if (!d.it.ok) continue;
          const int nt = d.it.t1 - d.it.t0;
          for (int j = 0; j < nt; ++j) {
            const uint32_t gg = g + j, st = gg % SG;
            if (!wait_warp(smem_u32(&full[st]), (gg / SG) & 1)) {
              stop = true;
              break;
            }
            uint8_t* vst = smem + T::kOffStages + (grp * SG + st) * T::kStageBytes + T::kPageBytes;
            const int keep = stage_ok[st] ? min(kPage, d.it.len - (d.it.t0 + j) * kPage) : 0;
            uint4 vw[8];
            load_e4m3_row(vst + ct * 128, ct, ct < keep, vw);
            store_f16_row(vw, vst + ct * 128, vst + T::kBoxBytes + ct * 128, ct);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tb[9 + st]));
          }
          g += nt;
        }
      }
    }
    // every warp of the CTA meets here; then the allocating warp frees TMEM
    tc_fence_before();
    __syncwarp();
    named_bar_sync(2, T::kThreads);
    if (warp == kTmemWarp) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
    return;
  }

  // The item's q words (this lane's share of the B operand Q^T of the 8 query
  // heads of its KV head, head = r) and, with the merge fused in, its
  // segment's first item and item count.  Issued one item ahead, so the
  // loads are in flight during the previous item's epilogue.
  auto load_item = [&](const Desc& d, uint32_t (&qw)[8][2], int& first, int& count) {
    first = 0;
    count = 0;
    if (d.i < 0 || !d.it.ok) return;
    if (fuse) {
      const int seg = d.it.seq * kHkv + d.it.h;
      first = seg_ptr[seg];
      count = seg_ptr[seg + 1] - first;
    }
    if (qj >= q_len) return;   // a warp of the 4-token layout without a query
    const int64_t qr = (static_cast<int64_t>(d.it.seq) * q_len + qj) * kHq + d.it.h * kGroup + r;
    if constexpr (kQ8) {
      // B operand of m16n8k32 for k-step kp: codes 32kp + 4c .. +3 and 32kp + 16 + 4c .. +3
      const uint8_t* qrow8 = static_cast<const uint8_t*>(q) + qr * kD;
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        qw[kp][0] = *reinterpret_cast<const uint32_t*>(qrow8 + 32 * kp + 4 * c);
        qw[kp][1] = *reinterpret_cast<const uint32_t*>(qrow8 + 32 * kp + 16 + 4 * c);
      }
      return;
    }
    const uint16_t* qrow = static_cast<const uint16_t*>(q) + qr * kD;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      if constexpr (kFp8) {
        const uint2 x = *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c);
        qw[ks][0] = x.x;
        qw[ks][1] = x.y;
      } else {
        qw[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c);
        qw[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * c);
      }
    }
  };

  Desc cur{-1, Item{-1, -1, 0, 0, 0, false}};
  uint32_t qw[8][2];
  int seg_first = 0, seg_items = 0;
  bool have = fetch_desc(0, cur);
  if (have) load_item(cur, qw, seg_first, seg_items);
  for (uint32_t n = 0; have && cur.i >= 0; ++n) {
    const int i = cur.i;
    const Item it = cur.it;

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2c, 2c+1
    float o[8][4];
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) o[mi][0] = o[mi][1] = o[mi][2] = o[mi][3] = 0.f;

    if (it.ok) {
      // B operand Q^T for the 8 query heads of this KV head (head = r)
      uint32_t bq[8][2];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if constexpr (kQ8) {
          bq[ks][0] = qw[ks][0];   // E4M3 codes as they are (entries 4..7 unused)
          bq[ks][1] = qw[ks][1];
        } else if constexpr (kFp8) {
          bq[ks][0] = pack_f16(bf16_lo(qw[ks][0]), bf16_hi(qw[ks][0]));
          bq[ks][1] = pack_f16(bf16_lo(qw[ks][1]), bf16_hi(qw[ks][1]));
        } else {
          bq[ks][0] = qw[ks][0];
          bq[ks][1] = qw[ks][1];
        }
      }

      for (int t = it.t0; t < it.t1; ++t, ++g) {
        if (dead) continue;
        const int s = static_cast<int>(g % SG);
        const uint32_t use = g / SG;
        bool tok = !*abort_flag && mbar_wait(smem_u32(&full[s]), use & 1, status);
        tok = __all_sync(0xffffffffu, tok);
        if (!tok) {
          if (lane == 0) *abort_flag = 1;
          dead = true;
          continue;
        }
        // keys this warp's query sees in the tile, counted from its first token:
        // new token qj sits at position len - q_len + qj and sees keys up to it
        const int nvalid = (it.len - (q_len - 1 - qj)) - t * kPage - tok0;
        if (stage_ok[s] && nvalid > 0) {
          const uint32_t kb = stage_base + s * T::kStageBytes;
          const uint32_t vb = kb + T::kPageBytes;

          // S^T = K Q^T per 16-token block (rows: tokens, cols: 8 heads); two chains
          // fragment: x[0] = S[tok r][head 2c], x[1] = [r][2c+1], x[2] = [r+8][2c], x[3] = [r+8][2c+1]
          float x[kMB][4];
#pragma unroll
          for (int mb = 0; mb < kMB; ++mb) {
            const int rowb = row + 16 * mb;
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (kQ8) {
              // the ldmatrix words of a 16-token x 32-byte slab are the m16n8k32
              // A fragments of the codes themselves: no conversion
#pragma unroll
              for (int kp = 0; kp < 4; ++kp) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kb + rowb * 128 + ((((2 * kp + hi) & 7) ^ sw) << 4), r0, r1, r2, r3);
                if (kp & 1) mma_e4m3(sb, r0, r1, r2, r3, bq[kp][0], bq[kp][1]);
                else        mma_e4m3(sa, r0, r1, r2, r3, bq[kp][0], bq[kp][1]);
              }
            } else if constexpr (kFp8) {
#pragma unroll
              for (int kp = 0; kp < 4; ++kp) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kb + rowb * 128 + ((((2 * kp + hi) & 7) ^ sw) << 4), r0, r1, r2, r3);
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
                ldsm_x4(kb + (ks >> 2) * T::kBoxBytes + rowb * 128 + ((((2 * ks + hi) & 7) ^ sw) << 4),
                        a0, a1, a2, a3);
                if (ks & 1) mma_bf16(sb, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
                else        mma_bf16(sa, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
              }
            }
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) x[mb][k4] = (sa[k4] + sb[k4]) * scale_log2;
          }
          // keys past the query's last visible one: p = 0, V entries zeroed
#pragma unroll
          for (int mb = 0; mb < kMB; ++mb) {
            const int nv = nvalid - 16 * mb;
            if (nv < 16) {
              if (r >= nv) x[mb][0] = x[mb][1] = -INFINITY;
              if (r + 8 >= nv) x[mb][2] = x[mb][3] = -INFINITY;
            }
          }
          float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
          for (int mb = 0; mb < kMB; ++mb) {
            mt0 = fmaxf(mt0, fmaxf(x[mb][0], x[mb][2]));
            mt1 = fmaxf(mt1, fmaxf(x[mb][1], x[mb][3]));
          }
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, off));
            mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, off));
          }
          const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
          const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
          const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = exp2_ftz(m0 - ms0), al1 = exp2_ftz(m1 - ms1);
          float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
          for (int mb = 0; mb < kMB; ++mb) {
            x[mb][0] = exp2_ftz(x[mb][0] - ms0);   // from here on x holds p
            x[mb][1] = exp2_ftz(x[mb][1] - ms1);
            x[mb][2] = exp2_ftz(x[mb][2] - ms0);
            x[mb][3] = exp2_ftz(x[mb][3] - ms1);
            ps0 += x[mb][0] + x[mb][2];
            ps1 += x[mb][1] + x[mb][3];
          }
          l0 = l0 * al0 + ps0;
          l1 = l1 * al1 + ps1;
          m0 = mn0;
          m1 = mn1;
          // the running max rarely moves after the first tiles: skip the
          // (exact, multiply-by-one) rescale when no lane needs it
          if (!__all_sync(0xffffffffu, al0 == 1.f && al1 == 1.f)) {
#pragma unroll
            for (int mi = 0; mi < 8; ++mi) {
              o[mi][0] *= al0;
              o[mi][1] *= al1;
              o[mi][2] *= al0;
              o[mi][3] *= al1;
            }
          }
          // P^T fragments -> B operands (k = token, n = head) by 8x8
          // transposes, all blocks first (the scores are then dead)
          uint32_t pb[kMB][2];
#pragma unroll
          for (int mb = 0; mb < kMB; ++mb) {
            if constexpr (kFp8) {
              pb[mb][0] = movmatrix_t(pack_f16(x[mb][0], x[mb][1]));
              pb[mb][1] = movmatrix_t(pack_f16(x[mb][2], x[mb][3]));
            } else {
              pb[mb][0] = movmatrix_t(pack_bf16(x[mb][0], x[mb][1]));
              pb[mb][1] = movmatrix_t(pack_bf16(x[mb][2], x[mb][3]));
            }
          }
#pragma unroll
          for (int mb = 0; mb < kMB; ++mb) {
            const int nv = nvalid - 16 * mb;   // V rows of tokens past it are zeroed
            if (nv < 16) {
              const uint32_t m01 = (2 * c < nv ? 0x0000ffffu : 0u) | (2 * c + 1 < nv ? 0xffff0000u : 0u);
              const uint32_t m23 = (2 * c + 8 < nv ? 0x0000ffffu : 0u) | (2 * c + 9 < nv ? 0xffff0000u : 0u);
              pv_tile<kFp8, true>(vb, row + 16 * mb, vtok_bf16 + 16 * mb, vsel_bf16, hi, sw, pb[mb][0],
                                  pb[mb][1], m01, m23, o);
            } else {
              pv_tile<kFp8, false>(vb, row + 16 * mb, vtok_bf16 + 16 * mb, vsel_bf16, hi, sw,
                                   pb[mb][0], pb[mb][1], 0xffffffffu, 0xffffffffu, o);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      }
    }
    if (dead) break;

    // the next item's descriptor, q words and segment bounds: their loads
    // overlap this item's epilogue
    Desc nxt{-1, Item{-1, -1, 0, 0, 0, false}};
    uint32_t qw_next[8][2];
    int next_first = 0, next_items = 0;
    have = fetch_desc(n + 1, nxt);
    if (!have) break;
    load_item(nxt, qw_next, next_first, next_items);

    // ---- merge the warps' states and write the item's partial: every warp
    // stores its raw (m, l, O) in its own slice; after one barrier each
    // output element is combined over the warps in a fixed order (the result
    // is bit-reproducible) with the log-sum-exp weights of its head
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
    {
      float* o_h0 = sm_o + (warp * kGroup + 2 * c) * T::kOStride;
      float* o_h1 = o_h0 + T::kOStride;
#pragma unroll
      for (int mi = 0; mi < 8; ++mi) {
        // rows of the O^T fragment: d_a for o[mi][0..1], d_b for o[mi][2..3]
        const int d_a = kFp8 ? 16 * mi + 2 * r : 16 * mi + r;
        const int d_b = kFp8 ? d_a + 1 : d_a + 8;
        o_h0[d_a] = o[mi][0];
        o_h1[d_a] = o[mi][1];
        o_h0[d_b] = o[mi][2];
        o_h1[d_b] = o[mi][3];
      }
    }
    if (!cons_sync()) break;
    // with the merge fused in: a segment of one item is final here; a segment
    // of several items is merged by the queue that finishes its last item.
    // Output row of query j, head hh of segment (seq, h): (seq*q_len + j)*64 + 8h + hh;
    // partial row of item i: (i*q_len + j)*8 + hh.
    const int seg = it.seq * kHkv + it.h;
    const bool direct = fuse && it.ok && seg_items == 1;
    const int w0 = grp * T::kWarpsPerGroup;   // the queue's first consumer warp
    {
      constexpr int kItemOut = kQ * kGroup * kD;   // outputs of an item over the layout's queries
#pragma unroll
      for (int ej = gt * 4; ej < kItemOut; ej += T::kGroupThreads * 4) {
        const int j = ej / (kGroup * kD);          // query of these 4 outputs
        if (j >= q_len) break;
        const int e = ej - j * kGroup * kD;
        const int hh = e >> 7;                     // head of these 4 outputs
        const int wa = w0 + j * kWq;               // the query's warps: wa .. wa + kWq - 1
        float* dst = partial_o + (static_cast<int64_t>(i) * q_len + j) * kGroup * kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = wa; w < wa + kWq; ++w) M = fmaxf(M, sm_m[w * kGroup + hh]);
        const float Ms = M == -INFINITY ? 0.f : M;
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = wa; w < wa + kWq; ++w) {
          const float wt = exp2_ftz(sm_m[w * kGroup + hh] - Ms);
          L += wt * sm_l[w * kGroup + hh];
          const float4 x =
              *reinterpret_cast<const float4*>(sm_o + (w * kGroup + hh) * T::kOStride + (e & 127));
          acc.x += wt * x.x;
          acc.y += wt * x.y;
          acc.z += wt * x.z;
          acc.w += wt * x.w;
        }
        const float inv = L > 0.f ? v_scale / L : 0.f;
        if (direct) {
          store_out4(out, ((static_cast<int64_t>(it.seq) * q_len + j) * kHq + it.h * kGroup) * kD + e,
                     acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv, out_dtype);
        } else {
          *reinterpret_cast<float4*>(dst + e) =
              make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          if ((e & 127) == 0)
            partial_lse[(static_cast<int64_t>(i) * q_len + j) * kGroup + hh] =
                L > 0.f ? (Ms + log2f(L)) * 0.6931471805599453f : -INFINITY;
        }
      }
    }
    if (fuse && it.ok && !direct) {
      if (!cons_sync()) break;     // every thread's share of the partial is written
      if (gt == 0) {
        // release: the queue's partial (ordered before by the barrier) is
        // visible device-wide before the count; acquire: the last arrival
        // sees every other item's partial
        const int done = atomic_add_acq_rel_gpu(&seg_done[seg], 1);
        *merge_flag = done == seg_items - 1;
        if (done == seg_items - 1) seg_done[seg] = 0;   // reset for the next run of this plan
      }
      if (!cons_sync()) break;
      if (*merge_flag) {
        // the last item of the segment: merge its partials.  The lse values
        // are staged in shared memory (the queue's merge slices are free now)
        // by one parallel load, so the per-thread loop is a single pass of
        // independent float4 loads through L2; segments of more than
        // kMergeChunk items are taken chunk by chunk with an online rescale.
        // With no next item the queue's stages hold nothing more, and the
        // partials land there too, by cp.async (no registers held while in
        // flight): a chunk of up to ring_items items is one round through L2
        // instead of a few, which matters most for the merges of long
        // segments, run after their queues' last items at the launch's end.
        // Not in the 2-token layout over E4M3 pages, whose 128 registers
        // would then spill in the streaming loop.
        constexpr bool kRingMerge = !(kFp8 && kQ == 2);
        constexpr int kMergeChunk = 512 / kQ;
        constexpr int kOuts = kQ * kGroup * kD / (4 * T::kGroupThreads);   // float4 outputs per thread
        static_assert(kMergeChunk * kQ * kGroup <= T::kWarpsPerGroup * kGroup * T::kOStride,
                      "the lse staging area must fit in the queue's merge slices");
        static_assert(kOuts * 4 * T::kGroupThreads == kQ * kGroup * kD, "outputs split evenly");
        float* lse_s = sm_o + w0 * kGroup * T::kOStride;
        const int i0 = seg_first;
        const int rows = q_len * kGroup;          // lse values per item
        const int item_floats = q_len * kGroup * kD;
        const int ring_items = kRingMerge && nxt.i < 0 ? SG * T::kStageBytes / (item_floats * 4) : 0;
        const int chunk = ring_items > 0 ? min(ring_items, kMergeChunk) : kMergeChunk;
        const float* ring_o = reinterpret_cast<const float*>(smem + T::kOffStages +
                                                             grp * SG * T::kStageBytes);
        float M[kOuts], W[kOuts];
        float4 acc[kOuts];
#pragma unroll
        for (int u = 0; u < kOuts; ++u) {
          M[u] = -INFINITY;
          W[u] = 0.f;
          acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        bool synced = true;
        for (int base = 0; base < seg_items && synced; base += chunk) {
          const int m = min(chunk, seg_items - base);
          if (kRingMerge && ring_items > 0) {
            const float* lsrc = partial_lse + static_cast<int64_t>(i0 + base) * rows;
            for (int x = gt; x < m * rows / 4; x += T::kGroupThreads)
              cp_async16_cg(smem_u32(lse_s) + 16 * x, lsrc + 4 * x);
            const float* psrc = partial_o + static_cast<int64_t>(i0 + base) * item_floats;
            for (int x = gt; x < m * item_floats / 4; x += T::kGroupThreads)
              cp_async16_cg(stage_base + 16 * x, psrc + 4 * x);
            cp_async_wait_all();
          } else {
            for (int x = gt; x < m * rows; x += T::kGroupThreads)
              lse_s[x] = __ldcg(partial_lse + static_cast<int64_t>(i0 + base) * rows + x);
          }
          if (!(synced = cons_sync())) break;
#pragma unroll
          for (int u = 0; u < kOuts; ++u) {
            const int ej = (gt + u * T::kGroupThreads) * 4;
            const int j = ej / (kGroup * kD);
            if (j >= q_len) continue;
            const int e = ej - j * kGroup * kD;
            const int row_l = j * kGroup + (e >> 7);   // lse row within an item
            float Mn = M[u];
            for (int k = 0; k < m; ++k) Mn = fmaxf(Mn, lse_s[k * rows + row_l]);
            if (Mn != -INFINITY) {
              const float sc = __expf(M[u] - Mn);   // 0 while M is still -inf
              acc[u].x *= sc; acc[u].y *= sc; acc[u].z *= sc; acc[u].w *= sc;
              W[u] *= sc;
              if (kRingMerge && ring_items > 0) {
                const float* ro = ring_o + j * kGroup * kD + e;
#pragma unroll 8
                for (int k = 0; k < m; ++k) {
                  const float w = __expf(lse_s[k * rows + row_l] - Mn);
                  const float4 x = *reinterpret_cast<const float4*>(ro + k * item_floats);
                  acc[u].x += w * x.x;
                  acc[u].y += w * x.y;
                  acc[u].z += w * x.z;
                  acc[u].w += w * x.w;
                  W[u] += w;
                }
              } else {
                const float* po =
                    partial_o + (static_cast<int64_t>(i0 + base) * q_len + j) * kGroup * kD + e;
#pragma unroll 8
                for (int k = 0; k < m; ++k) {
                  const float w = __expf(lse_s[k * rows + row_l] - Mn);
                  const float4 x = __ldcg(
                      reinterpret_cast<const float4*>(po + static_cast<int64_t>(k) * q_len * kGroup * kD));
                  acc[u].x += w * x.x;
                  acc[u].y += w * x.y;
                  acc[u].z += w * x.z;
                  acc[u].w += w * x.w;
                  W[u] += w;
                }
              }
              M[u] = Mn;
            }
          }
          synced = cons_sync();   // before the staging area is overwritten
        }
        if (!synced) break;
#pragma unroll
        for (int u = 0; u < kOuts; ++u) {
          const int ej = (gt + u * T::kGroupThreads) * 4;
          const int j = ej / (kGroup * kD);
          if (j >= q_len) continue;
          const int e = ej - j * kGroup * kD;
          const float inv = W[u] > 0.f ? 1.f / W[u] : 0.f;
          store_out4(out, ((static_cast<int64_t>(it.seq) * q_len + j) * kHq + it.h * kGroup) * kD + e,
                     acc[u].x * inv, acc[u].y * inv, acc[u].z * inv, acc[u].w * inv, out_dtype);
        }
      }
    }
    if (!cons_sync()) break;
    cur = nxt;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qw[ks][0] = qw_next[ks][0];
      qw[ks][1] = qw_next[ks][1];
    }
    seg_first = next_first;
    seg_items = next_items;
  }
  if (cta_clock != nullptr) {
    named_bar_sync(1, 32 * T::kConsumerWarps);   // every queue of the CTA is done
    if (threadIdx.x == 0) record_cta_clock(cta_clock, t_start);
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

template <bool kFp8, int kQ, bool kQ8, bool kTC = false>
cudaError_t ensure_smem_attr() {
  // once per device: the dynamic shared memory opt-in is a per-device setting
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(decode_attn_kernel<kFp8, kQ, kQ8, kTC>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           AttnTraits<kFp8, kTC>::kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

template <bool kFp8, int kQ, bool kQ8, bool kTC = false>
int launch_attn(const void* q, const void* kv_cache, const float* kv_scale, int32_t num_blocks,
                const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                int32_t batch, const hpc_attn_options& opts, const hpc_plan* plan,
                float* partial_o, float* partial_lse, float sm_scale, int32_t* status,
                unsigned long long* cta_clock, void* out, bool pdl, cudaStream_t stream) {
  using T = AttnTraits<kFp8, kTC>;
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return HPC_ERR_CUDA;
  if (ensure_smem_attr<kFp8, kQ, kQ8, kTC>() != cudaSuccess) return HPC_ERR_CUDA;
  // the tensor-core form writes single-item segments to the output and the
  // other items' partials; the merge pass after it combines the latter
  void* fused_out = out;
  if (kTC && cta_clock != nullptr) return HPC_ERR_UNSUPPORTED;
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((plan->num_ctas + T::kGroups - 1) / T::kGroups);   // kGroups queues per CTA
  cfg.blockDim = dim3(T::kThreads);
  cfg.dynamicSmemBytes = T::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, decode_attn_kernel<kFp8, kQ, kQ8, kTC>, map, q, opts.q_scale, kv_scale, block_table,
      max_blocks, num_blocks, seq_lens, batch, opts.q_len,
      static_cast<const hpc_work_item*>(plan->items),
      static_cast<const int32_t*>(plan->cta_ptr), static_cast<const int32_t*>(plan->home_end),
      plan->pool, plan->capacity, plan->num_ctas, partial_o, partial_lse, sm_scale, status, cta_clock,
      static_cast<const int32_t*>(plan->seg_ptr), plan->seg_done, fused_out, opts.out_dtype,
      pdl ? T::kL2PrefetchTiles : 0);
  if (e != cudaSuccess) return HPC_ERR_CUDA;
  if (kTC && out != nullptr)
    return launch_merge(partial_o, partial_lse, plan, batch, &opts, out, true, stream);
  return HPC_OK;
}

// The kernel instances of one query layout: BF16 cache, E4M3 cache with a
// BF16 q, E4M3 cache with an E4M3 q.
template <int kQ>
int launch_attn_layout(const void* q, const void* kv_cache, int32_t kv_dtype, const float* kv_scale,
                       int32_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                       const int32_t* seq_lens, int32_t batch, const hpc_attn_options& opts,
                       const hpc_plan* plan, float* partial_o, float* partial_lse, float sm_scale,
                       int32_t* status, unsigned long long* cta_clock, void* out, bool pdl,
                       cudaStream_t stream) {
  if (kv_dtype == HPC_KV_BF16) {
    if constexpr (kQ == 4)
      return launch_attn<false, kQ, false, true>(q, kv_cache, kv_scale, num_blocks, block_table,
                                                 max_blocks, seq_lens, batch, opts, plan,
                                                 partial_o, partial_lse, sm_scale, status,
                                                 cta_clock, out, pdl, stream);
    return launch_attn<false, kQ, false>(q, kv_cache, kv_scale, num_blocks, block_table, max_blocks,
                                         seq_lens, batch, opts, plan, partial_o, partial_lse,
                                         sm_scale, status, cta_clock, out, pdl, stream);
  }
  if constexpr (kQ == 4) {
    if (opts.q_dtype == HPC_Q_FP8_E4M3)
      return launch_attn<true, kQ, true, true>(q, kv_cache, kv_scale, num_blocks, block_table,
                                               max_blocks, seq_lens, batch, opts, plan, partial_o,
                                               partial_lse, sm_scale, status, cta_clock, out, pdl,
                                               stream);
    return launch_attn<true, kQ, false, true>(q, kv_cache, kv_scale, num_blocks, block_table,
                                              max_blocks, seq_lens, batch, opts, plan, partial_o,
                                              partial_lse, sm_scale, status, cta_clock, out, pdl,
                                              stream);
  }
  if (opts.q_dtype == HPC_Q_FP8_E4M3)
    return launch_attn<true, kQ, true>(q, kv_cache, kv_scale, num_blocks, block_table, max_blocks,
                                       seq_lens, batch, opts, plan, partial_o, partial_lse,
                                       sm_scale, status, cta_clock, out, pdl, stream);
  return launch_attn<true, kQ, false>(q, kv_cache, kv_scale, num_blocks, block_table, max_blocks,
                                      seq_lens, batch, opts, plan, partial_o, partial_lse, sm_scale,
                                      status, cta_clock, out, pdl, stream);
}

// The checks every attention entry point makes before launching.
inline int check_attn_args(const void* q, const void* kv_cache, int32_t kv_dtype,
                           const float* kv_scale, int32_t num_blocks, const int32_t* block_table,
                           int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                           const hpc_plan* plan, const float* partial_o, const float* partial_lse,
                           const int32_t* status, const void* out) {
  HPC_CHECK_ARG(q && kv_cache && block_table && seq_lens && plan && partial_o && partial_lse &&
                status && plan->items && plan->cta_ptr && plan->home_end && plan->pool);
  HPC_CHECK_ARG(num_blocks > 0 && max_blocks >= 1 && batch >= 0 && plan->num_ctas >= 1 &&
                plan->capacity >= 0);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(kv_cache) & 15) == 0);
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(plan->items) & 15) == 0);
  // partials are written and read 16 bytes at a time
  HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(partial_o) & 15) == 0 &&
                (reinterpret_cast<uintptr_t>(partial_lse) & 15) == 0);
  if (out != nullptr) HPC_CHECK_ARG(plan->seg_ptr && plan->seg_done);
  if (kv_dtype == HPC_KV_FP8_E4M3) HPC_CHECK_ARG(kv_scale != nullptr);
  else if (kv_dtype != HPC_KV_BF16) return HPC_ERR_UNSUPPORTED;
  if (num_blocks > HPC_MAX_NUM_BLOCKS) return HPC_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks) * kPage >= (int64_t{1} << 31)) return HPC_ERR_UNSUPPORTED;
  return HPC_OK;
}

// The checks of the attention options.
inline int check_attn_options(const hpc_attn_options& o, int32_t kv_dtype, const void* out) {
  HPC_CHECK_ARG(o.q_len >= 1 && o.q_len <= HPC_MAX_Q_LEN);
  if (o.q_dtype != HPC_Q_BF16 && o.q_dtype != HPC_Q_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
  if (o.q_dtype == HPC_Q_FP8_E4M3) {
    if (kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
    HPC_CHECK_ARG(o.q_scale > 0.0f && o.q_scale < 3.0e38f);
  }
  if (o.out_dtype != HPC_OUT_BF16 && o.out_dtype != HPC_OUT_FP16 && o.out_dtype != HPC_OUT_FP32)
    return HPC_ERR_UNSUPPORTED;
  if (out != nullptr)
    HPC_CHECK_ARG((reinterpret_cast<uintptr_t>(out) & (o.out_dtype == HPC_OUT_FP32 ? 15 : 7)) == 0);
  return HPC_OK;
}

}  // namespace
}  // namespace hpc

