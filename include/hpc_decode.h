/*
 * hpc_decode.h -- C ABI of the GB300 (sm_103a) paged GQA decode step.
 *
 * One decode step of an attention layer with 64 query heads, 8 KV heads and
 * head_dim 128 over a paged KV cache of 64-token blocks, in four calls:
 *
 *   1. hpc_rope_norm_kvwrite  fused prologue: RoPE -> per-head QK RMSNorm ->
 *                             BF16 q output + K/V write into the paged cache
 *   2. hpc_decode_plan        per-step split-KV plan dealing 64-token tiles to
 *                             CTAs in proportion to each sequence's length
 *   3. hpc_decode_attn        split-KV paged GQA decode attention -> partials
 *   4. hpc_merge              log-sum-exp merge of the partials -> BF16 output
 *
 * Sources: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
 * Hopper" (24-ai.news, 2026-07-06), intro of "Two new HPC backends in the vLLM
 * ecosystem" (model shape) and "Why does dynamic scheduling matter for
 * attention?" (static split-KV, the per-step length-proportional scheduler of
 * 64-token tiles, the fused RoPE / QK-Norm / KV-write prologue, BF16 and FP8);
 * page "[vllm] Introducing the HPC-Ops attention backend" (analysis of vLLM PR
 * #46020), "Code analysis" section 2 (a fused custom op that writes into a
 * caller-provided output and enters CUDA directly, which keeps it usable
 * inside CUDA graphs).
 *
 * Conventions for every call below:
 *   - Pointers marked (device) are device pointers; the caller owns all
 *     memory.  The library never allocates, frees or synchronises; every call
 *     enqueues its kernel(s) on `stream` and returns.  Kernel arguments are
 *     passed by value, so the calls can be captured in a CUDA graph, provided
 *     one call of each kind was made on the device before capture (the first
 *     call sets a kernel attribute and resolves a driver entry point).
 *   - Tensors are dense row-major with the shapes given.  "bf16" buffers hold
 *     IEEE bfloat16 bit patterns (uint16); "e4m3" buffers hold OCP FP8 E4M3
 *     codes (uint8).
 *   - The return value reports host-side argument checks and launch errors
 *     only: HPC_OK, HPC_ERR_INVALID_ARG (null pointer, negative or
 *     inconsistent size), HPC_ERR_UNSUPPORTED (a size beyond a stated limit,
 *     an unknown dtype), HPC_ERR_CUDA (a CUDA runtime error at launch; the
 *     error is left for cudaGetLastError to report).
 *   - Bad indices found on the device (a block id, a slot, a position, a
 *     length out of range, a plan that does not fit its buffers) never trap:
 *     the kernel ORs a HPC_STATUS_* bit into *status (device int32, zeroed by
 *     the caller), skips the offending item, and the step completes.
 */
#ifndef HPC_DECODE_H
#define HPC_DECODE_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HPC_NUM_Q_HEADS 64
#define HPC_NUM_KV_HEADS 8
#define HPC_HEAD_DIM 128
#define HPC_PAGE_TOKENS 64
#define HPC_MAX_BATCH 8192          /* planner limit on the batch size */
#define HPC_MAX_PLAN_CTAS 16384     /* length-proportional planner limit on num_ctas */
#define HPC_MAX_Q_LEN 4             /* new tokens per sequence in multi-token decode */
#define HPC_MAX_NUM_BLOCKS 2097151  /* cache blocks addressable by the TMA map */

typedef enum { HPC_KV_BF16 = 0, HPC_KV_FP8_E4M3 = 1 } hpc_kv_dtype;

/* Type of the attention query q: BF16, or E4M3 codes of q / q_scale (the
 * prologue quantises it; only with an FP8-E4M3 cache, whose products with it
 * run as E4M3 x E4M3 tensor-core products). */
typedef enum { HPC_Q_BF16 = 0, HPC_Q_FP8_E4M3 = 1 } hpc_q_dtype;

/* Type of the attention output, chosen by the caller. */
typedef enum { HPC_OUT_BF16 = 0, HPC_OUT_FP16 = 1, HPC_OUT_FP32 = 2 } hpc_out_dtype;

/* Options of the _ex attention calls; NULL means the single-token BF16 form
 * ({1, HPC_Q_BF16, 1.0f, HPC_OUT_BF16}). */
typedef struct {
  int32_t q_len;      /* new tokens per sequence, 1 .. HPC_MAX_Q_LEN */
  int32_t q_dtype;    /* hpc_q_dtype */
  float q_scale;      /* dequantisation scale of an E4M3 q (q = code * q_scale) */
  int32_t out_dtype;  /* hpc_out_dtype */
} hpc_attn_options;

enum {
  HPC_OK = 0,
  HPC_ERR_INVALID_ARG = -1,
  HPC_ERR_UNSUPPORTED = -2,
  HPC_ERR_CUDA = -3
};

/* Bits a kernel ORs into *status. */
enum {
  HPC_STATUS_BAD_BLOCK = 1,      /* block_table entry outside [0, num_blocks) */
  HPC_STATUS_BAD_SLOT = 2,       /* slot_mapping entry >= num_blocks * 64 */
  HPC_STATUS_BAD_SEQ_LEN = 4,    /* seq_len < 0 or > max_blocks * 64 */
  HPC_STATUS_BAD_POSITION = 8,   /* position outside [0, max_pos) */
  HPC_STATUS_PLAN_OVERFLOW = 16, /* the plan needs more items than capacity */
  HPC_STATUS_WAIT_TIMEOUT = 32,  /* a pipeline wait ran out its time limit */
  HPC_STATUS_BAD_PLAN = 64       /* a work item that does not fit the batch */
};

/* One work item: KV head `kv_head` of sequence `seq`, 64-token tiles
 * [tile_begin, tile_end) (tile t holds tokens 64t .. 64t+63). */
typedef struct {
  int32_t seq;
  int32_t kv_head;
  int32_t tile_begin;
  int32_t tile_end;
} hpc_work_item;

/* A split-KV plan.  The struct itself lives in host memory; its arrays are
 * device buffers owned by the caller:
 *   items    [capacity]        work items in flat (seq, kv_head, tile) order:
 *                              the items of one (seq, kv_head) segment are
 *                              contiguous
 *   cta_ptr  [num_ctas + 1]    CTA c's range holds items cta_ptr[c] ..
 *                              cta_ptr[c+1]-1
 *   home_end [num_ctas]        CTA c runs items cta_ptr[c] .. home_end[c]-1
 *                              itself; the rest of its range is pooled
 *   pool     [3 + capacity]    pool[0]: next claim, pool[1]: CTAs done
 *                              claiming (both zeroed by the planner and reset
 *                              by the attention kernel's last CTA, so a plan
 *                              can be run again), pool[2]: pool length,
 *                              pool[3..]: pooled item indices in claim order;
 *                              a CTA that has finished its home items claims
 *                              the next one
 *   seg_ptr  [batch * 8 + 1]   segment s = seq*8 + kv_head owns items
 *                              seg_ptr[s] .. seg_ptr[s+1]-1
 *   seg_done [batch * 8]       per-segment count of finished items, used by
 *                              hpc_decode_attn_merge (zeroed by the planner,
 *                              left at zero by every run)
 * num_ctas is the number of work queues ("CTA ranges") the plan deals to.
 * hpc_decode_attn runs each queue on one group of 4 consumer warps fed by its
 * own producer warp; a CTA hosts 2 queues (BF16) or 3 (FP8; 2 when q_len is 3
 * or 4), so the grid is ceil(num_ctas / queues per CTA) CTAs.  For the
 * length-proportional plan use hpc_decode_num_ctas() (q_len 1) or
 * hpc_decode_num_queues() (SMs x queues per CTA).  Any num_ctas >= 1 runs
 * correctly; another count than these leaves SMs idle or runs in waves.  A
 * length-proportional plan with J pool chunks needs
 * capacity >= num_ctas * (1 + J) + 8 * batch (hpc_plan_capacity).
 * items must be 16-byte aligned. */
typedef struct {
  hpc_work_item* items;
  int32_t* cta_ptr;
  int32_t* seg_ptr;
  int32_t* home_end;
  int32_t* pool;
  int32_t* seg_done;
  int32_t capacity;
  int32_t num_ctas;
} hpc_plan;

/* Knobs of the length-proportional planner (hpc_decode_plan):
 *   min_tiles       lower bound of the per-CTA quota q (>= 1)
 *   pool_chunks     J: pooled tail chunks per CTA range, 0..64 (0 = no pool)
 *   pool_min_tiles  shortest pooled chunk worth dealing at run time, in
 *                   tiles (>= 1); shorter chunks mean no pool
 * A NULL params pointer means {1, HPC_DEFAULT_POOL_CHUNKS,
 * HPC_DEFAULT_POOL_MIN_TILES}. */
typedef struct {
  int32_t min_tiles;
  int32_t pool_chunks;
  int32_t pool_min_tiles;
} hpc_plan_params;
#define HPC_DEFAULT_POOL_CHUNKS 4
#define HPC_DEFAULT_POOL_MIN_TILES 16

/* Fill the RoPE table cos_sin[pos][i] = cos(pos * theta^(-2i/128)) for
 * i < 64 and cos_sin[pos][64 + i] = sin(same angle), pos in [0, max_pos).
 * The angle and its sine and cosine are formed in float64 and rounded to
 * float32.
 *   cos_sin  (device) float32 [max_pos, 128], written.
 * Errors: HPC_ERR_INVALID_ARG if cos_sin is null, max_pos <= 0 or theta <= 0. */
int hpc_rope_cos_sin_cache(double theta, int32_t max_pos, float* cos_sin, cudaStream_t stream);

/* Fused prologue, one pass per sequence b in [0, batch).
 * Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
 * Hopper", section "Why does dynamic scheduling matter for attention?" (RoPE
 * rotation, QK-Norm and the KV write in one kernel pass, in that order), and
 * page "[vllm] Introducing the HPC-Ops attention backend", "Code analysis"
 * item 2 (the fused RoPE + QK-Norm + KV-cache-write op that writes into a
 * caller-provided output).
 *   q'  = RMSNorm(RoPE(q[b], positions[b]), q_norm_w)   for each of 64 heads
 *   k'  = RMSNorm(RoPE(k[b], positions[b]), k_norm_w)   for each of 8 heads
 *   q_out[b] = bf16(q')                  (round to nearest even)
 *   cache K/V at slot_mapping[b] = k', v[b]  (bf16 RNE, or e4m3 of x / scale,
 *                                        round to nearest even, saturating)
 * RoPE is the NeoX half rotation: element i pairs with i + 64 and turns by the
 * table angle of cos_sin[positions[b]].  RMSNorm: x / sqrt(mean(x^2) + eps) * w,
 * in float32.  v gets neither RoPE nor the norm.
 *   q             (device) bf16 [batch, 64, 128]
 *   k, v          (device) bf16 [batch, 8, 128]
 *   positions     (device) int32 [batch]
 *   cos_sin       (device) float32 [max_pos, 128] (hpc_rope_cos_sin_cache)
 *   q_norm_w, k_norm_w (device) bf16 [128]
 *   kv_cache      (device) [num_blocks][2 (K, V)][8][64][128] of bf16 or e4m3;
 *                 only the slots named by slot_mapping are written
 *   slot_mapping  (device) int64 [batch]; slot = block * 64 + offset; a
 *                 negative slot skips the cache write of that sequence
 *   kv_scale      (device) float32 [2] = {k_scale, v_scale}; required for
 *                 e4m3, ignored (may be NULL) for bf16
 *   q_out         (device) bf16 [batch, 64, 128]; may alias q
 *   status        (device) int32; BAD_POSITION skips the sequence entirely,
 *                 BAD_SLOT skips its cache write
 * The batch is a list of independent tokens: for multi-token decode and
 * prefill pass every new token with its own position and slot.
 * Errors: HPC_ERR_INVALID_ARG for a null required pointer, batch < 0,
 * max_pos <= 0 or num_blocks <= 0; HPC_ERR_UNSUPPORTED for an unknown dtype. */
int hpc_rope_norm_kvwrite(const void* q, const void* k, const void* v,
                          const int32_t* positions, const float* cos_sin, int32_t max_pos,
                          const void* q_norm_w, const void* k_norm_w, float eps,
                          void* kv_cache, int32_t kv_dtype, int32_t num_blocks,
                          const int64_t* slot_mapping, const float* kv_scale,
                          void* q_out, int32_t batch, int32_t* status, cudaStream_t stream);

/* Length-proportional split-KV plan (one CTA, on the device).
 * Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
 * Hopper", section "Why does dynamic scheduling matter for attention?": a
 * static split-KV schedule leaves compute units idle on mixed lengths; the
 * backend's scheduler deals 64-token KV tiles at every step in proportion to
 * each sequence's current length.
 * With n_b = ceil(seq_lens[b] / 64) tiles per (b, kv_head) and
 * T = 8 * sum_b n_b, every CTA c < num_ctas owns the flat tile range
 * [c*q, min((c+1)*q, T)) of the (seq, kv_head, tile) order, where
 * q = max(min_tiles, ceil(T / num_ctas)); its work items are that range cut
 * at (seq, kv_head) boundaries.  With pool_chunks = J > 0 the last
 * P = floor(q / 8) tiles of every range are cut into J chunks of
 * ceil(P / J) tiles and pooled, provided that is at least pool_min_tiles: a
 * CTA runs its home part, then claims pool chunks at run time until none is
 * left, so SMs that stream faster take more of the tail.  J = 0 (or chunks
 * below pool_min_tiles) deals everything statically.
 * Writes plan->items, cta_ptr, home_end, pool, seg_ptr.
 *   seq_lens   (device) int32 [batch], tokens per sequence including the new
 *              one; 0 is an empty sequence; < 0 or > max_blocks * 64 sets
 *              BAD_SEQ_LEN and the sequence is treated as empty
 *   plan       (host) plan->num_ctas and capacity set by the caller; if the
 *              items do not fit, PLAN_OVERFLOW is set and the plan is empty
 *   params     (host) planner knobs, or NULL for the defaults
 * Errors: HPC_ERR_INVALID_ARG for null pointers, batch < 0, max_blocks < 1,
 * knobs out of range or num_ctas < 1; HPC_ERR_UNSUPPORTED for batch > 8192,
 * num_ctas > HPC_MAX_PLAN_CTAS or batch * max_blocks * 8 >= 2^30. */
int hpc_decode_plan(const int32_t* seq_lens, int32_t batch, int32_t max_blocks,
                    const hpc_plan_params* params, hpc_plan* plan, int32_t* status,
                    cudaStream_t stream);

/* Static equal-split plan, the comparator of hpc_decode_plan: every
 * (seq, kv_head) is cut into `splits` chunks of ceil(n_b / splits) tiles
 * whatever its length, one chunk per CTA (item c runs on CTA c; no pool).
 * Requires plan->num_ctas == batch * 8 * splits and capacity >= num_ctas.
 * Same buffers, status bits and errors as hpc_decode_plan. */
int hpc_decode_plan_static(const int32_t* seq_lens, int32_t batch, int32_t max_blocks,
                           int32_t splits, hpc_plan* plan, int32_t* status, cudaStream_t stream);

/* Split-KV paged GQA decode attention.
 * Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
 * Hopper", intro of "Two new HPC backends in the vLLM ecosystem" (64 query
 * heads, 8 KV heads, head_dim 128) and "Why does dynamic scheduling matter
 * for attention?" (split-KV over 64-token tiles, BF16 and FP8 caches); page
 * "[vllm] Introducing the HPC-Ops attention backend", introduction (FP8 E4M3
 * models).  For every work item i = (b, h, t0, t1) and each of the 8 query
 * heads j = 8h .. 8h+7:
 *   s_t   = sm_scale * k_scale * q[b][j] . K[b][h][t]   for tokens t in tiles
 *           [t0, t1) with t < seq_lens[b]
 *   partial_o[i][j - 8h]   = v_scale * sum_t softmax(s)_t V[b][h][t]
 *   partial_lse[i][j - 8h] = log(sum_t exp(s_t))        (natural log)
 * Each 64-token K and V page is read from HBM once for all 8 query heads.
 *   q            (device) bf16 [batch, 64, 128] (q_out of the prologue)
 *   kv_cache     (device) as in hpc_rope_norm_kvwrite, 16-byte aligned
 *   kv_scale     (device) float32 [2]; required for e4m3, ignored for bf16
 *   block_table  (device) int32 [batch, max_blocks]; entry [b][t] is the cache
 *                block of tile t of sequence b (BAD_BLOCK if out of range:
 *                the tile is skipped)
 *   seq_lens     (device) int32 [batch]
 *   plan         (host) plan written by hpc_decode_plan / _static for the same
 *                seq_lens; its num_ctas queues set the grid.  A plan may be run any
 *                number of times, but launches that share one plan must not
 *                overlap on the GPU (they share its pool counters).
 *   partial_o    (device) float32 [plan->capacity, 8, 128], written per item,
 *                16-byte aligned
 *   partial_lse  (device) float32 [plan->capacity, 8], written per item,
 *                16-byte aligned (both alignments hold for every call that
 *                takes partial buffers: the attention writes and reads them,
 *                and the merges read them, 16 bytes at a time)
 * Errors: HPC_ERR_INVALID_ARG for null pointers, bad sizes or misaligned partials;
 * HPC_ERR_UNSUPPORTED for num_blocks > HPC_MAX_NUM_BLOCKS or unknown dtype. */
int hpc_decode_attn(const void* q, const void* kv_cache, int32_t kv_dtype, const float* kv_scale,
                    int32_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                    const int32_t* seq_lens, int32_t batch, const hpc_plan* plan,
                    float* partial_o, float* partial_lse, float sm_scale,
                    int32_t* status, cudaStream_t stream);

/* hpc_decode_attn with the log-sum-exp merge fused in: writes out (bf16
 * [batch, 64, 128], as hpc_merge would) in the same kernel.  A segment whose
 * tiles form one work item is normalised and written straight from the
 * item's epilogue; a segment of several items is merged by the CTA that
 * finishes its last item (plan->seg_done counts finished items; that CTA
 * resets the count), reading the other items' partials through L2.  The
 * partial buffers are still needed for segments of several items.
 * Same source passages as hpc_decode_attn and hpc_merge.
 * Errors: as hpc_decode_attn, and HPC_ERR_INVALID_ARG for a null out,
 * plan->seg_ptr or plan->seg_done. */
int hpc_decode_attn_merge(const void* q, const void* kv_cache, int32_t kv_dtype,
                          const float* kv_scale, int32_t num_blocks, const int32_t* block_table,
                          int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                          const hpc_plan* plan, float* partial_o, float* partial_lse, void* out,
                          float sm_scale, int32_t* status, cudaStream_t stream);

/* Diagnostic variant of hpc_decode_attn: the same kernel, which also writes
 * for every CTA c of the grid cta_clock[3c] = start and cta_clock[3c+1] = end
 * (the GPU's global timer, ns; the end is when the last of the CTA's queues
 * is done) and cta_clock[3c+2] = the SM it ran on.  Used to measure SM
 * occupancy and tail idle time of a schedule.
 *   cta_clock  (device) uint64 [plan->num_ctas * 3] (the grid's rows are
 *              written; the grid has at most plan->num_ctas CTAs).
 * Errors: as hpc_decode_attn, and HPC_ERR_INVALID_ARG if cta_clock is null. */
int hpc_decode_attn_profiled(const void* q, const void* kv_cache, int32_t kv_dtype,
                             const float* kv_scale, int32_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t batch, const hpc_plan* plan,
                             float* partial_o, float* partial_lse, float sm_scale,
                             int32_t* status, unsigned long long* cta_clock, cudaStream_t stream);

/* Log-sum-exp merge of the split partials.
 * Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
 * Hopper", section "Why does dynamic scheduling matter for attention?": a
 * split-KV schedule cuts a sequence's KV across compute units, which implies
 * combining their partial results into the sequence's output; the page does
 * not spell the combination out.  For each segment s = b*8 + h with items
 * K_s =
 * seg_ptr[s] .. seg_ptr[s+1]-1, in item order,
 *   M = max_k lse_k,  w_k = exp(lse_k - M),
 *   out[b][8h + r] = bf16( sum_k w_k partial_o[k][r] / sum_k w_k )
 * A segment with no items (an empty sequence) gets zeros.
 *   out  (device) bf16 [batch, 64, 128], written.
 * Errors: HPC_ERR_INVALID_ARG for null pointers or batch < 0. */
int hpc_merge(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
              int32_t batch, void* out, cudaStream_t stream);

/* No counterpart in the paper.  hpc_decode_attn followed by hpc_merge, for
 * callers that cannot allocate device memory (a fixed memory pool they may not
 * grow, another framework's allocator or graph hooks, an embedder that hands
 * over only its inputs and outputs): the fp32 partials live in a file-scope
 * device array of the library instead of caller buffers.  No allocation of
 * any kind is made.
 *   Arguments as in hpc_decode_attn, plus
 *   out  (device) bf16 [batch, 64, 128], written as by hpc_merge.
 * Limits and behaviour:
 *   - plan->capacity must be <= HPC_NOALLOC_MAX_ITEMS (4096 work items, a
 *     16.9 MB array that every GPU loading the library holds until exit);
 *     a larger plan returns HPC_ERR_UNSUPPORTED and launches nothing.  A
 *     length-proportional plan with the default 4 pool chunks on a 152-SM
 *     GPU fits batches up to 322 sequences (BF16, 304 queues) or 227 (FP8,
 *     456 queues).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it; make that first call before any
 *     stream capture.  The kept address belongs to the device's context of
 *     that moment: after the context is torn down and created again
 *     (cudaDeviceReset), the next call looks the address up anew, and that
 *     call, too, should come before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents;
 *     every item of a valid plan is rewritten before it is read, so nothing
 *     needs clearing.  Calls that overlap on the GPU (other streams, other
 *     threads) race on the array: serialise them.
 * Errors: as hpc_decode_attn and hpc_merge, plus the capacity limit above. */
#define HPC_NOALLOC_MAX_ITEMS 4096
int hpc_decode_attn_merge_noalloc(const void* q, const void* kv_cache, int32_t kv_dtype,
                                  const float* kv_scale, int32_t num_blocks,
                                  const int32_t* block_table, int32_t max_blocks,
                                  const int32_t* seq_lens, int32_t batch, const hpc_plan* plan,
                                  void* out, float sm_scale, int32_t* status, cudaStream_t stream);

/* The whole decode step in two launches: hpc_rope_norm_kvwrite and
 * hpc_decode_plan run in one kernel (one block plans while the others run
 * the prologue: they touch disjoint data), then hpc_decode_attn_merge is
 * launched as a programmatic dependent of it, so its CTAs are resident and
 * their pipelines set up when the plan and q become ready.  The result is the
 * same as the four calls in order (with the fused merge).
 * Arguments: those of hpc_rope_norm_kvwrite, hpc_decode_plan (params may be
 * NULL) and hpc_decode_attn_merge; q_out is the prologue's output and the
 * attention's q.  Same checks and errors as those calls.
 * Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
 * Hopper", "Why does dynamic scheduling matter for attention?" (per-step
 * scheduler, fused prologue) and "FP8 MoE pipeline as a single execution
 * path" (kernels chained with Programmatic Dependent Launch). */
int hpc_decode_step(const void* q, const void* k, const void* v, const int32_t* positions,
                    const float* cos_sin, int32_t max_pos, const void* q_norm_w,
                    const void* k_norm_w, float eps, void* kv_cache, int32_t kv_dtype,
                    int32_t num_blocks, const int64_t* slot_mapping, const float* kv_scale,
                    const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                    int32_t batch, const hpc_plan_params* params, hpc_plan* plan,
                    float* partial_o, float* partial_lse, void* q_out, void* out, float sm_scale,
                    int32_t* status, cudaStream_t stream);

/* Work queues of the persistent hpc_decode_attn grid on the current device
 * for the given KV dtype: SM count x queues per CTA (2 for BF16, 3 for FP8),
 * one CTA per SM.  The num_ctas to plan for. */
int hpc_decode_num_ctas(int32_t kv_dtype, int32_t* num_ctas);

/* The num_ctas to plan for when each sequence has q_len new tokens
 * (1 <= q_len <= HPC_MAX_Q_LEN) of the given q_dtype (HPC_Q_BF16 or
 * HPC_Q_FP8_E4M3): hpc_decode_num_ctas() except for E4M3 pages with q_len 3
 * or 4, or q_len 2 with an E4M3 q, which run the tensor-core form of the
 * attention at 2 queues per CTA (SMs x 2).
 * Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
 * Hopper", "Why does dynamic scheduling matter for attention?" (work dealt to
 * compute units in proportion to length).  Writes *num_queues; returns
 * HPC_ERR_INVALID_ARG for a null pointer, q_len out of range or another q_dtype,
 * HPC_ERR_UNSUPPORTED for another kv_dtype, HPC_ERR_CUDA if the device cannot
 * be queried. */
int hpc_decode_num_queues(int32_t kv_dtype, int32_t q_len, int32_t q_dtype, int32_t* num_queues);

/* Items a length-proportional plan may need:
 * num_ctas * (1 + pool_chunks) + 8 * batch. */
int32_t hpc_plan_capacity(int32_t batch, int32_t num_ctas, int32_t pool_chunks);

/* Multi-token decode: q_len = 2 .. HPC_MAX_Q_LEN new tokens per sequence,
 * decoded together (the draft tokens of a multi-token-prediction layer).
 * seq_lens counts every token of a sequence, the q_len new ones included;
 * new token j of sequence b sits at position seq_lens[b] - q_len + j and
 * attends to the keys at positions 0 .. seq_lens[b] - q_len + j (its
 * history and the new tokens up to itself).  A token that sees no key gets
 * zeros.  The prologue needs no variant: hpc_rope_norm_kvwrite treats its
 * batch as independent tokens, so call it with batch * q_len tokens, their
 * own positions and slots, in [batch][q_len] order.
 * Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
 * Hopper", intro of "Two new HPC backends in the vLLM ecosystem" (the served
 * model's multi-token-prediction layer); the attention is that of
 * hpc_decode_attn with the causal order among the new tokens.
 * Arguments as hpc_decode_attn / hpc_decode_attn_merge / hpc_merge, except:
 *   q            (device) bf16 [batch, q_len, 64, 128]
 *   q_len        1 .. HPC_MAX_Q_LEN (1 is hpc_decode_attn)
 *   partial_o    (device) float32 [plan->capacity, q_len, 8, 128]
 *   partial_lse  (device) float32 [plan->capacity, q_len, 8]
 *   out          (device) bf16 [batch, q_len, 64, 128]
 * The plan is the same as for single-token decode (tiles per sequence).
 * Errors: as the single-token calls, and HPC_ERR_INVALID_ARG for q_len out of
 * range. */
int hpc_decode_attn_mt(const void* q, const void* kv_cache, int32_t kv_dtype,
                       const float* kv_scale, int32_t num_blocks, const int32_t* block_table,
                       int32_t max_blocks, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                       const hpc_plan* plan, float* partial_o, float* partial_lse,
                       float sm_scale, int32_t* status, cudaStream_t stream);
int hpc_decode_attn_merge_mt(const void* q, const void* kv_cache, int32_t kv_dtype,
                             const float* kv_scale, int32_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t batch, int32_t q_len,
                             const hpc_plan* plan, float* partial_o, float* partial_lse,
                             void* out, float sm_scale, int32_t* status, cudaStream_t stream);
int hpc_merge_mt(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
                 int32_t batch, int32_t q_len, void* out, cudaStream_t stream);

/* The general forms of the prologue, the attention and the merge.
 * hpc_rope_norm_kvwrite_ex is hpc_rope_norm_kvwrite with the q output type
 * chosen: q_dtype = HPC_Q_FP8_E4M3 stores q_out as uint8 E4M3 codes of
 * q / q_scale ([batch, 64, 128], RNE, saturating at +-448) instead of BF16.
 * hpc_decode_attn_ex / hpc_decode_attn_merge_ex / hpc_merge_ex are the
 * attention calls with the options above: q is BF16 [batch, q_len, 64, 128]
 * or (HPC_Q_FP8_E4M3, FP8 cache only) uint8 codes of the same shape; out is
 * [batch, q_len, 64, 128] of the chosen out_dtype and 16-byte aligned;
 * partials are float32 [plan->capacity, q_len, 8, 128] and
 * [plan->capacity, q_len, 8].  The scores of an E4M3 q are
 * (q_code . k_code) * q_scale * k_scale * sm_scale, the code products
 * accumulated in fp32.
 * Source: page "[vllm] Introducing the HPC-Ops attention backend" (the
 * output dtype as a parameter of the caller; FP8 E4M3 models); page "vLLM and
 * Tencent Hunyuan upstream two HPC backends for NVIDIA Hopper" (FP8 attention).
 * Errors: as the plain calls; HPC_ERR_UNSUPPORTED for an E4M3 q with a BF16
 * cache or an unknown dtype; HPC_ERR_INVALID_ARG for q_len out of range or a
 * non-positive q_scale. */
int hpc_rope_norm_kvwrite_ex(const void* q, const void* k, const void* v,
                             const int32_t* positions, const float* cos_sin, int32_t max_pos,
                             const void* q_norm_w, const void* k_norm_w, float eps,
                             void* kv_cache, int32_t kv_dtype, int32_t num_blocks,
                             const int64_t* slot_mapping, const float* kv_scale,
                             int32_t q_dtype, float q_scale, void* q_out, int32_t batch,
                             int32_t* status, cudaStream_t stream);
int hpc_decode_attn_ex(const void* q, const void* kv_cache, int32_t kv_dtype,
                       const float* kv_scale, int32_t num_blocks, const int32_t* block_table,
                       int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                       const hpc_attn_options* opts, const hpc_plan* plan, float* partial_o,
                       float* partial_lse, float sm_scale, int32_t* status, cudaStream_t stream);
int hpc_decode_attn_merge_ex(const void* q, const void* kv_cache, int32_t kv_dtype,
                             const float* kv_scale, int32_t num_blocks,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t batch,
                             const hpc_attn_options* opts, const hpc_plan* plan,
                             float* partial_o, float* partial_lse, void* out, float sm_scale,
                             int32_t* status, cudaStream_t stream);
int hpc_merge_ex(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
                 int32_t batch, const hpc_attn_options* opts, void* out, cudaStream_t stream);

/* Prefill and mixed prefill + decode batches through the same paged cache.
 * Sequence b has q_len_b = query_start[b+1] - query_start[b] >= 0 new tokens
 * (a prompt chunk, a whole prompt, or one decode token), packed in
 * [query_start[b], query_start[b+1]) of q and out, and seq_lens[b] >= q_len_b
 * tokens in all, the new ones included.  New token i of sequence b sits at
 * position seq_lens[b] - q_len_b + i and attends to the keys at positions
 * 0 .. seq_lens[b] - q_len_b + i: its history and the new tokens up to
 * itself.  Write the new tokens' K and V first (hpc_rope_norm_kvwrite on the
 * packed tokens with their own positions and slots).  Decode sequences may
 * also go through hpc_decode_attn_* (split-KV, better for long histories);
 * both read the same cache.  With an E4M3 cache (kv_dtype HPC_KV_FP8_E4M3,
 * kv_scale = [k_scale, v_scale] on the device, required) the result is the
 * attention over the dequantised cache: the products run on F16 operands
 * (every E4M3 value is an F16 value; q is rounded to F16, exact for |q| in
 * [2^-14, 65504]).
 * hpc_prefill_plan: unit_ptr[b] = first work unit of sequence b (8 kv heads
 * x ceil(q_len_b / 32) token blocks), unit_ptr[batch] = all units; zeroes
 * counters.  hpc_prefill_attn deals the units to a persistent grid through
 * counters[0] and leaves both counters at zero (the plan can run again;
 * launches that share one plan must not overlap).
 * Source: page "[vllm] Introducing the HPC-Ops attention backend" (prefill,
 * decode and mixed batches); page "vLLM and Tencent Hunyuan upstream two HPC
 * backends for NVIDIA Hopper", intro of "Two new HPC backends in the vLLM
 * ecosystem" (heads, head_dim, paged cache).
 *   query_start  (device) int32 [batch + 1], nondecreasing
 *   unit_ptr     (device) int32 [batch + 1];  counters (device) int32 [2]
 *   q            (device) bf16 [num_tokens, 64, 128], 16-byte aligned
 *   out          (device) [num_tokens, 64, 128] of out_dtype, 16-byte aligned,
 *                written for every new token of a valid sequence
 *   status       BAD_SEQ_LEN for q_len_b < 0, q_len_b > seq_lens[b],
 *                seq_lens[b] > max_blocks * 64 or new tokens past num_tokens
 *                (the sequence is skipped);
 *                BAD_BLOCK for a block id out of range (the tile is skipped)
 * sm_scale must be positive (the softmax takes row maxima of unscaled scores).
 * Errors: HPC_ERR_INVALID_ARG for null pointers, bad sizes, sm_scale <= 0 or
 * misaligned q, out or kv_cache; HPC_ERR_INVALID_ARG for an E4M3 cache without kv_scale;
 * HPC_ERR_UNSUPPORTED for another kv_dtype, batch > 8192 or
 * num_blocks > HPC_MAX_NUM_BLOCKS. */
int hpc_prefill_plan(const int32_t* query_start, int32_t batch, int32_t* unit_ptr,
                     int32_t* counters, int32_t* status, cudaStream_t stream);
int hpc_prefill_attn(const void* q, int32_t num_tokens, const int32_t* query_start,
                     const void* kv_cache,
                     int32_t kv_dtype, const float* kv_scale, int32_t num_blocks,
                     const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                     int32_t batch, const int32_t* unit_ptr, int32_t* counters, void* out,
                     int32_t out_dtype, float sm_scale, int32_t* status, cudaStream_t stream);

/* hpc_prefill_attn with the pages of an E4M3 cache staged first.  Each tile
 * of a sequence is read by every unit of 32 new tokens that sees it (about
 * q_len / 64 units on average for a prompt), and the E4M3 kernel converts it
 * each time; this call instead converts every page the batch reads once, into
 * a caller-owned BF16 staging buffer (exact: every E4M3 value is a BF16
 * value), and runs the BF16 kernel over the staged pages with the K and V
 * scales.  Three launches: the page prefix, the conversion, the attention.
 * The result is the attention over the dequantised cache, with P stored as
 * BF16 (as for a BF16 cache) instead of F16.  For a BF16 cache this is
 * hpc_prefill_attn (staging unused).
 * Source: as hpc_prefill_attn.
 * Arguments as hpc_prefill_attn, and:
 *   staging        (device) [staging_pages][2][8][64][128] bf16, 16-byte
 *                  aligned, written: staged page page_ptr[b] + j holds block
 *                  block_table[b][j] of sequence b
 *   staging_pages  pages staging holds; it needs sum_b ceil(seq_lens[b] / 64)
 *   page_ptr       (device) int32 [batch + 1], written: page_ptr[b] = first
 *                  staged page of sequence b, page_ptr[batch] = all pages
 *   status         as hpc_prefill_attn, and PLAN_OVERFLOW for a sequence whose
 *                  pages do not fit in staging (the sequence is skipped)
 * Errors: as hpc_prefill_attn; HPC_ERR_INVALID_ARG for an E4M3 cache without
 * staging or page_ptr, staging_pages < 1 or misaligned staging;
 * HPC_ERR_UNSUPPORTED for staging_pages > HPC_MAX_NUM_BLOCKS. */
int hpc_prefill_attn_staged(const void* q, int32_t num_tokens, const int32_t* query_start,
                            const void* kv_cache, int32_t kv_dtype, const float* kv_scale,
                            int32_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                            const int32_t* seq_lens, int32_t batch, const int32_t* unit_ptr,
                            int32_t* counters, void* out, int32_t out_dtype, float sm_scale,
                            void* staging, int32_t staging_pages, int32_t* page_ptr,
                            int32_t* status, cudaStream_t stream);

/* Self-test of the bounded pipeline wait (no counterpart on the pages).
 * Every wait of the attention pipeline gives up after a time limit (1 s),
 * sets HPC_STATUS_WAIT_TIMEOUT and winds its CTA down, so a stuck pipeline
 * becomes a status word instead of a hung GPU.  This call runs that same wait
 * on an mbarrier phase that can never complete, with the given limit: on
 * return of the stream work, *status has HPC_STATUS_WAIT_TIMEOUT set and
 * *waited_ns (if not NULL) holds how long the wait lasted (>= limit_ns).
 * Nothing faults; the context stays usable.
 *   limit_ns   1e3 .. 1e9 (HPC_ERR_INVALID_ARG otherwise)
 *   status     (device) int32, bits or-ed in
 *   waited_ns  (device) uint64 [1] or NULL */
int hpc_selftest_wait_timeout(uint64_t limit_ns, int32_t* status, uint64_t* waited_ns,
                              cudaStream_t stream);

/* Self-test of the bounded polling wait (no counterpart on the pages).  The
 * tensor-core form of the 4-token attention layout has a warp that tests
 * several barriers without blocking on any; when none is ready for the time
 * limit (1 s) it gives up the same way: HPC_STATUS_WAIT_TIMEOUT, the CTA's
 * abort flag, wind-down.  This call runs that polling loop over two mbarrier
 * phases that never complete, with the given limit; arguments, results and
 * errors as hpc_selftest_wait_timeout. */
int hpc_selftest_poll_timeout(uint64_t limit_ns, int32_t* status, uint64_t* waited_ns,
                              cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HPC_DECODE_H */
