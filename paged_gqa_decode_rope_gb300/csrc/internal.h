// Library-internal entry points shared between translation units.
#pragma once

#include "hpc_decode.h"

namespace hpc {

// hpc_decode_attn / _merge / _profiled / _ex in one: checks the arguments and
// the options and launches the attention kernel.  out != nullptr fuses the
// merge; cta_clock != nullptr records per-CTA clocks; pdl launches the kernel
// as a programmatic dependent of the previous kernel on the stream.
int launch_decode_attn(const void* q, const void* kv_cache, int32_t kv_dtype, const float* kv_scale,
                       int32_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                       const int32_t* seq_lens, int32_t batch, const hpc_attn_options& opts,
                       const hpc_plan* plan, float* partial_o, float* partial_lse, float sm_scale,
                       int32_t* status, unsigned long long* cta_clock, void* out, bool pdl,
                       cudaStream_t stream);

// The launches of the 2- and 4-token query layouts (arguments already
// checked), each in its own translation unit so that the kernel instances
// compile in parallel.
#define HPC_LAYOUT_LAUNCH_ARGS                                                                    \
  const void *q, const void *kv_cache, int32_t kv_dtype, const float *kv_scale,                   \
      int32_t num_blocks, const int32_t *block_table, int32_t max_blocks,                         \
      const int32_t *seq_lens, int32_t batch, const hpc_attn_options &opts, const hpc_plan *plan, \
      float *partial_o, float *partial_lse, float sm_scale, int32_t *status,                      \
      unsigned long long *cta_clock, void *out, bool pdl, cudaStream_t stream
int launch_decode_attn_q2(HPC_LAYOUT_LAUNCH_ARGS);
int launch_decode_attn_q4(HPC_LAYOUT_LAUNCH_ARGS);

// hpc_merge_ex with its checks; skip_single leaves the output rows of
// single-item segments alone (the attention kernel wrote them directly).
int launch_merge(const float* partial_o, const float* partial_lse, const hpc_plan* plan,
                 int32_t batch, const hpc_attn_options* opts, void* out, bool skip_single,
                 cudaStream_t stream);

// Whether the attention runs the tensor-core form (the 4-token layout's
// kernel, two queues per CTA): every call with q_len 3 or 4, and q_len 2
// with an E4M3 q on an E4M3 cache.  hpc_decode_num_queues and the dispatch
// both follow it.
inline bool uses_tensor_form(int32_t kv_dtype, int32_t q_len, int32_t q_dtype) {
  return q_len >= 3 || (q_len == 2 && kv_dtype == HPC_KV_FP8_E4M3 && q_dtype == HPC_Q_FP8_E4M3);
}

// The single-token BF16 options: {1, HPC_Q_BF16, 1.0f, HPC_OUT_BF16}.
inline hpc_attn_options default_attn_options() {
  hpc_attn_options o;
  o.q_len = 1;
  o.q_dtype = HPC_Q_BF16;
  o.q_scale = 1.0f;
  o.out_dtype = HPC_OUT_BF16;
  return o;
}

}  // namespace hpc
