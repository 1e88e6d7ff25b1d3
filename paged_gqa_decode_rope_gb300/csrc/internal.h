// Library-internal entry points shared between translation units.
#pragma once

#include "hpc_decode.h"

namespace hpc {

// hpc_decode_attn / _merge / _profiled and their multi-token forms in one:
// checks the arguments and launches the attention kernel for q_len new
// tokens per sequence (1 .. HPC_MAX_Q_LEN).  out != nullptr fuses the merge;
// cta_clock != nullptr records per-CTA clocks; pdl launches the kernel as a
// programmatic dependent of the previous kernel on the stream.
int launch_decode_attn(const void* q, const void* kv_cache, int32_t kv_dtype, const float* kv_scale,
                       int32_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                       const int32_t* seq_lens, int32_t batch, int32_t q_len, const hpc_plan* plan,
                       float* partial_o, float* partial_lse, float sm_scale, int32_t* status,
                       unsigned long long* cta_clock, void* out, bool pdl, cudaStream_t stream);

// The multi-token launches (q_len 2 .. HPC_MAX_Q_LEN), arguments already
// checked; in their own translation unit so that the kernel instances
// compile in parallel.
int launch_decode_attn_multi(const void* q, const void* kv_cache, int32_t kv_dtype,
                             const float* kv_scale, int32_t num_blocks, const int32_t* block_table,
                             int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                             int32_t q_len, const hpc_plan* plan, float* partial_o,
                             float* partial_lse, float sm_scale, int32_t* status,
                             unsigned long long* cta_clock, void* out, bool pdl,
                             cudaStream_t stream);

}  // namespace hpc
