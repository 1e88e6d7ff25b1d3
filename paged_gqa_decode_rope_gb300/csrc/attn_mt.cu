// Multi-token decode attention: q_len = 2 .. 4 new tokens per sequence, each
// seeing the history and the new tokens up to itself.  The kernel is the one
// of attn_kernel.cuh; this unit holds its 2-token query layout and the
// multi-token entry points, attn_mt4.cu the 4-token layout (q_len 3 and 4).
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper", intro of "Two new HPC backends in the vLLM ecosystem": the served
// model has a multi-token-prediction layer, whose draft tokens a decode step
// verifies together; the attention is the paged GQA decode attention of the
// same page, with the causal order among the new tokens.
#include "attn_kernel.cuh"

namespace {
hpc_attn_options opts_of(int32_t q_len) {
  hpc_attn_options o = hpc::default_attn_options();
  o.q_len = q_len;
  return o;
}
}  // namespace

int hpc::launch_decode_attn_q2(HPC_LAYOUT_LAUNCH_ARGS) {
  return hpc::launch_attn_layout<2>(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                    max_blocks, seq_lens, batch, opts, plan, partial_o, partial_lse,
                                    sm_scale, status, cta_clock, out, pdl, stream);
}

extern "C" int hpc_decode_attn_mt(const void* q, const void* kv_cache, int32_t kv_dtype,
                                  const float* kv_scale, int32_t num_blocks,
                                  const int32_t* block_table, int32_t max_blocks,
                                  const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                  const hpc_plan* plan, float* partial_o, float* partial_lse,
                                  float sm_scale, int32_t* status, cudaStream_t stream) {
  return hpc::launch_decode_attn(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, opts_of(q_len), plan, partial_o,
                                 partial_lse,
                                 sm_scale, status, nullptr, nullptr, false, stream);
}

extern "C" int hpc_decode_attn_merge_mt(const void* q, const void* kv_cache, int32_t kv_dtype,
                                        const float* kv_scale, int32_t num_blocks,
                                        const int32_t* block_table, int32_t max_blocks,
                                        const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                        const hpc_plan* plan, float* partial_o,
                                        float* partial_lse, void* out, float sm_scale,
                                        int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(out != nullptr);
  return hpc::launch_decode_attn(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, opts_of(q_len), plan, partial_o,
                                 partial_lse,
                                 sm_scale, status, nullptr, out, false, stream);
}
