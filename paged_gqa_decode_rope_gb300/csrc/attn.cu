// Single-token decode attention entry points (q_len = 1) and the attention
// launcher shared with the step and the no-allocation entry point.  The
// kernel itself is in attn_kernel.cuh; multi-token decode is in attn_mt.cu.
#include "attn_kernel.cuh"

int hpc::launch_decode_attn(const void* q, const void* kv_cache, int32_t kv_dtype,
                            const float* kv_scale, int32_t num_blocks, const int32_t* block_table,
                            int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                            const hpc_attn_options& opts, const hpc_plan* plan, float* partial_o,
                            float* partial_lse, float sm_scale, int32_t* status,
                            unsigned long long* cta_clock, void* out, bool pdl,
                            cudaStream_t stream) {
  int rc = hpc::check_attn_args(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                max_blocks, seq_lens, batch, plan, partial_o, partial_lse, status,
                                out);
  if (rc != HPC_OK) return rc;
  rc = hpc::check_attn_options(opts, kv_dtype, out);
  if (rc != HPC_OK) return rc;
  if (opts.q_len == 1)
    return hpc::launch_attn_layout<1>(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                      max_blocks, seq_lens, batch, opts, plan, partial_o,
                                      partial_lse, sm_scale, status, cta_clock, out, pdl, stream);
  if (opts.q_len == 2 && !hpc::uses_tensor_form(kv_dtype, opts.q_len, opts.q_dtype))
    return hpc::launch_decode_attn_q2(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                      max_blocks, seq_lens, batch, opts, plan, partial_o,
                                      partial_lse, sm_scale, status, cta_clock, out, pdl, stream);
  return hpc::launch_decode_attn_q4(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                    max_blocks, seq_lens, batch, opts, plan, partial_o, partial_lse,
                                    sm_scale, status, cta_clock, out, pdl, stream);
}

extern "C" int hpc_decode_attn(const void* q, const void* kv_cache, int32_t kv_dtype,
                               const float* kv_scale, int32_t num_blocks,
                               const int32_t* block_table, int32_t max_blocks,
                               const int32_t* seq_lens, int32_t batch, const hpc_plan* plan,
                               float* partial_o, float* partial_lse, float sm_scale,
                               int32_t* status, cudaStream_t stream) {
  return hpc::launch_decode_attn(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, hpc::default_attn_options(), plan,
                                 partial_o, partial_lse,
                                 sm_scale, status, nullptr, nullptr, false, stream);
}

extern "C" int hpc_decode_attn_profiled(const void* q, const void* kv_cache, int32_t kv_dtype,
                                        const float* kv_scale, int32_t num_blocks,
                                        const int32_t* block_table, int32_t max_blocks,
                                        const int32_t* seq_lens, int32_t batch,
                                        const hpc_plan* plan, float* partial_o,
                                        float* partial_lse, float sm_scale, int32_t* status,
                                        unsigned long long* cta_clock, cudaStream_t stream) {
  HPC_CHECK_ARG(cta_clock != nullptr);
  return hpc::launch_decode_attn(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, hpc::default_attn_options(), plan,
                                 partial_o, partial_lse,
                                 sm_scale, status, cta_clock, nullptr, false, stream);
}

extern "C" int hpc_decode_attn_merge(const void* q, const void* kv_cache, int32_t kv_dtype,
                                     const float* kv_scale, int32_t num_blocks,
                                     const int32_t* block_table, int32_t max_blocks,
                                     const int32_t* seq_lens, int32_t batch, const hpc_plan* plan,
                                     float* partial_o, float* partial_lse, void* out,
                                     float sm_scale, int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(out != nullptr);
  return hpc::launch_decode_attn(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, hpc::default_attn_options(), plan,
                                 partial_o, partial_lse,
                                 sm_scale, status, nullptr, out, false, stream);
}

extern "C" int hpc_decode_num_ctas(int32_t kv_dtype, int32_t* num_ctas) {
  HPC_CHECK_ARG(num_ctas != nullptr);
  if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HPC_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HPC_ERR_CUDA;
  // one resident CTA per SM (the stage rings take ~200 KB), each running
  // 2 (BF16) or 3 (FP8) work queues
  *num_ctas = sms * (kv_dtype == HPC_KV_BF16 ? hpc::AttnTraits<false>::kGroups
                                             : hpc::AttnTraits<true>::kGroups);
  return HPC_OK;
}

extern "C" int hpc_decode_num_queues(int32_t kv_dtype, int32_t q_len, int32_t q_dtype,
                                     int32_t* num_queues) {
  HPC_CHECK_ARG(num_queues != nullptr && q_len >= 1 && q_len <= HPC_MAX_Q_LEN);
  HPC_CHECK_ARG(q_dtype == HPC_Q_BF16 || q_dtype == HPC_Q_FP8_E4M3);
  // the tensor-core form runs two queues per CTA on both cache types, like
  // the BF16 cache's other layouts; the E4M3 cache's mma.sync layouts run three
  if (kv_dtype != HPC_KV_FP8_E4M3 || !hpc::uses_tensor_form(kv_dtype, q_len, q_dtype))
    return hpc_decode_num_ctas(kv_dtype, num_queues);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HPC_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HPC_ERR_CUDA;
  *num_queues = sms * hpc::AttnTraits<true, true>::kGroups;
  return HPC_OK;
}

extern "C" int hpc_decode_attn_ex(const void* q, const void* kv_cache, int32_t kv_dtype,
                                  const float* kv_scale, int32_t num_blocks,
                                  const int32_t* block_table, int32_t max_blocks,
                                  const int32_t* seq_lens, int32_t batch,
                                  const hpc_attn_options* opts, const hpc_plan* plan,
                                  float* partial_o, float* partial_lse, float sm_scale,
                                  int32_t* status, cudaStream_t stream) {
  const hpc_attn_options o = opts != nullptr ? *opts : hpc::default_attn_options();
  return hpc::launch_decode_attn(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, o, plan, partial_o, partial_lse,
                                 sm_scale, status, nullptr, nullptr, false, stream);
}

extern "C" int hpc_decode_attn_merge_ex(const void* q, const void* kv_cache, int32_t kv_dtype,
                                        const float* kv_scale, int32_t num_blocks,
                                        const int32_t* block_table, int32_t max_blocks,
                                        const int32_t* seq_lens, int32_t batch,
                                        const hpc_attn_options* opts, const hpc_plan* plan,
                                        float* partial_o, float* partial_lse, void* out,
                                        float sm_scale, int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(out != nullptr);
  const hpc_attn_options o = opts != nullptr ? *opts : hpc::default_attn_options();
  return hpc::launch_decode_attn(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, o, plan, partial_o, partial_lse,
                                 sm_scale, status, nullptr, out, false, stream);
}
