// The 4-token query layout of the decode attention kernel (attn_kernel.cuh):
// multi-token decode with q_len = 3 or 4 new tokens per sequence (q_len = 3
// leaves one query's warp of every queue idle).  In its own translation unit
// so that its kernel instances compile in parallel with the others.
//
// Source: page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA
// Hopper", intro of "Two new HPC backends in the vLLM ecosystem" (the served
// model's multi-token-prediction layer).
#include "attn_kernel.cuh"

int hpc::launch_decode_attn_q4(HPC_LAYOUT_LAUNCH_ARGS) {
  return hpc::launch_attn_layout<4>(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                    max_blocks, seq_lens, batch, opts, plan, partial_o, partial_lse,
                                    sm_scale, status, cta_clock, out, pdl, stream);
}
