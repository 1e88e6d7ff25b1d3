// Decode attention + merge for callers that cannot allocate device memory.
//
// The regular path needs two caller-allocated scratch buffers between the
// attention and the merge (the fp32 partial outputs and log-sum-exps of the
// split-KV work items).  Some callers cannot call cudaMalloc: code that runs
// with a device memory pool it may not grow, code inside another framework's
// allocator or graph-replay hooks, or embedders that hand the library only
// their own input and output buffers.  This entry point keeps that scratch in
// a file-scope device array instead, sized for at most HPC_NOALLOC_MAX_ITEMS
// work items (8.5 MB), which every GPU that loads the library holds until the
// process exits.  It makes no allocation of any kind; it runs the very same
// hpc_decode_attn and hpc_merge kernels with the array as their scratch.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kPartialFloats = static_cast<size_t>(HPC_NOALLOC_MAX_ITEMS) * hpc::kGroup * hpc::kD;
constexpr size_t kLseFloats = static_cast<size_t>(HPC_NOALLOC_MAX_ITEMS) * hpc::kGroup;

// [HPC_NOALLOC_MAX_ITEMS][8][128] partial outputs, then [..][8] log-sum-exps.
static __device__ __align__(256) float g_noalloc_scratch[kPartialFloats + kLseFloats];

// Device address of the array on the current device.  The name of a
// __device__ variable in host code is only a host-side stand-in, so the
// address is looked up once per device (with that device current) and kept.
cudaError_t scratch_address(float** out) {
  static std::mutex mu;
  static float* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int hpc_decode_attn_merge_noalloc(const void* q, const void* kv_cache, int32_t kv_dtype,
                                             const float* kv_scale, int32_t num_blocks,
                                             const int32_t* block_table, int32_t max_blocks,
                                             const int32_t* seq_lens, int32_t batch,
                                             const hpc_plan* plan, void* out, float sm_scale,
                                             int32_t* status, cudaStream_t stream) {
  HPC_CHECK_ARG(plan != nullptr && out != nullptr);
  if (plan->capacity < 0 || plan->capacity > HPC_NOALLOC_MAX_ITEMS) return HPC_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return HPC_ERR_CUDA;
  float* partial_o = scratch;
  float* partial_lse = scratch + kPartialFloats;
  // Every item of a valid plan is written by the attention kernel before the
  // merge reads it, so nothing left in the array by an earlier call is read.
  const int rc = hpc_decode_attn(q, kv_cache, kv_dtype, kv_scale, num_blocks, block_table,
                                 max_blocks, seq_lens, batch, plan, partial_o, partial_lse,
                                 sm_scale, status, stream);
  if (rc != HPC_OK) return rc;
  return hpc_merge(partial_o, partial_lse, plan, batch, out, stream);
}
