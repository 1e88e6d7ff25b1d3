// Decode attention + merge for callers that cannot allocate device memory.
//
// The regular path needs two caller-allocated scratch buffers between the
// attention and the merge (the fp32 partial outputs and log-sum-exps of the
// split-KV work items).  Some callers cannot call cudaMalloc: code that runs
// with a device memory pool it may not grow, code inside another framework's
// allocator or graph-replay hooks, or embedders that hand the library only
// their own input and output buffers.  This entry point keeps that scratch in
// a file-scope device array instead, sized for at most HPC_NOALLOC_MAX_ITEMS
// work items (4096 x 8 x 128 fp32 partial outputs + 4096 x 8 fp32
// log-sum-exps = 16.9 MB), which every GPU that loads the library holds until
// the process exits.  It makes no allocation of any kind; it runs the very same
// hpc_decode_attn and hpc_merge kernels with the array as their scratch.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace {

constexpr size_t kPartialFloats = static_cast<size_t>(HPC_NOALLOC_MAX_ITEMS) * hpc::kGroup * hpc::kD;
constexpr size_t kLseFloats = static_cast<size_t>(HPC_NOALLOC_MAX_ITEMS) * hpc::kGroup;

// [HPC_NOALLOC_MAX_ITEMS][8][128] partial outputs, then [..][8] log-sum-exps.
static __device__ __align__(256) float g_noalloc_scratch[kPartialFloats + kLseFloats];

// Id of the calling thread's current CUDA context, or 0 if there is none yet
// (or the driver cannot say).  Resolved through the runtime's driver entry
// points, so the library links no libcuda.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &qr) ==
            cudaSuccess && qr == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess && qr == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the array on the current device.  The name of a
// __device__ variable in host code is only a host-side stand-in, so the
// address is looked up (with that device current) and kept per device,
// together with the id of the context it belongs to: a context that was torn
// down and created again (cudaDeviceReset) loads the module anew, possibly at
// another address, so a cached address is used only while the context it was
// looked up in is still the current one.
cudaError_t scratch_address(float** out) {
  static std::mutex mu;
  static float* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float*>(p);
    ctx_of[dev] = current_context_id();   // the lookup made the context current if it was not
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
