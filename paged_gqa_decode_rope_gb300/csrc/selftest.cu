// Self-test of the bounded pipeline wait.  Every wait of the attention
// pipeline goes through mbar_wait, which gives up after a time limit, records
// HPC_STATUS_WAIT_TIMEOUT and lets the CTA wind down, so a stuck pipeline ends
// as a status the host reads and the context stays usable.  This kernel makes
// that wait run out on purpose, without any fault: it waits on the phase of
// an mbarrier that expects two arrivals and only ever gets one.
#include "common.cuh"

namespace hpc {
namespace {

__global__ void wait_timeout_kernel(unsigned long long limit_ns, int32_t* status,
                                    unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 2);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(smem_u32(&bar));   // the second arrival never comes
  const unsigned long long t0 = globaltimer_ns();
  const bool done = mbar_wait(smem_u32(&bar), 0, status, limit_ns);
  const unsigned long long t1 = globaltimer_ns();
  if (threadIdx.x == 0 && waited_ns != nullptr) waited_ns[0] = done ? 0ull : t1 - t0;
}

// The polling form of the same wait (the tensor-core form's MMA warp tests
// several barriers without blocking on any, then calls poll_give_up): one
// warp polls two barriers that nothing ever completes until the limit runs
// out.
__global__ void poll_timeout_kernel(unsigned long long limit_ns, int32_t* status,
                                    unsigned long long* waited_ns) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const unsigned long long t0 = globaltimer_ns();
  unsigned long long idle_since = 0ull;
  bool gave_up = false;
  while (true) {
    const bool ready = mbar_test_wait(smem_u32(&bar[0]), 0) || mbar_test_wait(smem_u32(&bar[1]), 0);
    if (__any_sync(0xffffffffu, ready)) break;
    if (poll_give_up(idle_since, &abort_flag, status, limit_ns)) {
      gave_up = true;
      break;
    }
    __nanosleep(64);
  }
  const unsigned long long t1 = globaltimer_ns();
  if (threadIdx.x == 0 && waited_ns != nullptr) waited_ns[0] = gave_up ? t1 - t0 : 0ull;
}

}  // namespace
}  // namespace hpc

extern "C" int hpc_selftest_wait_timeout(uint64_t limit_ns, int32_t* status, uint64_t* waited_ns,
                                         cudaStream_t stream) {
  HPC_CHECK_ARG(status != nullptr);
  HPC_CHECK_ARG(limit_ns >= 1000ull && limit_ns <= 1000000000ull);
  hpc::wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, status,
                                                  reinterpret_cast<unsigned long long*>(waited_ns));
  return HPC_LAUNCH_STATUS();
}

extern "C" int hpc_selftest_poll_timeout(uint64_t limit_ns, int32_t* status, uint64_t* waited_ns,
                                         cudaStream_t stream) {
  HPC_CHECK_ARG(status != nullptr);
  HPC_CHECK_ARG(limit_ns >= 1000ull && limit_ns <= 1000000000ull);
  hpc::poll_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, status,
                                                  reinterpret_cast<unsigned long long*>(waited_ns));
  return HPC_LAUNCH_STATUS();
}
