// Self-test of the bounded waits every kernel relies on for failure
// detection: one thread waits, through the same routine the kernels use, on
// a shared-memory mbarrier that nothing arrives on.  The wait gives up after
// the limit, the thread ORs PKD_DEV_TIMEOUT into the status word and the
// kernel returns, leaving the context usable.  Nothing faults or traps.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace pkd {
namespace {

__global__ void selftest_wait_kernel(uint32_t* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  // Phase 0 of a fresh barrier completes only when one thread arrives; none does.
  if (threadIdx.x == 0 && !sm100::mbar_wait(&bar, 0, limit_ns)) flag(status, PKD_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t* status, long long limit_ns, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(status, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

}  // namespace pkd
