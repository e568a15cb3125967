// test_hooks.cu -- entry points that exist only in a test build of the
// library (compiled with PK_TEST_HOOKS; the product library exports none of
// them).  The test build also shortens the bounded-wait limit
// (PK_WAIT_LIMIT_CYCLES) so that a wait that can never finish gives up within
// microseconds.
#ifdef PK_TEST_HOOKS

#include "pk_common.cuh"
#include "pk_internal.h"

namespace {

// Every thread waits on an mbarrier that nothing arrives on and no copy
// completes on (no TMA or other asynchronous copy is issued).  The bounded
// wait the kernels use must give up after the limit; the kernel then reports
// PA_DEV_TIMEOUT in the status word, counts the threads that gave up, and
// returns.
__global__ void wait_gives_up_kernel(int32_t* status, int32_t* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    pk::mbar_init(&bar, 1);
    pk::fence_mbar_init();
  }
  __syncthreads();
  if (!pk::mbar_wait(&bar, 0)) {
    if (threadIdx.x == 0) pk::flag_status(status, PA_DEV_TIMEOUT);
    atomicAdd(gave_up, 1);
  }
}

}  // namespace

extern "C" long long pk_test_wait_limit_cycles(void) { return pk::kWaitLimitCycles; }

// Launches one CTA of `threads` threads (1..1024) of wait_gives_up_kernel on
// `stream`; returns a cudaError_t value (0 = launched).
extern "C" int pk_test_wait_gives_up(int32_t* status, int32_t* gave_up, int threads,
                                     cudaStream_t stream) {
  if (status == nullptr || gave_up == nullptr || threads < 1 || threads > 1024)
    return (int)cudaErrorInvalidValue;
  wait_gives_up_kernel<<<1, threads, 0, stream>>>(status, gave_up);
  return (int)cudaGetLastError();
}

#endif  // PK_TEST_HOOKS
