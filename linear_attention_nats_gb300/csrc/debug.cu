// debug.cu - test hook of the bounded waits: one thread waits, with a short
// limit, on an mbarrier phase that nothing completes, so the wait gives up,
// sets the caller's flag and returns (the same path every tensor-core kernel
// takes when one of its waits expires).  No fault, no hang.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace nats {
namespace {

__global__ void bounded_wait_kernel(int* flag, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  // phase 0 of a fresh barrier completes only after one arrival; none comes
  if (threadIdx.x == 0) tc::mbar_wait_for(&bar, 0, flag, limit_ns);
}

}  // namespace

cudaError_t launch_bounded_wait(int* flag, long long limit_ns, cudaStream_t st) {
  bounded_wait_kernel<<<1, 32, 0, st>>>(flag, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

}  // namespace nats
