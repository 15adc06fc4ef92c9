// Self-test of the bounded mbarrier wait every kernel of the library uses:
// a kernel waits on a barrier that nothing ever arrives at.  The wait must give
// up after its poll limit, the kernel must record the timeout status and
// return, and the context must stay usable for the next launch.
// Built by tests/test_bounded_wait_gpu.py with a short RVQ_SPIN_LIMIT.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace {

__global__ void k_wait_forever(int *status, unsigned long long *polls_clock) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    rvq::ptx::mbar_init(&bar, 1);  // expects one arrival that never comes
    rvq::ptx::fence_mbar_init();
  }
  __syncthreads();
  const long long t0 = clock64();
  const bool done = rvq::ptx::mbar_wait(&bar, 0);
  if (threadIdx.x == 0) {
    *polls_clock = (unsigned long long)(clock64() - t0);
    if (!done) atomicCAS(status, 0, 5);
  }
}

__global__ void k_after(int *out) { out[threadIdx.x] = 1000 + threadIdx.x; }

}  // namespace

extern "C" int selftest_bounded_wait(int *status, unsigned long long *clk, int *after) {
  k_wait_forever<<<1, 64>>>(status, clk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  k_after<<<1, 32>>>(after);
  e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  return (int)cudaDeviceSynchronize();
}
