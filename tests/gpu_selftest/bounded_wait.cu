// Self-test of the bounded mbarrier waits every kernel of the library uses:
// a kernel (and a 2-CTA cluster kernel, for the cluster-scope waits) waits on
// a barrier that nothing ever arrives at.  The wait must give
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

// The same for the cluster-scope waits of the small-batch kernels: in a
// 2-CTA cluster, every CTA waits (acquire at cluster scope, the polling form
// first) on a barrier whose arrivals would come from the other CTA's
// st.async / remote arrive, which never come.  Both give up, record the
// status, and still meet at the closing cluster barrier.
__global__ void k_cluster_wait_forever(int *status, unsigned long long *polls_clock) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    rvq::ptx::mbar_init(&bar, 2);
    rvq::ptx::fence_mbar_init();
  }
  __syncthreads();
  rvq::ptx::cluster_sync_all();  // both CTAs' barriers are initialised
  const long long t0 = clock64();
  const bool done = rvq::ptx::mbar_wait_cluster_hot(&bar, 0);
  if (threadIdx.x == 0) {
    if (rvq::ptx::cluster_ctarank() == 0) polls_clock[1] = (unsigned long long)(clock64() - t0);
    if (!done) atomicAdd(status + 1, 1);
  }
  rvq::ptx::cluster_sync_all();
}

__global__ void k_after(int *out) { out[threadIdx.x] = 1000 + threadIdx.x; }

}  // namespace

extern "C" int selftest_bounded_wait(int *status, unsigned long long *clk, int *after) {
  k_wait_forever<<<1, 64>>>(status, clk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(64, 1, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_cluster_wait_forever, status, clk);
  if (e != cudaSuccess) return (int)e;
  k_after<<<1, 32>>>(after);
  e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  return (int)cudaDeviceSynchronize();
}
