// RVQ decode: y[n] = sum_{q < n_q} Z[q][codes[n][q]]
//
// The decode graph of omnivoice.cpp ARCHITECTURE.md ("RVQ codec": per stage
// gather the codeword, project_out, add the bias, accumulate) with the
// projection and bias folded into the prepared table Z[q][k] = w_out[q] .
// codebook[q][k] + b_out[q].  Per frame this reads n_q codes and writes D
// floats; the gathers hit Z, which stays resident in L2.
#include "rvq_internal.cuh"

namespace rvq {
namespace {

// One warp-row of threads per frame: each thread owns float4 column groups.
// blockDim = (TX, FY): TX threads across the row, FY frames per block.
__global__ void __launch_bounds__(256) k_decode_gather(const float4 *__restrict__ Z4,
                                                       const int32_t *__restrict__ codes,
                                                       float4 *__restrict__ y4, int64_t n_rows,
                                                       int n_q, int K, int D4,
                                                       unsigned long long *__restrict__ bad) {
  const int64_t n = (int64_t)blockIdx.x * blockDim.y + threadIdx.y;
  int n_bad = 0;
  if (n < n_rows) {
    const int32_t *cn = codes + n * n_q;
    for (int c = threadIdx.x; c < D4; c += blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < n_q; ++q) {
        const int32_t code = __ldg(cn + q);
        if (code < 0 || code >= K) {
          n_bad += (c == threadIdx.x && threadIdx.x == 0);
          continue;
        }
        const float4 z = __ldg(Z4 + ((int64_t)q * K + code) * D4 + c);
        acc.x += z.x;
        acc.y += z.y;
        acc.z += z.z;
        acc.w += z.w;
      }
      __stcs(y4 + n * D4 + c, acc);
    }
  }
  if (bad && n_bad) atomicAdd(bad, (unsigned long long)n_bad);
}

}  // namespace

cudaError_t launch_decode(const rvq_dims &dm, const void *tables, const int32_t *codes, int64_t n, int n_q,
                          float *y, int64_t *bad, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  const int D4 = dm.D / 4;
  const int tx = D4 >= 256 ? 256 : (D4 >= 128 ? 128 : (D4 >= 64 ? 64 : 32));
  const int fy = 256 / tx;
  dim3 block(tx, fy);
  const unsigned grid = (unsigned)((n + fy - 1) / fy);
  k_decode_gather<<<grid, block, 0, st>>>(at<float4>(tables, L.z), codes, reinterpret_cast<float4 *>(y), n, n_q,
                                          dm.K, D4, reinterpret_cast<unsigned long long *>(bad));
  return cudaGetLastError();
}

}  // namespace rvq
