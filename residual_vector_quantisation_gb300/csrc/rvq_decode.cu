// RVQ decode: y[n] = b_dec + sum_{q < n_q} Z[q][codes[n][q]]
//
// The decode graph of omnivoice.cpp ARCHITECTURE.md ("RVQ codec": per stage
// gather the codeword, project_out, add the bias, accumulate) with the
// projection and bias folded into the prepared table Z[q][k] = w_out[q] .
// codebook[q][k] + b_out[q].  Per frame the work is n_q codes in and D floats
// out, but each output float needs n_q table reads: the on-chip gathers, not
// HBM, set the pace.  The table (33.6 MB at D=1024, Q=8) stays in L2; one row
// of threads per frame sums its float4 column of the n_q rows in stage order,
// so each warp instruction reads 512 contiguous bytes of one table row.
// With the codec's fc2 folded into Z (Z = fc2_w . stage output, D_out wide)
// the sum starts at fc2_b; without it, at zero.
//
// (A variant that staged 64 KB blocks of a slice-major copy of the table in
// shared memory by bulk copy measured slower on the 192 000-frame workload --
// 772 us against 502 us: with the table re-read once per 2048-frame block it
// still moves 16 KB per frame through L2, and its per-stage copies serialise.)
#include "rvq_internal.cuh"

namespace rvq {
namespace {

// One row of threads per frame; each thread sums one float4 column group.
__global__ void __launch_bounds__(256) k_decode_gather(const float4 *__restrict__ Z4, const float4 *__restrict__ b4,
                                                       const int32_t *__restrict__ codes, float4 *__restrict__ y4,
                                                       int64_t n_rows, int n_q, int K, int D4,
                                                       unsigned long long *__restrict__ bad) {
  const int64_t n = (int64_t)blockIdx.x * blockDim.y + threadIdx.y;
  int n_bad = 0;
  if (n < n_rows) {
    const int32_t *cn = codes + n * n_q;
    for (int c = threadIdx.x; c < D4; c += blockDim.x) {
      float4 acc = __ldg(b4 + c);
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

cudaError_t launch_decode(const rvq_dims &dm, const void *tables, const int32_t *codes, int64_t n, int n_q, float *y,
                          int64_t *bad, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  unsigned long long *bad_u = reinterpret_cast<unsigned long long *>(bad);
  const int D4 = dim_out(dm) / 4;
  const int tx = D4 >= 256 ? 256 : (D4 >= 128 ? 128 : (D4 >= 64 ? 64 : 32));
  const int fy = 256 / tx;
  k_decode_gather<<<(unsigned)((n + fy - 1) / fy), dim3(tx, fy), 0, st>>>(
      at<float4>(tables, L.z), at<float4>(tables, L.b_dec), codes, reinterpret_cast<float4 *>(y), n, n_q, dm.K, D4,
      bad_u);
  return cudaGetLastError();
}

}  // namespace rvq
