// RVQ encode, FP32 SIMT kernels.
//
// The encode loop of omnivoice.cpp ARCHITECTURE.md ("RVQ codec", Encode
// (residual loop)) is evaluated in the re-associated form prepared by
// rvq_prepare:
//
//   step 1  P0[n][q*d + j] = w_in[q][j] . x[n] + b_in[q][j]      for all q < n_q
//           (one GEMM over the frame dimension D for every stage at once)
//   step 2  for q = 0 .. n_q-1 (per frame):
//             p_q    = P0[n][q] - sum_{s<q} G[q][s][code_s]
//             code_q = argmin_k  ||c_k||^2 - 2 p_q . c_k           (lowest k on ties)
//
// ||p_q||^2 is common to every k and is dropped from the distance.  The
// D-dimensional residual is never materialised: G carries each earlier
// stage's contribution into stage q's code space.
#include <atomic>

#include "rvq_internal.cuh"

namespace rvq {
namespace {

// ---------------------------------------------------------------------------
// step 1: P0 = x . w_in^T + b_in   ("NT" SGEMM, 128 x 128 tiles, 8 x 8 per thread)
// ---------------------------------------------------------------------------
constexpr int P_BM = 128, P_BN = 128, P_BK = 16, P_PAD = 4;

__global__ void __launch_bounds__(256) k_project_simt(const float *__restrict__ x,
                                                      const float *__restrict__ w,
                                                      const float *__restrict__ bias,
                                                      float *__restrict__ P, int64_t n_rows,
                                                      int n_cols, int D) {
  __shared__ __align__(16) float As[2][P_BK][P_BM + P_PAD];
  __shared__ __align__(16) float Bs[2][P_BK][P_BN + P_PAD];
  const int tid = threadIdx.x;
  const int64_t m0 = (int64_t)blockIdx.x * P_BM;
  const int c0 = blockIdx.y * P_BN;
  // loader mapping: two float4 per operand per thread
  const int lr = tid >> 2, lk = (tid & 3) * 4;
  const float *a_src[2];
  const float *b_src[2];
  bool a_ok[2], b_ok[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int64_t r = m0 + lr + u * 64;
    a_ok[u] = r < n_rows;
    a_src[u] = x + (a_ok[u] ? r : 0) * (int64_t)D + lk;
    const int c = c0 + lr + u * 64;
    b_ok[u] = c < n_cols;
    b_src[u] = w + (int64_t)(b_ok[u] ? c : 0) * D + lk;
  }
  float4 ra[2], rb[2];
  auto gload = [&](int k0) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      ra[u] = a_ok[u] ? *reinterpret_cast<const float4 *>(a_src[u] + k0) : make_float4(0, 0, 0, 0);
      rb[u] = b_ok[u] ? *reinterpret_cast<const float4 *>(b_src[u] + k0) : make_float4(0, 0, 0, 0);
    }
  };
  auto sstore = [&](int buf) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = lr + u * 64;
      As[buf][lk + 0][r] = ra[u].x;
      As[buf][lk + 1][r] = ra[u].y;
      As[buf][lk + 2][r] = ra[u].z;
      As[buf][lk + 3][r] = ra[u].w;
      Bs[buf][lk + 0][r] = rb[u].x;
      Bs[buf][lk + 1][r] = rb[u].y;
      Bs[buf][lk + 2][r] = rb[u].z;
      Bs[buf][lk + 3][r] = rb[u].w;
    }
  };
  const int tr = tid >> 4, tc = tid & 15;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  gload(0);
  sstore(0);
  __syncthreads();
  const int nk = D / P_BK;
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) gload((kt + 1) * P_BK);
#pragma unroll
    for (int kk = 0; kk < P_BK; ++kk) {
      float a[8], b[8];
      *reinterpret_cast<float4 *>(&a[0]) = *reinterpret_cast<const float4 *>(&As[buf][kk][tr * 4]);
      *reinterpret_cast<float4 *>(&a[4]) = *reinterpret_cast<const float4 *>(&As[buf][kk][64 + tr * 4]);
      *reinterpret_cast<float4 *>(&b[0]) = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tc * 4]);
      *reinterpret_cast<float4 *>(&b[4]) = *reinterpret_cast<const float4 *>(&Bs[buf][kk][64 + tc * 4]);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (kt + 1 < nk) {
      sstore(buf ^ 1);
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = m0 + (i < 4 ? tr * 4 + i : 64 + tr * 4 + i - 4);
    if (r >= n_rows) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + h * 64 + tc * 4;
      if (c >= n_cols) continue;  // n_cols is a multiple of 64: whole float4 in or out
      float4 v = make_float4(acc[i][h * 4 + 0] + bias[c + 0], acc[i][h * 4 + 1] + bias[c + 1],
                             acc[i][h * 4 + 2] + bias[c + 2], acc[i][h * 4 + 3] + bias[c + 3]);
      *reinterpret_cast<float4 *>(P + r * (int64_t)n_cols + c) = v;
    }
  }
}

// ---------------------------------------------------------------------------
// step 2: the stage loop.  One CTA owns 64 frames for all n_q stages.
// 256 threads as 16 (ty) x 16 (tx): thread (ty, tx) scores frames 4ty..4ty+3
// against codewords 8tx..8tx+7 of each 128-entry chunk of the codebook.
// ---------------------------------------------------------------------------
constexpr int S_FR = 64;     // frames per CTA
constexpr int S_KC = 128;    // codewords per chunk

struct SearchSmem {
  float pT[kCodeDim][S_FR];     // -2 * p, code-space-major
  float cT[kCodeDim][S_KC];     // codebook chunk, code-space-major
  float cn[S_KC];
};

__global__ void __launch_bounds__(256) k_search_simt(const float *__restrict__ P0,
                                                     const float *__restrict__ G,
                                                     const float *__restrict__ cbT,
                                                     const float *__restrict__ cnorm,
                                                     int32_t *__restrict__ codes, int64_t n_rows,
                                                     int n_q, int K) {
  constexpr int d = kCodeDim;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SearchSmem &S = *reinterpret_cast<SearchSmem *>(smem_raw);
  int *codes_s = reinterpret_cast<int *>(smem_raw + sizeof(SearchSmem));  // [S_FR][n_q]
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int64_t f0 = (int64_t)blockIdx.x * S_FR;
  const int ld = n_q * d;

  for (int q = 0; q < n_q; ++q) {
    // ---- query tile: p_q = P0[n][q] - sum_{s<q} G[q][s][code_s]; store -2 p_q
    {
      const int f = tid >> 2, j0 = (tid & 3) * 16;
      const int64_t n = f0 + f;
      float p[16];
      if (n < n_rows) {
        const float *src = P0 + n * ld + q * d + j0;
#pragma unroll
        for (int u = 0; u < 4; ++u) *reinterpret_cast<float4 *>(&p[4 * u]) = reinterpret_cast<const float4 *>(src)[u];
        for (int s = 0; s < q; ++s) {
          const int c = codes_s[f * n_q + s];
          const float *gr = G + ((pair_index(q, s) * K) + c) * d + j0;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float4 g4 = reinterpret_cast<const float4 *>(gr)[u];
            p[4 * u + 0] -= g4.x;
            p[4 * u + 1] -= g4.y;
            p[4 * u + 2] -= g4.z;
            p[4 * u + 3] -= g4.w;
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) p[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) S.pT[j0 + u][f] = -2.0f * p[u];
    }
    float best_v[4];
    int best_k[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      best_v[i] = __int_as_float(0x7f800000);  // +inf
      best_k[i] = tx * 8;  // a valid index even if every distance is NaN (inputs must be finite)
    }
    const float *cbq = cbT + (int64_t)q * d * K;
    const float *cnq = cnorm + (int64_t)q * K;
    for (int k0 = 0; k0 < K; k0 += S_KC) {
      __syncthreads();  // previous chunk consumed (and query tile written)
      for (int e = tid; e < d * S_KC / 4; e += 256) {
        const int j = e / (S_KC / 4), c4 = e % (S_KC / 4);
        reinterpret_cast<float4 *>(&S.cT[j][0])[c4] =
            *reinterpret_cast<const float4 *>(cbq + (int64_t)j * K + k0 + c4 * 4);
      }
      if (tid < S_KC) S.cn[tid] = cnq[k0 + tid];
      __syncthreads();
      float acc[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[i][c] = 0.f;
#pragma unroll 8
      for (int j = 0; j < d; ++j) {
        const float4 a = *reinterpret_cast<const float4 *>(&S.pT[j][ty * 4]);
        const float4 b0 = *reinterpret_cast<const float4 *>(&S.cT[j][tx * 8]);
        const float4 b1 = *reinterpret_cast<const float4 *>(&S.cT[j][tx * 8 + 4]);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[i][c] = fmaf(av[i], bv[c], acc[i][c]);
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float cnv = S.cn[tx * 8 + c];
        const int k = k0 + tx * 8 + c;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float v = acc[i][c] + cnv;
          if (v < best_v[i]) {  // ascending k within the thread: strict '<' keeps the lowest
            best_v[i] = v;
            best_k[i] = k;
          }
        }
      }
    }
    // ---- lexicographic (value, index) minimum over the 16 tx lanes of each frame
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v = best_v[i];
      int k = best_k[i];
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int ok = __shfl_xor_sync(0xffffffffu, k, o);
        if (ov < v || (ov == v && ok < k)) {
          v = ov;
          k = ok;
        }
      }
      if (tx == 0) {
        const int f = ty * 4 + i;
        codes_s[f * n_q + q] = k;
        const int64_t n = f0 + f;
        if (n < n_rows) codes[n * n_q + q] = k;
      }
    }
    __syncthreads();  // codes_s visible before the next query tile
  }
}

}  // namespace

size_t search_smem_bytes(int n_q) { return sizeof(SearchSmem) + (size_t)S_FR * n_q * sizeof(int); }

cudaError_t launch_encode_chunk(const rvq_dims &dm, const void *tables, const float *x, int64_t n0,
                                int64_t n, int n_q, int32_t *codes, float *p0, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  const int D = dm.D, d = dm.d, K = dm.K;
  const int n_cols = n_q * d;
  dim3 g1((unsigned)((n + P_BM - 1) / P_BM), (unsigned)((n_cols + P_BN - 1) / P_BN));
  k_project_simt<<<g1, 256, 0, st>>>(x + n0 * D, at<float>(tables, L.w_in), at<float>(tables, L.b_in), p0, n,
                                     n_cols, D);
  const size_t smem = search_smem_bytes(n_q);
  // the shared-memory opt-in is a per-device property of the function
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    e = cudaFuncSetAttribute(k_search_simt, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)search_smem_bytes(kMaxStages));
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit);
  }
  k_search_simt<<<(unsigned)((n + S_FR - 1) / S_FR), 256, smem, st>>>(
      p0, at<float>(tables, L.g), at<float>(tables, L.cbT), at<float>(tables, L.cnorm), codes + n0 * n_q, n, n_q,
      K);
  return cudaGetLastError();
}

}  // namespace rvq
