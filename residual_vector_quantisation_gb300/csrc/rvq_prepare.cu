// Table preparation: everything encode and decode read besides the frames.
//
// All sums run in float64 and are rounded once to float32, so each table
// entry is the correctly rounded value of its exact-arithmetic definition up
// to float64 summation error (about 1e-16 relative).
//
//   cnorm[q][k]   = ||codebook[q][k]||^2        (cosine metric: ||c / n(c)||^2,
//                                               n(c) = max(||c||_2, 1e-12))
//   Z[q][k]       = w_out[q] . codebook[q][k] + b_out[q]         (decode table)
//   G[q][s][k]    = w_in[q] . Z[s][k]            for s < q      (cross-stage table)
//
// With the codec's Linear layers (omnivoice.cpp ARCHITECTURE.md, "Audio
// tokenizer": fc before the RVQ encode, fc2 after the RVQ decode):
//   w_in'[q] = w_in[q] . fc_w,  b_in'[q] = w_in[q] . fc_b + b_in[q]   (projection of raw frames)
//   Z'[q][k] = fc2_w . Z[q][k]  (so the decode table is D_out wide), decode bias fc2_b
// while G stays in the quantizer's own space.
//
// Z re-associates the decode graph of omnivoice.cpp ARCHITECTURE.md ("RVQ
// codec": gather, project_out, add bias, accumulate) into one gather per
// stage.  G re-associates the encode loop of the same section: since
// residual_q = x - sum_{s<q} Z[s][code_s], the stage-q projection is
// w_in[q] . x + b_in[q] - sum_{s<q} G[q][s][code_s].
#include "rvq_internal.cuh"
#include "sm103_ptx.cuh"

namespace rvq {
namespace {

__device__ __forceinline__ float tf32_trunc(float v) {
  return __uint_as_float(__float_as_uint(v) & 0xffffe000u);
}

// w_in TF32 hi / lo split and b_in.
__global__ void k_prep_w_in(const float *__restrict__ w_in, const float *__restrict__ b_in, float *__restrict__ hi,
                            float *__restrict__ lo, float *__restrict__ b_in_copy, int64_t n, int64_t nb) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = i; e < n; e += stride) {
    float v = w_in[e];
    float h = tf32_trunc(v);
    hi[e] = h;
    lo[e] = v - h;
  }
  for (int64_t e = i; e < nb; e += stride) b_in_copy[e] = b_in ? b_in[e] : 0.0f;
}

// n(c) = max(||c||_2, 1e-12) of one codeword (float64), the divisor of the
// cosine metric (moss-tts.cpp AGENTS.md, gotcha 9); 1 for the plain metric.
__device__ __forceinline__ double codeword_divisor(const float *c, int d, int metric) {
  if (metric != RVQ_METRIC_COSINE) return 1.0;
  double s = 0.0;
  for (int j = 0; j < d; ++j) s += (double)c[j] * (double)c[j];
  return fmax(sqrt(s), 1e-12);
}

// w_in' = w_in . fc_w (float64 sums), split into TF32 hi / lo, and
// b_in' = w_in . fc_b + b_in.  grid: (Q*d, ceil(D_in/256)); 256 threads.
__global__ void __launch_bounds__(256) k_prep_w_in_fc(const float *__restrict__ w_in, const float *__restrict__ b_in,
                                                      const float *__restrict__ fc_w, const float *__restrict__ fc_b,
                                                      float *__restrict__ hi, float *__restrict__ lo,
                                                      float *__restrict__ b_in_out, int D, int D_in) {
  const int64_t r = blockIdx.x;  // row q*d + j
  const int i = blockIdx.y * blockDim.x + threadIdx.x;
  const float *wr = w_in + r * D;
  if (i < D_in) {
    double s = 0.0;
    for (int m = 0; m < D; ++m) s += (double)wr[m] * (double)fc_w[(int64_t)m * D_in + i];
    const float v = (float)s;
    const float h = tf32_trunc(v);
    hi[r * D_in + i] = h;
    lo[r * D_in + i] = v - h;
  }
  if (blockIdx.y == 0 && threadIdx.x < 32) {  // the bias, one warp
    double s = 0.0;
    if (fc_b)
      for (int m = threadIdx.x; m < D; m += 32) s += (double)wr[m] * (double)fc_b[m];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) b_in_out[r] = (float)(s + (b_in ? (double)b_in[r] : 0.0));
  }
}

// fc2 folded into the stage outputs: M2[q][o][j] = sum_i fc2_w[o][i] w_out[q][i][j],
// v2[q][o] = sum_i fc2_w[o][i] b_out[q][i] (float64).  grid: (Q, D_out); block: d + 32.
template <int d>
__global__ void k_prep_m2(const float *__restrict__ fc2_w, const float *__restrict__ w_out,
                          const float *__restrict__ b_out, double *__restrict__ m2, double *__restrict__ v2, int D,
                          int D_out) {
  const int q = blockIdx.x, o = blockIdx.y;
  const float *fr = fc2_w + (int64_t)o * D;
  constexpr int kJThreads = (d + 31) / 32 * 32;
  if (threadIdx.x < kJThreads) {
    const int j = threadIdx.x;
    if (j >= d) return;
    const float *wo = w_out + (int64_t)q * D * d + j;
    double acc = 0.0;
    for (int i = 0; i < D; ++i) acc += (double)fr[i] * (double)wo[(int64_t)i * d];
    m2[((int64_t)q * D_out + o) * d + j] = acc;
  } else {
    const int lane = threadIdx.x - kJThreads;  // one whole warp
    double acc = 0.0;
    if (b_out)
      for (int i = lane; i < D; i += 32) acc += (double)fr[i] * (double)b_out[(int64_t)q * D + i];
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) v2[(int64_t)q * D_out + o] = acc;
  }
}

// The streaming path's tables: w_in' in float32 (hi + lo, exact), and the
// codebook (normalised for the cosine metric) cut into CS slices of kc = K/CS
// codewords, each slice stored [j/4][kk] in float4 units.
__global__ void k_prep_w_in_f(const float *__restrict__ hi, const float *__restrict__ lo, float *__restrict__ wf,
                              int64_t n) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e < n) wf[e] = hi[e] + lo[e];
}

__global__ void k_prep_cb_stream(const float *__restrict__ cb, float *__restrict__ out, int d, int K, int CS,
                                 int64_t n, int metric) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // over Q*K*d, output order
  if (e >= n) return;
  const int kc = K / CS, n4 = d / 4;
  const int c = (int)(e % 4);
  int64_t r = e / 4;
  const int kk = (int)(r % kc);
  r /= kc;
  const int jb = (int)(r % n4);
  r /= n4;
  const int rank = (int)(r % CS);
  const int64_t q = r / CS;
  const int64_t row = q * K + (int64_t)rank * kc + kk;
  out[e] = (float)((double)cb[row * d + 4 * jb + c] / codeword_divisor(cb + row * d, d, metric));
}

// The decode bias: fc2_b, or zeros; and whether decode needs to add it.
__global__ void k_prep_b_dec(const float *__restrict__ fc2_b, float *__restrict__ b_dec, int D_out,
                             int *__restrict__ b_dec_used) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < D_out) b_dec[i] = fc2_b ? fc2_b[i] : 0.0f;
  if (i == 0) *b_dec_used = fc2_b ? 1 : 0;
}

// Squared norms of the codewords as the distance uses them (float64 sums).
__global__ void k_prep_cnorm(const float *__restrict__ cb, float *__restrict__ cnorm, int d, int64_t n_rows,
                             int metric) {
  int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // row = q*K + k
  if (r >= n_rows) return;
  const float *src = cb + r * d;
  const double nrm = codeword_divisor(src, d, metric);
  double s = 0.0;
  for (int j = 0; j < d; ++j) {
    const double v = (double)src[j] / nrm;
    s += v * v;
  }
  cnorm[r] = (float)s;
}

// -2 * codebook (each codeword divided by n(c) first for the cosine metric)
// in TF32 hi/lo halves, laid out as the shared-memory image the tensor-core
// search loads with one bulk copy per half chunk:
// [q][chunk of 128][hi, lo][atom j/32][sw128(row = k % 128, j % 32)].
__global__ void k_prep_cb_img(const float *__restrict__ cb, float *__restrict__ img, int K, int64_t n, int metric) {
  constexpr int d = kCodeDim;
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // over Q*K*d
  if (e >= n) return;
  const int j = (int)(e % d);
  const int64_t qk = e / d;
  const int q = (int)(qk / K), k = (int)(qk % K);
  const int c = k / kChunkCodes, kk = k % kChunkCodes;
  const float v = (float)(-2.0 * (double)cb[e] / codeword_divisor(cb + qk * d, d, metric));
  const float hi = tf32_trunc(v);
  const float lo = v - hi;
  const int64_t chunk = ((int64_t)q * (K / kChunkCodes) + c) * 2;
  const uint32_t off = ptx::sw128_offset(kk, j & 31) / 4 + (j >> 5) * (128 * 32);
  img[(chunk + 0) * (2 * 128 * 32) + off] = hi;
  img[(chunk + 1) * (2 * 128 * 32) + off] = lo;
}

// The same for d = 8: [q][chunk of 128][hi, lo][sw32(row = k % 128, j)], a
// 4 KB block per half; a stage's chunks are contiguous, so one bulk copy
// brings a whole stage.
__global__ void k_prep_cb_img8(const float *__restrict__ cb, float *__restrict__ img, int K, int64_t n, int metric) {
  constexpr int d = kCodeDimSmall;
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // over Q*K*d
  if (e >= n) return;
  const int j = (int)(e % d);
  const int64_t qk = e / d;
  const int q = (int)(qk / K), k = (int)(qk % K);
  const int c = k / kChunkCodes, kk = k % kChunkCodes;
  const float v = (float)(-2.0 * (double)cb[e] / codeword_divisor(cb + qk * d, d, metric));
  const float hi = tf32_trunc(v);
  const float lo = v - hi;
  const int64_t chunk = ((int64_t)q * (K / kChunkCodes) + c) * 2;
  const uint32_t off = ptx::sw32_offset(kk, j) / 4;
  img[(chunk + 0) * (128 * d) + off] = hi;
  img[(chunk + 1) * (128 * d) + off] = lo;
}

// The d = 8 search's norm operand: ||c||^2 (as rounded once into cnorm) split
// into three TF32 parts n1 = tf32(n), n2 = tf32(n - n1), n3 = n - n1 - n2,
// whose sum is n exactly, in the sw32 layout of a 128 x 8 B block:
// [q][chunk pair][sw32(row = k % 128, slot)], slots 0-2 for the even chunk of
// the pair and 4-6 for the odd one, zeros elsewhere.  An MMA of this block
// with A rows [1 1 1 0 0 0 0 0] (even) or [0 0 0 0 1 1 1 0] (odd) adds the
// chunk's norms to its distances.
__global__ void k_prep_cn_img8(const float *__restrict__ cnorm, float *__restrict__ img, int K, int64_t n) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // over Q * blocks * 128 * 8
  if (e >= n) return;
  const int slot = (int)(e & 7), kk = (int)((e >> 3) & 127);
  const int64_t qb = e >> 10;  // q * blocks + pair
  const int64_t blocks = (int64_t)cn_img8_blocks(K);
  const int q = (int)(qb / blocks), pair = (int)(qb % blocks);
  const int c = 2 * pair + (slot >> 2);  // chunk
  float v = 0.0f;
  if ((slot & 3) < 3 && c < K / kChunkCodes) {
    const float nrm = cnorm[(int64_t)q * K + c * kChunkCodes + kk];
    const float n1 = tf32_trunc(nrm);
    const float n2 = tf32_trunc(nrm - n1);
    const float n3 = (nrm - n1) - n2;
    v = (slot & 3) == 0 ? n1 : (slot & 3) == 1 ? n2 : n3;
  }
  img[qb * (128 * 8) + ptx::sw32_offset(kk, slot) / 4] = v;
}

// Z[q][k][i] = sum_j w_out[q][i][j] codebook[q][k][j] + b_out[q][i]  (f64);
// with fc2 the same with M2, v2 of width D_out for w_out, b_out.
// grid: (ceil(D/256), Q*K/16); each block handles 16 codewords of one stage.
template <int d, class TW>
__global__ void __launch_bounds__(256) k_prep_z(const TW *__restrict__ w_out,
                                                const TW *__restrict__ b_out,
                                                const float *__restrict__ cb, float *__restrict__ z,
                                                int D, int K) {
  __shared__ double sc[16][d];
  const int64_t row0 = (int64_t)blockIdx.y * 16;  // q*K + k0
  const int q = (int)(row0 / K);
  for (int e = threadIdx.x; e < 16 * d; e += blockDim.x)
    sc[e / d][e % d] = (double)cb[(row0 + e / d) * d + e % d];
  __syncthreads();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= D) return;
  const TW *wr = w_out + ((int64_t)q * D + i) * d;
  double w[d];
#pragma unroll
  for (int j = 0; j < d; ++j) w[j] = (double)wr[j];
  const double bias = b_out ? (double)b_out[(int64_t)q * D + i] : 0.0;
  for (int kk = 0; kk < 16; ++kk) {
    double s = 0.0;
#pragma unroll
    for (int j = 0; j < d; ++j) s += w[j] * sc[kk][j];
    z[(row0 + kk) * D + i] = (float)(s + bias);
  }
}

// M[t][j][m] = sum_i w_in[q][j][i] w_out[s][i][m];  vb[t][j] = sum_i w_in[q][j][i] b_out[s][i].
// grid: (P, d); block: d threads (one per m), rounded up to whole warps, plus
// one warp for vb.
template <int d>
__global__ void k_prep_m(const float *__restrict__ w_in, const float *__restrict__ w_out,
                         const float *__restrict__ b_out, double *__restrict__ m64,
                         double *__restrict__ vb64, int D, int Q) {
  const int t = blockIdx.x, j = blockIdx.y;
  int q = 1;
  while ((int64_t)(q + 1) * q / 2 <= t) ++q;  // t = q(q-1)/2 + s
  const int s = t - q * (q - 1) / 2;
  const float *wi = w_in + ((int64_t)q * d + j) * D;
  constexpr int kMThreads = (d + 31) / 32 * 32;
  if (threadIdx.x < kMThreads) {
    const int m = threadIdx.x;
    if (m >= d) return;
    const float *wo = w_out + (int64_t)s * D * d + m;
    double acc = 0.0;
    for (int i = 0; i < D; ++i) acc += (double)wi[i] * (double)wo[(int64_t)i * d];
    m64[((int64_t)t * d + j) * d + m] = acc;
  } else {
    const int lane = threadIdx.x - kMThreads;  // one whole warp
    double acc = 0.0;
    if (b_out)
      for (int i = lane; i < D; i += 32) acc += (double)wi[i] * (double)b_out[(int64_t)s * D + i];
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) vb64[(int64_t)t * d + j] = acc;
  }
  (void)Q;
}

// G[t][k][j] = sum_m M[t][j][m] codebook[s][k][m] + vb[t][j]   (f64 -> f32).
// grid: (P, K/16); 256 threads = 16 codewords x 16 groups of d/16 j.
template <int d>
__global__ void __launch_bounds__(256) k_prep_g(const double *__restrict__ m64,
                                                const double *__restrict__ vb64,
                                                const float *__restrict__ cb, float *__restrict__ g,
                                                int K) {
  __shared__ double sm[d][d + 1];
  __shared__ double sc[16][d];
  const int t = blockIdx.x;
  int q = 1;
  while ((int64_t)(q + 1) * q / 2 <= t) ++q;
  const int s = t - q * (q - 1) / 2;
  const int k0 = blockIdx.y * 16;
  for (int e = threadIdx.x; e < d * d; e += blockDim.x) sm[e / d][e % d] = m64[(int64_t)t * d * d + e];
  for (int e = threadIdx.x; e < 16 * d; e += blockDim.x)
    sc[e / d][e % d] = (double)cb[(((int64_t)s * K) + k0 + e / d) * d + e % d];
  __syncthreads();
  const int kk = threadIdx.x / 16, jg = threadIdx.x % 16;
  for (int u = 0; u < (d + 15) / 16; ++u) {
    const int j = jg * ((d + 15) / 16) + u;
    if (j >= d) break;
    double acc = vb64[(int64_t)t * d + j];
    for (int m = 0; m < d; ++m) acc += sm[j][m] * sc[kk][m];
    g[(((int64_t)t * K) + k0 + kk) * d + j] = (float)acc;
  }
}

}  // namespace

template <int d>
void launch_tables(const rvq_dims &dm, const rvq_weights &w, void *tables, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  const int D = dm.D, K = dm.K, Q = dm.Q;
  const int64_t rows = (int64_t)Q * K, P = n_pairs(Q);
  const int D_out = dim_out(dm);
  if (w.fc2_w) {
    double *m2 = at<double>(tables, L.m2_64), *v2 = m2 + (size_t)Q * D_out * d;
    k_prep_m2<d><<<dim3((unsigned)Q, (unsigned)D_out), (d + 31) / 32 * 32 + 32, 0, st>>>(w.fc2_w, w.w_out, w.b_out, m2,
                                                                                         v2, D, D_out);
    k_prep_z<d, double><<<dim3((D_out + 255) / 256, (unsigned)(rows / 16)), 256, 0, st>>>(
        m2, v2, w.codebook, at<float>(tables, L.z), D_out, K);
  } else {
    k_prep_z<d, float><<<dim3((D + 255) / 256, (unsigned)(rows / 16)), 256, 0, st>>>(w.w_out, w.b_out, w.codebook,
                                                                                     at<float>(tables, L.z), D, K);
  }
  k_prep_b_dec<<<(D_out + 255) / 256, 256, 0, st>>>(w.fc2_b, at<float>(tables, L.b_dec), D_out,
                                                     at<int>(tables, L.b_dec_used));
  if (P > 0) {
    k_prep_m<d><<<dim3((unsigned)P, d), (d + 31) / 32 * 32 + 32, 0, st>>>(w.w_in, w.w_out, w.b_out, at<double>(tables, L.m64),
                                                         at<double>(tables, L.vb64), D, Q);
    k_prep_g<d><<<dim3((unsigned)P, K / 16), 256, 0, st>>>(at<double>(tables, L.m64), at<double>(tables, L.vb64),
                                                           w.codebook, at<float>(tables, L.g), K);
  }
}

cudaError_t launch_prepare(const rvq_dims &dm, const rvq_weights &w, void *tables, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  const int D = dm.D, d = dm.d, K = dm.K, Q = dm.Q;
  if (w.fc_w) {
    const int D_in = dim_in(dm);
    k_prep_w_in_fc<<<dim3((unsigned)(Q * d), (unsigned)((D_in + 255) / 256)), 256, 0, st>>>(
        w.w_in, w.b_in, w.fc_w, w.fc_b, at<float>(tables, L.w_in_hi), at<float>(tables, L.w_in_lo),
        at<float>(tables, L.b_in), D, D_in);
  } else {
    const int64_t nw = (int64_t)Q * d * D;
    k_prep_w_in<<<608, 256, 0, st>>>(w.w_in, w.b_in, at<float>(tables, L.w_in_hi), at<float>(tables, L.w_in_lo),
                                     at<float>(tables, L.b_in), nw, (int64_t)Q * d);
  }
  if (stream_tables(dm)) {  // the streaming path's copies: w_in' in float32, the sliced (normalised) codebook
    const int D_in = dim_in(dm);
    const int64_t nt = (int64_t)Q * D_in * d, nc = (int64_t)Q * K * d;
    k_prep_w_in_f<<<(unsigned)((nt + 255) / 256), 256, 0, st>>>(at<float>(tables, L.w_in_hi),
                                                                  at<float>(tables, L.w_in_lo),
                                                                  at<float>(tables, L.w_in_f), nt);
    k_prep_cb_stream<<<(unsigned)((nc + 255) / 256), 256, 0, st>>>(w.codebook, at<float>(tables, L.cb_stream), d, K,
                                                                     stream_cluster_size(K), nc, dm.metric);
  }
  const int64_t rows = (int64_t)Q * K;
  k_prep_cnorm<<<(unsigned)((rows + 255) / 256), 256, 0, st>>>(w.codebook, at<float>(tables, L.cnorm), d, rows,
                                                               dm.metric);
  const int64_t ncb = (int64_t)Q * K * d;
  if (d == kCodeDim) {
    k_prep_cb_img<<<(unsigned)((ncb + 255) / 256), 256, 0, st>>>(w.codebook, at<float>(tables, L.cb_img), K, ncb,
                                                                 dm.metric);
    launch_tables<kCodeDim>(dm, w, tables, st);
  } else {
    k_prep_cb_img8<<<(unsigned)((ncb + 255) / 256), 256, 0, st>>>(w.codebook, at<float>(tables, L.cb_img), K, ncb,
                                                                  dm.metric);
    const int64_t nn = (int64_t)Q * (int64_t)cn_img8_blocks(K) * 128 * 8;
    k_prep_cn_img8<<<(unsigned)((nn + 255) / 256), 256, 0, st>>>(at<float>(tables, L.cnorm),
                                                                  at<float>(tables, L.cn_img8), K, nn);
    launch_tables<kCodeDimSmall>(dm, w, tables, st);
  }
  return cudaGetLastError();
}

}  // namespace rvq
