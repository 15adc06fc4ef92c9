// Low-latency RVQ encode of small batches: the streaming path.
//
// Realtime callers encode a few frames at a time: omnivoice.cpp
// ARCHITECTURE.md ("CLI tools", omnivoice-tts) starts synthesis from stdin as
// soon as the first sentence is complete, and moss-tts.cpp AGENTS.md has a
// realtime TTS front end.  For such calls the tile path (128-frame tiles, one
// CTA per tile walking all K codewords of every stage) leaves the GPU idle
// and its latency is the serial walk over Q*K codewords.  Here each group of
// up to 16 frames runs on one thread-block cluster of CS = min(8, K/128) CTAs,
// CTA r owning codewords [r*kc, (r+1)*kc), kc = K/CS, of every stage:
//
//   projection  CTA r computes P0[q] = w_in'[q] . x + b_in'[q] for its stages
//               q = r, r+CS, ... (float32 FMA, the sum over D_in split over
//               thread groups) and stores it into the shared memory of every
//               CTA of the cluster; a cluster barrier publishes them.
//   stage q     each CTA scores its slice (staged in shared memory by a bulk
//               copy issued NB stages ahead) against the frames' p_q:
//               dist = ||c||^2 - 2 s p.c  (s = 1, or 1/max(||p||, 1e-12) for
//               the cosine metric), keeping per frame the minimum of the key
//               (distance, index); the CS keys of each frame are exchanged
//               through distributed shared memory (remote stores, then one
//               release-arrive per source on the destination's mbarrier); the
//               smallest key is the code -- distance first, then the lowest
//               index, as the plain argmin of the pages.
//   update      p_{q+1} -= G[q+1][q][code_q] right after the exchange (the
//               cross-stage table of rvq_prepare); the terms for later stages
//               are applied while the next exchange is in flight.
//
// The distances are float32 FMA dot products on the CUDA cores, not tensor
// core tiles: with at most 16 frames a stage is a [kc x d] by [d x 16] product
// per CTA, far below one tcgen05 tile, and the path is bound by the exchange
// and gather latencies, not by arithmetic.
//
// Every mbarrier wait is bounded: a timeout records RVQ_DEVICE_TIMEOUT in the
// status word and the kernel carries on (codes are clamped to [0, K), so no
// access leaves its buffer); every CTA reaches the closing cluster barrier.
#include <atomic>

#include "rvq_internal.cuh"
#include "sm103_ptx.cuh"

namespace rvq {
namespace {

using namespace ptx;

constexpr int ST_THREADS = 256;
constexpr int ST_F = kStreamFrames;            // frames per cluster
constexpr int ST_MAX_CS = 8;                    // cluster size limit (portable)
constexpr uint32_t ST_SMEM_LIMIT = 232448;      // opt-in dynamic shared memory per block
constexpr int ST_BATCH = 8;                     // table rows in flight per thread in the deferred update

// Dynamic shared memory layout (byte offsets), the same on host and device.
struct StreamShape {
  int CS, kc, NB, slots;
  uint32_t p, cbuf, cnb, red, xch, loc, cs, sv, bars, total;
};

__host__ __device__ inline uint32_t up16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline StreamShape stream_shape(int d, int K, int n_q, int NB) {
  StreamShape S{};
  S.CS = stream_cluster_size(K);
  S.kc = K / S.CS;
  S.NB = NB;
  S.slots = S.kc == 128 ? 128 : 256;  // key-writing threads per frame
  uint32_t o = 0;
  S.p = o;    o = up16(o + (uint32_t)n_q * ST_F * d * 4);                 // [n_q][F][d] stage projections
  o = (o + 127u) & ~127u;
  S.cbuf = o; o = up16(o + (uint32_t)NB * S.kc * d * 4);                  // [NB][d/4][kc] float4 slices
  S.cnb = o;  o = up16(o + (uint32_t)NB * S.kc * 4);                      // [NB][kc] squared norms
  const uint32_t red_keys = (uint32_t)ST_F * S.slots * 8, red_proj = ST_THREADS * 16 * 4;
  S.red = o;  o = up16(o + (red_keys > red_proj ? red_keys : red_proj));  // keys / projection partials
  S.xch = o;  o = up16(o + 2u * ST_MAX_CS * ST_F * 8);                   // [2][rank][F] exchanged keys
  S.loc = o;  o = up16(o + ST_F * 8);                                     // [F] this CTA's best keys
  S.cs = o;   o = up16(o + 2u * ST_F * 4);                                // [2][F] codes of the last stages
  S.sv = o;   o = up16(o + ST_F * 4);                                     // [F] distance scale s
  S.bars = o; o = up16(o + 4u * 8);                                       // cb_full[2], x_full[2]
  S.total = o;
  return S;
}

// Buffers for the codebook slices: 2 when two fit, else 1 (0: the shape does not fit).
int stream_nb(int d, int K, int n_q) {
  if (stream_shape(d, K, n_q, 2).total <= ST_SMEM_LIMIT) return 2;
  if (stream_shape(d, K, n_q, 1).total <= ST_SMEM_LIMIT) return 1;
  return 0;
}

__device__ __forceinline__ void st_error(int *status, int code) { atomicCAS(status, 0, code); }

// Order key of (distance, index): smaller distance first, then lower index.
// The float is mapped to an unsigned integer of the same order (-0 taken as
// +0, NaN after every number).
__device__ __forceinline__ uint64_t dist_key(float v, uint32_t k) {
  uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  if (v != v) b = 0xffffffffu;
  return ((uint64_t)b << 32) | k;
}

__device__ __forceinline__ uint64_t min_u64(uint64_t a, uint64_t b) { return a < b ? a : b; }

__device__ __forceinline__ void sub4(float4 &p, const float4 g) {
  p.x -= g.x;
  p.y -= g.y;
  p.z -= g.z;
  p.w -= g.w;
}

// x [n][D_in] (frames of this call), codes [n][n_q].  grid: CS * ceil(n/16)
// CTAs in clusters of CS; ST_THREADS threads.  SPLITJ: threads per codeword
// (2 when kc == 128, each taking every other float4 column).
template <int d, int SPLITJ>
__global__ void __launch_bounds__(ST_THREADS, 1)
    k_encode_stream(const float *__restrict__ x, const float4 *__restrict__ w_t, const float4 *__restrict__ b_in,
                    const float4 *__restrict__ cb_s, const float *__restrict__ cnorm, const float4 *__restrict__ g,
                    int32_t *__restrict__ codes, int64_t n, int D_in, int K, int n_q, int NB, int metric,
                    int *__restrict__ status) {
  constexpr int TPF = d / 4;            // float4 columns of a row of d
  constexpr int DJ4 = TPF / SPLITJ;     // float4 columns of a codeword per thread
  extern __shared__ __align__(128) unsigned char smem[];
  const StreamShape S = stream_shape(d, K, n_q, NB);
  const int t = threadIdx.x;
  const int CS = S.CS, kc = S.kc;
  if (cluster_nctarank() != (uint32_t)CS || blockDim.x != ST_THREADS || dynamic_smem_size() < S.total ||
      (SPLITJ == 2) != (kc == 128) || (NB != 1 && NB != 2)) {
    if (t == 0) st_error(status, RVQ_DEVICE_BAD_LAUNCH);
    return;  // uniform over the cluster: no CTA reaches a cluster barrier
  }
  const uint32_t rank = cluster_ctarank();
  const int64_t f0 = (int64_t)(blockIdx.x / CS) * ST_F;
  const int nf = (int)(n - f0 < ST_F ? n - f0 : ST_F);

  float4 *P = reinterpret_cast<float4 *>(smem + S.p);          // [n_q][F][TPF]
  float4 *cbuf = reinterpret_cast<float4 *>(smem + S.cbuf);    // [NB][TPF][kc]
  float *cnb = reinterpret_cast<float *>(smem + S.cnb);        // [NB][kc]
  uint64_t *red = reinterpret_cast<uint64_t *>(smem + S.red);  // [F][slots]
  uint64_t *xch = reinterpret_cast<uint64_t *>(smem + S.xch);  // [2][ST_MAX_CS][F]
  uint64_t *loc = reinterpret_cast<uint64_t *>(smem + S.loc);  // [F]
  int *csm = reinterpret_cast<int *>(smem + S.cs);             // [2][F]
  float *sv = reinterpret_cast<float *>(smem + S.sv);          // [F]
  uint64_t *cb_full = reinterpret_cast<uint64_t *>(smem + S.bars);
  uint64_t *x_full = cb_full + 2;

  const uint32_t slice_bytes = (uint32_t)kc * d * 4, norm_bytes = (uint32_t)kc * 4;
  auto issue = [&](int q, int b) {  // one thread: stage q's slice into buffer b
    mbar_arrive_expect_tx(&cb_full[b], slice_bytes + norm_bytes);
    bulk_g2s(cbuf + (size_t)b * TPF * kc, cb_s + ((int64_t)q * CS + rank) * TPF * kc, slice_bytes, &cb_full[b]);
    bulk_g2s(cnb + (size_t)b * kc, cnorm + (int64_t)q * K + (int64_t)rank * kc, norm_bytes, &cb_full[b]);
  };

  if (t == 0) {
    for (int b = 0; b < NB; ++b) mbar_init(&cb_full[b], 1);
    mbar_init(&x_full[0], (uint32_t)CS);
    mbar_init(&x_full[1], (uint32_t)CS);
    fence_mbar_init();
  }
  if (t < ST_F) sv[t] = 1.0f;
  __syncthreads();
  cluster_arrive();  // barriers initialised; waited for before the first remote access
  if (t == 32)
    for (int q = 0; q < NB && q < n_q; ++q) issue(q, q);

  // ---- projection of this CTA's stages, stored into every CTA's P ----------
  {
    const int nfe = nf <= 4 ? 4 : (nf <= 8 ? 8 : 16);  // frames computed, whole blocks of 4
    const int TG = (nfe / 4) * TPF;                    // threads per slice of D_in
    const int KG = ST_THREADS / TG;                    // slices of D_in
    const int gi = t / TG, tg = t % TG, fb = tg / TPF, jb = tg % TPF;
    const float *xr[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int f = 4 * fb + v < nf ? 4 * fb + v : nf - 1;  // padding rows repeat a real frame
      xr[v] = x + (f0 + f) * (int64_t)D_in;
    }
    float4 *part = reinterpret_cast<float4 *>(red);  // [KG][nfe][TPF]
    bool joined = false;
    for (int q = (int)rank; q < n_q; q += CS) {
      float acc[4][4] = {};
      const float4 *wq = w_t + (int64_t)q * D_in * TPF + jb;
      for (int i = 4 * gi; i < D_in; i += 4 * KG) {
        float4 xv[4], wv[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) xv[v] = __ldg(reinterpret_cast<const float4 *>(xr[v] + i));
#pragma unroll
        for (int u = 0; u < 4; ++u) wv[u] = __ldg(wq + (int64_t)(i + u) * TPF);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float xs[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[v][0] = fmaf(xs[u], wv[u].x, acc[v][0]);
            acc[v][1] = fmaf(xs[u], wv[u].y, acc[v][1]);
            acc[v][2] = fmaf(xs[u], wv[u].z, acc[v][2]);
            acc[v][3] = fmaf(xs[u], wv[u].w, acc[v][3]);
          }
        }
      }
#pragma unroll
      for (int v = 0; v < 4; ++v)
        part[(gi * nfe + 4 * fb + v) * TPF + jb] = make_float4(acc[v][0], acc[v][1], acc[v][2], acc[v][3]);
      __syncthreads();
      if (!joined) {
        cluster_wait();
        joined = true;
      }
      for (int e = t; e < nfe * TPF; e += ST_THREADS) {
        const int f = e / TPF, j4 = e % TPF;
        float4 s = __ldg(b_in + q * TPF + j4);
        for (int k = 0; k < KG; ++k) {
          const float4 v = part[(k * nfe + f) * TPF + j4];
          s.x += v.x;
          s.y += v.y;
          s.z += v.z;
          s.w += v.w;
        }
        const uint32_t off = smem_addr(P + ((int64_t)q * ST_F + f) * TPF + j4);
        for (int r = 0; r < CS; ++r) st_cluster_v4(cluster_map(off, (uint32_t)r), s);
      }
      __syncthreads();
    }
    if (!joined) cluster_wait();
  }
  cluster_sync_all();  // every stage projection is in every CTA

  if (metric == RVQ_METRIC_COSINE && t < ST_F * TPF) {  // s of stage 0
    const int f = t / TPF, j4 = t % TPF;
    const float4 v = P[f * TPF + j4];
    float ss = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
    for (int o = TPF / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (j4 == 0) sv[f] = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
  }
  __syncthreads();

  // ---- the stage loop -------------------------------------------------------
  const int h = SPLITJ == 2 ? (t & 1) : 0;
  const int kk0 = SPLITJ == 2 ? (t >> 1) : t;
  for (int q = 0; q < n_q; ++q) {
    const int b = NB == 2 ? (q & 1) : 0;
    if (!mbar_wait(&cb_full[b], (uint32_t)((NB == 2 ? q >> 1 : q) & 1))) st_error(status, RVQ_DEVICE_TIMEOUT);

    // distances of this CTA's slice; per frame the smallest key
    uint64_t best[ST_F];
#pragma unroll
    for (int f = 0; f < ST_F; ++f) best[f] = ~0ull;
    {
      const float4 *cq = cbuf + (size_t)b * TPF * kc;
      const float *cnq = cnb + (size_t)b * kc;
      const float4 *pq = P + (int64_t)q * ST_F * TPF;
      for (int kk = kk0; kk < kc; kk += ST_THREADS / SPLITJ) {
        float4 c[DJ4];
#pragma unroll
        for (int m = 0; m < DJ4; ++m) c[m] = cq[(m * SPLITJ + h) * kc + kk];
        const float cn = cnq[kk];
        const uint32_t kg = rank * (uint32_t)kc + (uint32_t)kk;
#pragma unroll
        for (int f = 0; f < ST_F; ++f) {
          if (f < nf) {
            const float4 *pf = pq + f * TPF + h;
            float a = 0.0f;
#pragma unroll
            for (int m = 0; m < DJ4; ++m) {
              const float4 pv = pf[m * SPLITJ];
              a = fmaf(c[m].x, pv.x, a);
              a = fmaf(c[m].y, pv.y, a);
              a = fmaf(c[m].z, pv.z, a);
              a = fmaf(c[m].w, pv.w, a);
            }
            if (SPLITJ == 2) a += __shfl_xor_sync(0xffffffffu, a, 1);
            best[f] = min_u64(best[f], dist_key(fmaf(-2.0f * sv[f], a, cn), kg));
          }
        }
      }
    }
    if (SPLITJ == 1 || h == 0) {
#pragma unroll
      for (int f = 0; f < ST_F; ++f)
        if (f < nf) red[f * S.slots + kk0] = best[f];
    }
    __syncthreads();
    {  // 16 threads per frame reduce its slots
      const int f = t >> 4, sub = t & 15;
      uint64_t k = ~0ull;
      for (int m = sub; m < S.slots; m += 16) k = min_u64(k, red[f * S.slots + m]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) k = min_u64(k, __shfl_xor_sync(0xffffffffu, k, o));
      if (sub == 0) loc[f] = k;
    }
    __syncthreads();
    if (t == 32 && q + NB < n_q) {  // every read of buffer b is done: refill it
      fence_proxy_async_smem();
      issue(q + NB, b);
    }
    if (t < CS) {  // send this CTA's keys to rank t
      const uint32_t dst = cluster_map(smem_addr(xch + ((q & 1) * ST_MAX_CS + rank) * ST_F), (uint32_t)t);
      const uint4 *l4 = reinterpret_cast<const uint4 *>(loc);
#pragma unroll
      for (int i = 0; i < ST_F / 2; ++i) st_cluster_u4(dst + 16u * i, l4[i]);
      mbar_arrive_cluster(cluster_map(smem_addr(&x_full[q & 1]), (uint32_t)t));
    }

    // deferred terms of the previous code: p_{q'} -= G[q'][q-1][code_{q-1}], q' > q
    if (q >= 1) {
      const int *cprev = csm + ((q - 1) & 1) * ST_F;
      const int items = (n_q - q - 1) * ST_F * TPF;
      for (int e0 = t; e0 < items; e0 += ST_THREADS * ST_BATCH) {
        float4 gv[ST_BATCH];
#pragma unroll
        for (int u = 0; u < ST_BATCH; ++u) {
          const int e = e0 + u * ST_THREADS;
          if (e < items) {
            const int m = e / (ST_F * TPF), fj = e % (ST_F * TPF);
            const int qq = q + 1 + m, f = fj / TPF, j4 = fj % TPF;
            gv[u] = __ldg(g + (pair_index(qq, q - 1) * K + cprev[f]) * TPF + j4);
          }
        }
#pragma unroll
        for (int u = 0; u < ST_BATCH; ++u) {
          const int e = e0 + u * ST_THREADS;
          if (e < items) {
            const int m = e / (ST_F * TPF), fj = e % (ST_F * TPF);
            sub4(P[((int64_t)(q + 1 + m) * ST_F) * TPF + fj], gv[u]);
          }
        }
      }
    }

    // the exchange: the code of every frame
    if (!mbar_wait_cluster_hot(&x_full[q & 1], (uint32_t)((q >> 1) & 1))) st_error(status, RVQ_DEVICE_TIMEOUT);
    if (t < ST_F * TPF) {
      const int f = t / TPF, j4 = t % TPF;
      const uint64_t *xs = xch + (q & 1) * ST_MAX_CS * ST_F + f;
      uint64_t kb = xs[0];
      for (int r = 1; r < CS; ++r) kb = min_u64(kb, xs[r * ST_F]);
      uint32_t code = (uint32_t)kb;
      if (code >= (uint32_t)K) code = (uint32_t)K - 1;  // only after a timeout
      if (j4 == 0) {
        csm[(q & 1) * ST_F + f] = (int)code;
        if (rank == 0 && f < nf) codes[(f0 + f) * n_q + q] = (int32_t)code;
      }
      if (q + 1 < n_q) {
        const float4 gq = __ldg(g + (pair_index(q + 1, q) * K + code) * TPF + j4);
        float4 &pv = P[((int64_t)(q + 1) * ST_F + f) * TPF + j4];
        sub4(pv, gq);
        if (metric == RVQ_METRIC_COSINE) {
          float ss = pv.x * pv.x + pv.y * pv.y + pv.z * pv.z + pv.w * pv.w;
#pragma unroll
          for (int o = TPF / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (j4 == 0) sv[f] = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
        }
      }
    }
    __syncthreads();
  }

  // a slice copy whose wait gave up may still be landing: wait (bounded) for it
  if (t == 32) {
    for (int b = 0; b < NB; ++b) {
      int last = -1;
      for (int q = b; q < n_q; q += NB) last = q;
      if (last >= 0) mbar_wait(&cb_full[b], (uint32_t)((NB == 2 ? last >> 1 : last) & 1));
    }
  }
  cluster_sync_all();  // no CTA leaves while another may still address its shared memory
}

std::atomic<unsigned long long> g_stream_attr_done{0};
std::atomic<int64_t> g_stream_max_frames{kStreamMaxFramesDefault};

template <int d, int SPLITJ>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(k_encode_stream<d, SPLITJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)ST_SMEM_LIMIT);
}

cudaError_t ensure_stream_attributes() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (g_stream_attr_done.load() & bit) return cudaSuccess;
  if ((e = set_smem_attr<kCodeDim, 2>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<kCodeDim, 1>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<kCodeDimSmall, 2>()) != cudaSuccess) return e;
  g_stream_attr_done.fetch_or(bit);
  return cudaSuccess;
}

}  // namespace

bool stream_supported(const rvq_dims &dm, int n_q, int64_t n_frames) {
  if (n_frames < 1 || n_frames > g_stream_max_frames.load()) return false;
  if (dm.K % 128 != 0 || dm.K < 128) return false;
  if (dm.d == kCodeDim) {
    if (dm.K > 4096) return false;  // slices of at most 512 codewords
  } else if (dm.d != kCodeDimSmall || dm.K > kMaxKSmall) {
    return false;
  }
  return stream_nb(dm.d, dm.K, n_q) > 0;
}

cudaError_t launch_encode_stream(const rvq_dims &dm, const void *tables, const float *x, int64_t n, int n_q,
                                 int32_t *codes, int *status, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  cudaError_t e = ensure_stream_attributes();
  if (e != cudaSuccess) return e;
  const int NB = stream_nb(dm.d, dm.K, n_q);
  const StreamShape S = stream_shape(dm.d, dm.K, n_q, NB);
  const int64_t clusters = (n + ST_F - 1) / ST_F;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(clusters * S.CS), 1, 1);
  cfg.blockDim = dim3(ST_THREADS, 1, 1);
  cfg.dynamicSmemBytes = S.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float4 *w_t = at<float4>(tables, L.w_in_t), *b_in = at<float4>(tables, L.b_in);
  const float4 *cb_s = at<float4>(tables, L.cb_stream), *g = at<float4>(tables, L.g);
  const float *cn = at<float>(tables, L.cnorm);
  const int D_in = dim_in(dm);
  if (dm.d == kCodeDimSmall)
    return cudaLaunchKernelEx(&cfg, k_encode_stream<kCodeDimSmall, 2>, x, w_t, b_in, cb_s, cn, g, codes, n, D_in,
                              dm.K, n_q, NB, dm.metric, status);
  if (S.kc == 128)
    return cudaLaunchKernelEx(&cfg, k_encode_stream<kCodeDim, 2>, x, w_t, b_in, cb_s, cn, g, codes, n, D_in, dm.K,
                              n_q, NB, dm.metric, status);
  return cudaLaunchKernelEx(&cfg, k_encode_stream<kCodeDim, 1>, x, w_t, b_in, cb_s, cn, g, codes, n, D_in, dm.K,
                            n_q, NB, dm.metric, status);
}

}  // namespace rvq

// Process-wide threshold of the streaming path (documented in include/rvq.h).
extern "C" RVQ_API int64_t rvq_set_stream_max_frames(int64_t max_frames) {
  if (max_frames < 0) return rvq::g_stream_max_frames.load();
  return rvq::g_stream_max_frames.exchange(max_frames);
}
