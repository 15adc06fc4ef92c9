// Low-latency RVQ encode of small batches: the streaming path.
//
// Realtime callers encode a few frames at a time: the omnivoice-tts tool of
// omnivoice.cpp ARCHITECTURE.md ("CLI tools") begins synthesising once a first
// sentence of its streamed text is complete, and moss-tts.cpp AGENTS.md has a
// realtime TTS front end.  For such calls the tile path (128-frame tiles, one
// CTA per tile walking all K codewords of every stage) leaves the GPU idle
// and its latency is the serial walk over Q*K codewords.  Here:
//
//   k_project_small   P0[n][q*d + j] = w_in'[q][j] . x[n] + b_in'[q][j] for
//                     every stage, spread over (n_q*d/8) x ceil(n/16) CTAs
//                     (8 output columns and 16 frames each; frames and weight
//                     rows staged in shared memory by bulk copies, float32
//                     FMA).  It lets the next kernel launch at once
//                     (programmatic dependent launch).
//   k_stream_search   groups of up to 16 frames on thread-block clusters of
//                     CS = min(8, K/128) CTAs, G groups a cluster (G > 1
//                     only for calls of more than 16 frames: the fewest
//                     groups that fit the call in one wave of clusters, at
//                     most 8), scored one group at a time.  CTA r owns
//                     codewords [r*kc, (r+1)*kc), kc = K/CS, of every stage
//                     (staged in shared memory by a bulk copy NB stages ahead)
//                     and the projections of stages q = r (mod CS).  Stage q:
//       distances     dist = ||c||^2 - 2 s p.c for the CTA's slice (s = 1, or
//                     1/max(||p||, 1e-12) for the cosine metric), float32 FMA;
//                     per frame the minimum of the key (distance, index);
//       exchange      the CS keys of each frame go to every CTA by st.async
//                     into its shared memory, counted by an mbarrier's
//                     transaction bytes; the smallest key is the code --
//                     distance first, then the lowest index, as the plain
//                     argmin;
//       update        p_{q+1} -= G[q+1][q][code_q] in every CTA (the
//                     cross-stage table of rvq_prepare).  The owner of stage
//                     q+2 applies the same term for it and pushes that stage's
//                     projection (every term but the last) into every CTA,
//                     one stage ahead of its use; owners apply the terms of
//                     later stages to their own copies only.
//
// The distances run on the CUDA cores, not tensor core tiles: with at most 16
// frames a stage is a [kc x d] by [d x 16] product per CTA, far below one
// tcgen05 tile, and the path is bound by latency, not arithmetic.
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

__device__ __forceinline__ void st_error(int *status, int code) { atomicCAS(status, 0, code); }

// ===========================================================================
// k_project_small
// ===========================================================================
// Calls whose projection is at least this many multiply-adds (frames x D_in x
// n_q*d) take the tensor-core projection of the tile path instead
// (k_project_tc in 128-frame items): it has a fixed latency of about
// 20 us, and measured faster from about 2e8 (omnivoice 384 frames, moss_deep
// 128, moss_lfq 1024).
#ifndef RVQ_STREAM_TC_PROJECTION_MACS
#define RVQ_STREAM_TC_PROJECTION_MACS (int64_t(3) << 26)
#endif
constexpr int PS_THREADS = 256;
constexpr int PS_COLS = 8;   // output columns (rows of w_in') per CTA
constexpr int PS_F = 16;     // frames per CTA
constexpr int PS_DC = 512;   // D_in elements per staged chunk
constexpr size_t PS_SMEM = (size_t)2 * (PS_F + PS_COLS) * PS_DC * 4 + 16;

// x [n][D_in], w_f [n_cols][D_in], b_in [n_cols], P0 [n][n_cols].
// grid (n_cols/8, ceil(n/16)).  Warp w: columns 2(w%4), 2(w%4)+1 of the CTA's
// 8 and frames 8(w/4) .. +7; lane l: elements 4l + 128m of each chunk.
__global__ void __launch_bounds__(PS_THREADS)
    k_project_small(const float *__restrict__ x, const float *__restrict__ w_f, const float *__restrict__ b_in,
                    float *__restrict__ P0, int64_t n, int D_in, int n_cols, int *__restrict__ status,
                    int zero_status) {
  extern __shared__ __align__(128) unsigned char smem[];
  float *xs = reinterpret_cast<float *>(smem);   // [2][PS_F][PS_DC]
  float *ws = xs + 2 * PS_F * PS_DC;             // [2][PS_COLS][PS_DC]
  uint64_t *bar = reinterpret_cast<uint64_t *>(ws + 2 * PS_COLS * PS_DC);
  griddep_launch_dependents();  // the search kernel may start its prologue
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int c0 = blockIdx.x * PS_COLS;
  const int64_t f0 = (int64_t)blockIdx.y * PS_F;
  const int nf = (int)(n - f0 < PS_F ? n - f0 : PS_F);
  if (zero_status && blockIdx.x == 0 && blockIdx.y == 0 && t == 0) *status = 0;
  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int nch = (D_in + PS_DC - 1) / PS_DC;
  auto issue = [&](int c) {  // warp 0: chunk c into buffer c & 1
    const int b = c & 1, i0 = c * PS_DC;
    const uint32_t bytes = (uint32_t)((D_in - i0 < PS_DC ? D_in - i0 : PS_DC) * 4);
    if (c >= 2) fence_proxy_async_smem();  // the buffer's last reads were generic loads
    if (lane == 0) mbar_arrive_expect_tx(&bar[b], bytes * (uint32_t)(nf + PS_COLS));
    __syncwarp();
    if (lane < nf)
      bulk_g2s(xs + (b * PS_F + lane) * PS_DC, x + (f0 + lane) * (int64_t)D_in + i0, bytes, &bar[b]);
    else if (lane >= 16 && lane < 16 + PS_COLS)
      bulk_g2s(ws + (b * PS_COLS + lane - 16) * PS_DC, w_f + (int64_t)(c0 + lane - 16) * D_in + i0, bytes,
               &bar[b]);
  };
  if (warp == 0) {
    issue(0);
    if (nch > 1) issue(1);
  }
  const int cp = warp & 3, fh = warp >> 2;
  const bool active = 8 * fh < nf;
  float acc[2][8] = {};
  for (int c = 0; c < nch; ++c) {
    const int b = c & 1;
    if (!mbar_wait(&bar[b], (uint32_t)((c >> 1) & 1))) st_error(status, RVQ_DEVICE_TIMEOUT);
    const int len = D_in - c * PS_DC < PS_DC ? D_in - c * PS_DC : PS_DC;
    if (active) {
      const float4 *w0 = reinterpret_cast<const float4 *>(ws + (b * PS_COLS + 2 * cp) * PS_DC);
      const float4 *w1 = w0 + PS_DC / 4;
      const float4 *xb = reinterpret_cast<const float4 *>(xs + (b * PS_F + 8 * fh) * PS_DC);
      for (int i4 = lane; 4 * i4 < len; i4 += 32) {
        const float4 a = w0[i4], e = w1[i4];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 xv = xb[v * (PS_DC / 4) + i4];
          acc[0][v] = fmaf(xv.x, a.x, acc[0][v]);
          acc[0][v] = fmaf(xv.y, a.y, acc[0][v]);
          acc[0][v] = fmaf(xv.z, a.z, acc[0][v]);
          acc[0][v] = fmaf(xv.w, a.w, acc[0][v]);
          acc[1][v] = fmaf(xv.x, e.x, acc[1][v]);
          acc[1][v] = fmaf(xv.y, e.y, acc[1][v]);
          acc[1][v] = fmaf(xv.z, e.z, acc[1][v]);
          acc[1][v] = fmaf(xv.w, e.w, acc[1][v]);
        }
      }
    }
    __syncthreads();  // buffer b is free
    if (warp == 0 && c + 2 < nch) issue(c + 2);
  }
  if (active) {
#pragma unroll
    for (int col = 0; col < 2; ++col)
#pragma unroll
      for (int v = 0; v < 8; ++v)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[col][v] += __shfl_xor_sync(0xffffffffu, acc[col][v], o);
    if (lane < 16) {
      const int col = lane >> 3, v = lane & 7, f = 8 * fh + v;
      float s = 0.0f;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int vv = 0; vv < 8; ++vv)
          if (cc == col && vv == v) s = acc[cc][vv];
      const int jc = c0 + 2 * cp + col;
      if (f < nf) P0[(f0 + f) * n_cols + jc] = s + __ldg(b_in + jc);
    }
  }
}

// ===========================================================================
// k_stream_search
// ===========================================================================
constexpr int ST_THREADS = 256;
constexpr int ST_FG = kStreamFrames;       // frames per group (scored together in registers)
constexpr int ST_MAX_G = 8;                 // groups per cluster (frames per cluster <= 128)
constexpr int ST_MAX_CS = 8;                // cluster size limit (portable)
constexpr uint32_t ST_SMEM_LIMIT = 232448;  // opt-in dynamic shared memory per block
constexpr int ST_BATCH = 8;                 // table rows in flight per thread in the owners' updates

// Dynamic shared memory layout (byte offsets), the same on host and device.
struct StreamShape {
  int CS, kc, NB, slots, n_own;
  uint32_t pown, pin, cbuf, cnb, red, xch, loc, csm, sv, bars, total;
};

__host__ __device__ inline uint32_t up16(uint32_t v) { return (v + 15u) & ~15u; }

// FPC: frames per cluster (a multiple of 16, or the whole call when it has fewer).
__host__ __device__ inline StreamShape stream_shape(int d, int K, int n_q, int NB, int FPC) {
  StreamShape S{};
  S.CS = stream_cluster_size(K);
  S.kc = K / S.CS;
  S.NB = NB;
  S.slots = S.kc == 128 ? 128 : 256;       // key-writing threads per frame
  S.n_own = (n_q + S.CS - 1) / S.CS;       // stages owned by rank 0 (the most)
  const uint32_t row = (uint32_t)FPC * d * 4;
  uint32_t o = 0;
  S.pown = o; o = up16(o + (uint32_t)S.n_own * row);                     // [n_own][FPC][d] owned stages
  S.pin = o;  o = up16(o + 2u * row);                                    // [2][FPC][d] pushed stages
  o = (o + 127u) & ~127u;
  S.cbuf = o; o = up16(o + (uint32_t)NB * S.kc * d * 4);                 // [NB][d/4][kc] float4 slices
  S.cnb = o;  o = up16(o + (uint32_t)NB * S.kc * 4);                     // [NB][kc] squared norms
  S.red = o;  o = up16(o + (uint32_t)ST_FG * S.slots * 8);               // [16][slots] keys of a group
  S.xch = o;  o = up16(o + 2u * ST_MAX_CS * (uint32_t)((FPC + 1) & ~1) * 8);  // [2][rank][FPC, even] exchanged keys
  S.loc = o;  o = up16(o + (uint32_t)(FPC + 1) * 8);                     // [FPC] this CTA's best keys
  S.csm = o;  o = up16(o + 2u * FPC * 4);                                // [2][FPC] codes of the last two stages
  S.sv = o;   o = up16(o + (uint32_t)FPC * 4);                           // [FPC] distance scale s
  S.bars = o; o = up16(o + 7u * 8);                                      // cb_full[3] x_full[2] p_full[2]
  S.total = o;
  return S;
}

// Buffers for the codebook slices: 2 when two fit, else 1 (0: the shape does
// not fit).  (A third buffer measured no faster: the copies land in time.)
int stream_nb(int d, int K, int n_q, int FPC) {
  if (stream_shape(d, K, n_q, 2, FPC).total <= ST_SMEM_LIMIT) return 2;
  if (stream_shape(d, K, n_q, 1, FPC).total <= ST_SMEM_LIMIT) return 1;
  return 0;
}

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

// P0 [n][n_q*d] (k_project_small), codes [n][n_q].  grid: CS * ceil(n/FPC)
// CTAs in clusters of CS; ST_THREADS threads.  A cluster takes FPC = NF * G
// frames: G groups of NF, scored one group at a time (G > 1 only with
// NF = 16).  SPLITJ: threads per codeword (2 when kc == 128, each taking
// every other float4 column); NF: frames per group (16, or fewer when the
// whole call has fewer); CW: codewords a thread scores together (2 when kc is
// a multiple of 512, sharing the loads of the frames' projections; otherwise a
// thread takes codewords kk, kk + 256, ... one at a time, and kc need not be a
// multiple of 256).  MULTI: several groups a cluster (G_arg of them); without
// it G = 1 at compile time, so that the one-group kernel of the smallest calls
// keeps its constant trip counts.
template <int d, int SPLITJ, int NF, int CW, bool MULTI>
__global__ void __launch_bounds__(ST_THREADS, 1)
    k_stream_search(const float *__restrict__ P0, const float4 *__restrict__ cb_s, const float *__restrict__ cnorm,
                    const float4 *__restrict__ g, int32_t *__restrict__ codes, int64_t n, int K, int n_q, int NB,
                    int G_arg, int metric, int *__restrict__ status) {
  constexpr int TPF = d / 4;            // float4 columns of a row of d
  constexpr int DJ4 = TPF / SPLITJ;     // float4 columns of a codeword per thread
  constexpr unsigned kRedMask = 16 * NF >= 32 ? 0xffffffffu : 0x0000ffffu;
  extern __shared__ __align__(128) unsigned char smem[];
  const int G = MULTI ? G_arg : 1;      // groups per cluster
  const int FPC = NF * G;               // frames per cluster
  const int NU = (FPC + 1) / 2;         // 16-byte units of FPC keys
  const int FPX = 2 * NU;               // stride of a rank's keys in xch
  const int n_rows = FPC * TPF;         // (frame, float4 column) elements of a stage's projection
  // lanes of warp 0 taking part when fewer than 32 elements are worked on
  const unsigned row_mask = n_rows >= 32 ? 0xffffffffu : (1u << n_rows) - 1u;
  const StreamShape S = stream_shape(d, K, n_q, NB, FPC);
  const int t = threadIdx.x;
  const int CS = S.CS, kc = S.kc;
  if (cluster_nctarank() != (uint32_t)CS || blockDim.x != ST_THREADS || dynamic_smem_size() < S.total ||
      (SPLITJ == 2) != (kc == 128) || (CW == 2 && kc % (2 * ST_THREADS) != 0) || (NB != 1 && NB != 2 && NB != 3) ||
      G_arg < 1 || G_arg > ST_MAX_G || (MULTI ? NF != ST_FG : G_arg != 1) || (NF < ST_FG && n > NF)) {
    griddep_wait();  // after the projection kernel, which may clear the status word
    if (t == 0) st_error(status, RVQ_DEVICE_BAD_LAUNCH);
    return;  // uniform over the cluster: no CTA reaches a cluster barrier
  }
  const uint32_t rank = cluster_ctarank();
  const int64_t f0 = (int64_t)(blockIdx.x / CS) * FPC;
  const int nf = (int)(n - f0 < FPC ? n - f0 : FPC);
  const int n_cols = n_q * d;

  float4 *Pown = reinterpret_cast<float4 *>(smem + S.pown);   // [n_own][FPC][TPF]
  float4 *Pin = reinterpret_cast<float4 *>(smem + S.pin);     // [2][FPC][TPF]
  float4 *cbuf = reinterpret_cast<float4 *>(smem + S.cbuf);   // [NB][TPF][kc]
  float *cnb = reinterpret_cast<float *>(smem + S.cnb);       // [NB][kc]
  uint64_t *red = reinterpret_cast<uint64_t *>(smem + S.red); // [16][slots]
  uint64_t *xch = reinterpret_cast<uint64_t *>(smem + S.xch); // [2][ST_MAX_CS][FPX]
  uint64_t *loc = reinterpret_cast<uint64_t *>(smem + S.loc); // [FPC]
  int *csm = reinterpret_cast<int *>(smem + S.csm);           // [2][FPC]
  float *sv = reinterpret_cast<float *>(smem + S.sv);         // [FPC]
  uint64_t *cb_full = reinterpret_cast<uint64_t *>(smem + S.bars);
  uint64_t *x_full = cb_full + 3, *p_full = cb_full + 5;

  const uint32_t slice_bytes = (uint32_t)kc * d * 4, norm_bytes = (uint32_t)kc * 4;
  // transaction bytes of one exchange (keys from the other CS-1 CTAs) and of
  // one push (a stage projection from its owner, unless this CTA owns it)
  const uint32_t x_bytes = (uint32_t)(CS - 1) * NU * 16;
  auto p_bytes = [&](int q) { return q % CS == (int)rank ? 0u : (uint32_t)n_rows * 16; };
  auto issue = [&](int q, int b) {  // one thread: stage q's slice into buffer b
    mbar_arrive_expect_tx(&cb_full[b], slice_bytes + norm_bytes);
    bulk_g2s(cbuf + (size_t)b * TPF * kc, cb_s + ((int64_t)q * CS + rank) * TPF * kc, slice_bytes, &cb_full[b]);
    bulk_g2s(cnb + (size_t)b * kc, cnorm + (int64_t)q * K + (int64_t)rank * kc, norm_bytes, &cb_full[b]);
  };
  // Push owned stage q's projection (rows 0 .. FPC-1, every term but its
  // last) into the other CTAs: lane 0 of warp r bulk-copies it to rank r (one
  // copy per warp, so that no warp is held up issuing several).  The rows were
  // written by generic stores, each writer fenced them for the async proxy,
  // and a CTA barrier came in between.  This CTA's own copy is a plain store
  // by the thread that owns the element.
  auto push_remote = [&](int q) {
    const int r = t >> 5;
    if ((t & 31) == 0 && r < CS && r != (int)rank) {
      const uint32_t dst = cluster_map(smem_addr(Pin + (q & 1) * n_rows), (uint32_t)r);
      const uint32_t bar = cluster_map(smem_addr(&p_full[q & 1]), (uint32_t)r);
      bulk_s2cluster(dst, Pown + (q / CS) * n_rows, (uint32_t)n_rows * 16, bar);
    }
  };

  if (t == 0) {
    for (int b = 0; b < NB; ++b) mbar_init(&cb_full[b], 1);  // NB <= 3: the layout has three slice barriers
    for (int b = 0; b < 2; ++b) {
      mbar_init(&x_full[b], 1);
      mbar_init(&p_full[b], 1);
    }
    fence_mbar_init();
    // this CTA's own arrival for the exchanges and pushes of stages 0 and 1
    for (int q = 0; q < 2 && q < n_q; ++q) {
      mbar_arrive_expect_tx(&x_full[q], x_bytes);
      mbar_arrive_expect_tx(&p_full[q], p_bytes(q));
    }
  }
  for (int e = t; e < FPC; e += ST_THREADS) sv[e] = 1.0f;
  __syncthreads();
  cluster_arrive();  // barriers armed; waited for before the first remote access
  if (t == 32)
    for (int q = 0; q < NB && q < n_q; ++q) issue(q, q);

  // ---- the owned stages' projections (zero rows past the last frame) --------
  griddep_wait();  // k_project_small has finished; P0 is visible
  for (int e = t; e < S.n_own * n_rows; e += ST_THREADS) {
    const int i = e / n_rows, fj = e % n_rows, f = fj / TPF, j4 = fj % TPF;
    const int q = (int)rank + i * CS;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    // (through L2 only: P0 was written by the kernel this one overlapped)
    if (q < n_q && f < nf) v = __ldcg(reinterpret_cast<const float4 *>(P0 + (f0 + f) * n_cols + q * d) + j4);
    Pown[e] = v;
  }
  fence_proxy_async_smem();
  __syncthreads();
  cluster_wait();
  for (int q = 0; q < 2 && q < n_q; ++q)  // stages 0 and 1 need no cross-stage term before the push
    if (q % CS == (int)rank) {
      push_remote(q);
      for (int e = t; e < n_rows; e += ST_THREADS) Pin[(q & 1) * n_rows + e] = Pown[(q / CS) * n_rows + e];
    }
  if (!mbar_wait_cluster_hot(&p_full[0], 0)) st_error(status, RVQ_DEVICE_TIMEOUT);
  __syncthreads();  // this CTA's own pushes are visible
  if (metric == RVQ_METRIC_COSINE)  // s of stage 0
    for (int e = t; e < n_rows; e += ST_THREADS) {  // whole warps, or the first n_rows lanes of warp 0
      const int f = e / TPF, j4 = e % TPF;
      const float4 v = Pin[e];
      float ss = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
      for (int o = TPF / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(row_mask, ss, o);
      if (j4 == 0) sv[f] = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
    }
  __syncthreads();

  // ---- the stage loop -------------------------------------------------------
  const int h = SPLITJ == 2 ? (t & 1) : 0;
  const int kk0 = SPLITJ == 2 ? (t >> 1) : t;
  int b = 0;         // slice buffer of stage q (q mod NB)
  uint32_t ph = 0;   // its phase parity ((q / NB) & 1)
  for (int q = 0; q < n_q; ++q) {
    // Re-arm the barriers whose last phase every thread has now seen (stage
    // q's push, stage q-1's exchange).  Not earlier: an arm that expects no
    // bytes completes the next phase at once, and a thread still waiting on
    // the previous phase would then miss it.  The last thread does it: it
    // stores no codes, so its arrive (a release) waits for no global store.
    if (t == ST_THREADS - 1) {
      if (q + 2 < n_q) mbar_arrive_expect_tx(&p_full[q & 1], p_bytes(q + 2));
      if (q >= 1 && q + 1 < n_q) mbar_arrive_expect_tx(&x_full[(q + 1) & 1], x_bytes);
    }
    if (q >= 1 && q + 1 < n_q && (q + 1) % CS == (int)rank) push_remote(q + 1);  // updated at the end of stage q-1

    // The previous code's terms for this CTA's stages q' >= q+2 (q' = rank mod
    // CS), applied while this stage's keys travel.  The rows of the first PF
    // items of each thread are loaded now, so that their latency passes during
    // the distances; item e is (owned stage first + e / n_rows, element e mod
    // n_rows), so stage q+2's element e goes to thread e mod ST_THREADS -- the
    // thread that applies its next term at the end of this stage.
    constexpr int PF = SPLITJ == 2 ? 4 : (NF == 16 ? 1 : 2);
    const int later_first = (q + 2 - (int)rank + CS - 1) / CS;  // owned index of the first such stage
    const int later_items = q >= 1 && S.n_own > later_first ? (S.n_own - later_first) * n_rows : 0;
    const int *cprev = csm + ((q - 1) & 1) * FPC;
    auto later_stage = [&](int e) { return (int)rank + (later_first + e / n_rows) * CS; };
    auto later_row = [&](int e) -> const float4 * {  // nullptr past the last stage
      const int fj = e % n_rows, f = fj / TPF, j4 = fj % TPF, qq = later_stage(e);
      return qq < n_q ? g + (pair_index(qq, q - 1) * K + cprev[f]) * TPF + j4 : nullptr;
    };
    auto later_part = [&](int e) -> float4 & {  // the owned stage's element of item e
      return Pown[(later_first + e / n_rows) * n_rows + e % n_rows];
    };
    float4 pre[PF];
#pragma unroll
    for (int u = 0; u < PF; ++u) {
      const int e = t + u * ST_THREADS;
      const float4 *row = e < later_items ? later_row(e) : nullptr;
      if (row) pre[u] = __ldg(row);
    }
    if (!mbar_wait_hot(&cb_full[b], ph)) st_error(status, RVQ_DEVICE_TIMEOUT);

    // distances of this CTA's slice, one group of NF frames at a time; per
    // frame the smallest key
    const float4 *cq = cbuf + (size_t)b * TPF * kc;
    const float *cnq = cnb + (size_t)b * kc;
#pragma unroll 1
    for (int grp = 0; grp < G; ++grp) {
      uint64_t best[NF];
#pragma unroll
      for (int f = 0; f < NF; ++f) best[f] = ~0ull;
      const float4 *pq = Pin + ((q & 1) * FPC + grp * NF) * TPF;
      const float *sg = sv + grp * NF;
      constexpr int KSTEP = ST_THREADS / SPLITJ;  // codewords scored by the CTA per pass
      for (int kk = kk0; kk < kc; kk += CW * KSTEP) {
        // dot products of the thread's CW codewords with every frame of the
        // group, the columns taken CH float4 at a time (in column order) to
        // bound the registers; each frame's projection is loaded once for all CW
        constexpr int CH = DJ4 < 8 ? DJ4 : (SPLITJ == 2 ? 4 : 8);
        float a[CW][NF];
#pragma unroll
        for (int w = 0; w < CW; ++w)
#pragma unroll
          for (int f = 0; f < NF; ++f) a[w][f] = 0.0f;
#pragma unroll 1
        for (int m0 = 0; m0 < DJ4; m0 += CH) {
          float4 c[CW][CH];
#pragma unroll
          for (int w = 0; w < CW; ++w)
#pragma unroll
            for (int m = 0; m < CH; ++m) c[w][m] = cq[((m0 + m) * SPLITJ + h) * kc + kk + w * KSTEP];
#pragma unroll
          for (int f = 0; f < NF; ++f) {
            const float4 *pf = pq + f * TPF + h;
#pragma unroll
            for (int m = 0; m < CH; ++m) {
              const float4 pv = pf[(m0 + m) * SPLITJ];
#pragma unroll
              for (int w = 0; w < CW; ++w) {
                a[w][f] = fmaf(c[w][m].x, pv.x, a[w][f]);
                a[w][f] = fmaf(c[w][m].y, pv.y, a[w][f]);
                a[w][f] = fmaf(c[w][m].z, pv.z, a[w][f]);
                a[w][f] = fmaf(c[w][m].w, pv.w, a[w][f]);
              }
            }
          }
        }
#pragma unroll
        for (int w = 0; w < CW; ++w) {
          const float cn = cnq[kk + w * KSTEP];
          const uint32_t kg = rank * (uint32_t)kc + (uint32_t)(kk + w * KSTEP);
#pragma unroll
          for (int f = 0; f < NF; ++f) {
            if (SPLITJ == 2) a[w][f] += __shfl_xor_sync(0xffffffffu, a[w][f], 1);
            best[f] = min_u64(best[f], dist_key(fmaf(-2.0f * sg[f], a[w][f], cn), kg));
          }
        }
      }
      if (SPLITJ == 1 || h == 0) {
#pragma unroll
        for (int f = 0; f < NF; ++f) red[f * S.slots + kk0] = best[f];
      }
      __syncthreads();
      if (t < 16 * NF) {  // 16 threads per frame reduce its slots
        const int f = t >> 4, sub = t & 15;
        uint64_t k = ~0ull;
        for (int m = sub; m < S.slots; m += 16) k = min_u64(k, red[f * S.slots + m]);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) k = min_u64(k, __shfl_xor_sync(kRedMask, k, o, 16));
        if (sub == 0) loc[grp * NF + f] = k;
      }
      __syncthreads();
    }
    if (t == 32 && q + NB < n_q) {  // every read of buffer b is done: refill it
      fence_proxy_async_smem();
      issue(q + NB, b);
    }
    // this CTA's keys to the other ranks, 16 bytes a thread (its own stay in loc)
    for (int e = t; e < (CS - 1) * NU; e += ST_THREADS) {
      const int di = e / NU, u = e % NU, r = di < (int)rank ? di : di + 1;
      const uint32_t dst = cluster_map(smem_addr(xch + ((q & 1) * ST_MAX_CS + rank) * FPX), (uint32_t)r);
      const uint32_t bar = cluster_map(smem_addr(&x_full[q & 1]), (uint32_t)r);
      st_async_u4(dst + 16u * u, reinterpret_cast<const uint4 *>(loc)[u], bar);
    }

    // while the keys travel: apply the deferred terms (the prefetched rows
    // first, then any further items in batches)
    if (later_items > 0) {
#pragma unroll
      for (int u = 0; u < PF; ++u) {
        const int e = t + u * ST_THREADS;
        if (e < later_items && later_stage(e) < n_q) sub4(later_part(e), pre[u]);
      }
      for (int e0 = t + PF * ST_THREADS; e0 < later_items; e0 += ST_THREADS * ST_BATCH) {
        float4 gv[ST_BATCH];
#pragma unroll
        for (int u = 0; u < ST_BATCH; ++u) {
          const int e = e0 + u * ST_THREADS;
          const float4 *row = e < later_items ? later_row(e) : nullptr;
          if (row) gv[u] = __ldg(row);
        }
#pragma unroll
        for (int u = 0; u < ST_BATCH; ++u) {
          const int e = e0 + u * ST_THREADS;
          if (e < later_items && later_stage(e) < n_q) sub4(later_part(e), gv[u]);
        }
      }
    }

    // the exchange: the code of every frame
    if (!mbar_wait_cluster_hot(&x_full[q & 1], (uint32_t)((q >> 1) & 1))) st_error(status, RVQ_DEVICE_TIMEOUT);
    if (q + 1 < n_q)  // stage q+1's pushed projection
      if (!mbar_wait_cluster_hot(&p_full[(q + 1) & 1], (uint32_t)(((q + 1) >> 1) & 1)))
        st_error(status, RVQ_DEVICE_TIMEOUT);
    const uint64_t *xq = xch + (q & 1) * ST_MAX_CS * FPX;
    auto code_of = [&](int f) {
      uint64_t kb = loc[f];
      for (int r = 0; r < CS; ++r)
        if (r != (int)rank) kb = min_u64(kb, xq[r * FPX + f]);
      const uint32_t code = (uint32_t)kb;
      return code < (uint32_t)K ? code : (uint32_t)K - 1;  // (past K only after a timeout)
    };
    const bool own2 = q + 2 < n_q && (q + 2) % CS == (int)rank;
    for (int e = t; e < n_rows; e += ST_THREADS) {  // whole warps, or the first n_rows lanes of warp 0
      const int f = e / TPF, j4 = e % TPF;
      const uint32_t code = code_of(f);
      if (j4 == 0) {
        csm[(q & 1) * FPC + f] = (int)code;
        if (rank == 0 && f < nf) codes[(f0 + f) * n_q + q] = (int32_t)code;
      }
      float4 g1, g2;
      if (q + 1 < n_q) g1 = __ldg(g + (pair_index(q + 1, q) * K + code) * TPF + j4);
      if (own2) g2 = __ldg(g + (pair_index(q + 2, q) * K + code) * TPF + j4);
      if (q + 1 < n_q) {  // p_{q+1} complete
        float4 &pv = Pin[((q + 1) & 1) * n_rows + e];
        sub4(pv, g1);
        if (metric == RVQ_METRIC_COSINE) {
          float ss = pv.x * pv.x + pv.y * pv.y + pv.z * pv.z + pv.w * pv.w;
#pragma unroll
          for (int o = TPF / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(row_mask, ss, o);
          if (j4 == 0) sv[f] = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
        }
      }
      if (own2) {  // stage q+2 has every term but its last: pushed at the top of the next stage
        float4 &pv = Pown[((q + 2) / CS) * n_rows + e];
        sub4(pv, g2);
        Pin[((q + 2) & 1) * n_rows + e] = pv;
        fence_proxy_async_smem();
      }
    }
    __syncthreads();
    if (++b == NB) {
      b = 0;
      ph ^= 1u;
    }
  }

  // a slice copy whose wait gave up may still be landing: wait (bounded) for it
  if (t == 32) {
    for (int bb = 0; bb < NB; ++bb) {
      int last = -1;
      for (int q = bb; q < n_q; q += NB) last = q;
      if (last >= 0) mbar_wait(&cb_full[bb], (uint32_t)((last / NB) & 1));
    }
  }
  cluster_sync_all();  // no CTA leaves while another may still address its shared memory
}

std::atomic<unsigned long long> g_stream_attr_done{0};
std::atomic<int64_t> g_stream_max_frames{kStreamMaxFramesDefault};

template <int d, int SPLITJ, int CW>
cudaError_t set_search_attrs() {
  cudaError_t e = cudaSuccess;
  auto set = [&](auto kern) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ST_SMEM_LIMIT);
  };
  set(k_stream_search<d, SPLITJ, 1, CW, false>);
  set(k_stream_search<d, SPLITJ, 2, CW, false>);
  set(k_stream_search<d, SPLITJ, 4, CW, false>);
  set(k_stream_search<d, SPLITJ, 8, CW, false>);
  set(k_stream_search<d, SPLITJ, 16, CW, false>);
  set(k_stream_search<d, SPLITJ, 16, CW, true>);
  return e;
}

cudaError_t ensure_stream_attributes() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (g_stream_attr_done.load() & bit) return cudaSuccess;
  if ((e = cudaFuncSetAttribute(k_project_small, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PS_SMEM)) !=
      cudaSuccess)
    return e;
  if ((e = set_search_attrs<kCodeDim, 2, 1>()) != cudaSuccess) return e;
  if ((e = set_search_attrs<kCodeDim, 1, 1>()) != cudaSuccess) return e;
  if ((e = set_search_attrs<kCodeDim, 1, 2>()) != cudaSuccess) return e;
  if ((e = set_search_attrs<kCodeDimSmall, 2, 1>()) != cudaSuccess) return e;
  g_stream_attr_done.fetch_or(bit);
  return cudaSuccess;
}

template <int d, int SPLITJ, int CW>
cudaError_t launch_search(cudaLaunchConfig_t &cfg, int nf, const float *p0, const float4 *cb_s, const float *cn,
                          const float4 *g, int32_t *codes, int64_t n, int K, int n_q, int NB, int G, int metric,
                          int *status) {
  if (G > 1)
    return cudaLaunchKernelEx(&cfg, k_stream_search<d, SPLITJ, 16, CW, true>, p0, cb_s, cn, g, codes, n, K, n_q, NB,
                              G, metric, status);
  switch (nf) {
    case 1:
      return cudaLaunchKernelEx(&cfg, k_stream_search<d, SPLITJ, 1, CW, false>, p0, cb_s, cn, g, codes, n, K, n_q,
                                NB, G, metric, status);
    case 2:
      return cudaLaunchKernelEx(&cfg, k_stream_search<d, SPLITJ, 2, CW, false>, p0, cb_s, cn, g, codes, n, K, n_q,
                                NB, G, metric, status);
    case 4:
      return cudaLaunchKernelEx(&cfg, k_stream_search<d, SPLITJ, 4, CW, false>, p0, cb_s, cn, g, codes, n, K, n_q,
                                NB, G, metric, status);
    case 8:
      return cudaLaunchKernelEx(&cfg, k_stream_search<d, SPLITJ, 8, CW, false>, p0, cb_s, cn, g, codes, n, K, n_q,
                                NB, G, metric, status);
    default:
      return cudaLaunchKernelEx(&cfg, k_stream_search<d, SPLITJ, 16, CW, false>, p0, cb_s, cn, g, codes, n, K, n_q,
                                NB, G, metric, status);
  }
}

// Clusters of CS CTAs (one CTA per SM: 256 threads of about 200 registers)
// that can be resident at once on the current device, cached per device and
// cluster size; the SM count over CS if the query fails.
int max_active_clusters(int CS) {
  static std::atomic<int> cache[64][4];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const int slot = CS == 1 ? 0 : CS == 2 ? 1 : CS == 4 ? 2 : 3;
  std::atomic<int> &c = cache[dev & 63][slot];
  int v = c.load();
  if (v > 0) return v;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
  v = sms / CS > 0 ? sms / CS : 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(CS * v), 1, 1);
  cfg.blockDim = dim3(ST_THREADS, 1, 1);
  cfg.dynamicSmemBytes = ST_SMEM_LIMIT;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nc = 0;
  if (cudaOccupancyMaxActiveClusters(&nc, k_stream_search<kCodeDim, 1, 16, 1, true>, &cfg) == cudaSuccess && nc > 0)
    v = nc;
  else
    (void)cudaGetLastError();  // the query's error is not the caller's
  c.store(v);
  return v;
}

// Groups of 16 frames a cluster takes: the fewest that put the whole call in
// one wave of clusters, at most ST_MAX_G and at most what fits in shared memory
// with as many slice buffers as one group gets.
int stream_groups(const rvq_dims &dm, int n_q, int64_t n, int CS) {
  if (n <= ST_FG) return 1;
  const int64_t g16 = (n + ST_FG - 1) / ST_FG;
  const int64_t m = max_active_clusters(CS);
  int G = (int)((g16 + m - 1) / m);
  if (G > ST_MAX_G) G = ST_MAX_G;
  if (G < 1) G = 1;
  const int nb1 = stream_nb(dm.d, dm.K, n_q, ST_FG);
  while (G > 1 && stream_nb(dm.d, dm.K, n_q, ST_FG * G) != nb1) --G;
  return G;
}

}  // namespace

bool stream_supported(const rvq_dims &dm, int n_q, int64_t n_frames) {
  if (n_frames < 1 || n_frames > g_stream_max_frames.load()) return false;
  if (dm.K % 128 != 0 || dm.K < 128) return false;
  if (!stream_tables(dm)) return false;  // d = 64 with K > 4096: slices of more than 512 codewords
  if (dm.d != kCodeDim && (dm.d != kCodeDimSmall || dm.K > kMaxKSmall)) return false;
  return stream_nb(dm.d, dm.K, n_q, ST_FG) > 0;
}

cudaError_t stream_plan(const rvq_dims &dm, int n_q, int64_t n, int64_t plan[6]) {
  for (int i = 0; i < 6; ++i) plan[i] = 0;
  if (!stream_supported(dm, n_q, n)) return cudaSuccess;
  const cudaError_t e = ensure_stream_attributes();
  if (e != cudaSuccess) return e;
  const int nf = n > 8 ? ST_FG : n > 4 ? 8 : n > 2 ? 4 : (int)n;
  const int CS = stream_cluster_size(dm.K);
  const int G = stream_groups(dm, n_q, n, CS);
  plan[0] = 1;
  plan[1] = CS;
  plan[2] = nf;
  plan[3] = G;
  plan[4] = (n + (int64_t)nf * G - 1) / ((int64_t)nf * G);
  plan[5] = stream_nb(dm.d, dm.K, n_q, nf * G);
  return cudaSuccess;
}

cudaError_t launch_encode_stream(const rvq_dims &dm, const void *tables, const float *x, int64_t n, int n_q,
                                 int32_t *codes, float *p0, int *status, bool zero_status, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  cudaError_t e = ensure_stream_attributes();
  if (e != cudaSuccess) return e;
  const int D_in = dim_in(dm), n_cols = n_q * dm.d;
  if (n * D_in * n_cols >= RVQ_STREAM_TC_PROJECTION_MACS) {
    // enough frames for the tensor cores to pay: 128-frame tiles of 3xTF32 MMAs
    if ((e = launch_project_tc(dm, tables, x, n, n_q, p0, status, zero_status, st, -1)) != cudaSuccess) return e;
  } else {
    const int64_t groups = (n + PS_F - 1) / PS_F;
    k_project_small<<<dim3((unsigned)(n_cols / PS_COLS), (unsigned)groups), PS_THREADS, PS_SMEM, st>>>(
        x, at<float>(tables, L.w_in_f), at<float>(tables, L.b_in), p0, n, D_in, n_cols, status, zero_status ? 1 : 0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  const int nf = n > 8 ? ST_FG : n > 4 ? 8 : n > 2 ? 4 : (int)n;  // frames per group, >= min(n, 16)
  const int G = stream_groups(dm, n_q, n, stream_cluster_size(dm.K));
  const int FPC = nf * G;
  const int NB = stream_nb(dm.d, dm.K, n_q, FPC);
  const StreamShape S = stream_shape(dm.d, dm.K, n_q, NB, FPC);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(((n + FPC - 1) / FPC) * S.CS), 1, 1);
  cfg.blockDim = dim3(ST_THREADS, 1, 1);
  cfg.dynamicSmemBytes = S.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const float4 *cb_s = at<float4>(tables, L.cb_stream), *g = at<float4>(tables, L.g);
  const float *cn = at<float>(tables, L.cnorm);
  if (dm.d == kCodeDimSmall)
    return launch_search<kCodeDimSmall, 2, 1>(cfg, nf, p0, cb_s, cn, g, codes, n, dm.K, n_q, NB, G, dm.metric,
                                              status);
  if (S.kc == 128)
    return launch_search<kCodeDim, 2, 1>(cfg, nf, p0, cb_s, cn, g, codes, n, dm.K, n_q, NB, G, dm.metric, status);
  if (S.kc % (2 * ST_THREADS) == 0)
    return launch_search<kCodeDim, 1, 2>(cfg, nf, p0, cb_s, cn, g, codes, n, dm.K, n_q, NB, G, dm.metric, status);
  return launch_search<kCodeDim, 1, 1>(cfg, nf, p0, cb_s, cn, g, codes, n, dm.K, n_q, NB, G, dm.metric, status);
}

}  // namespace rvq

// Process-wide threshold of the streaming path (documented in include/rvq.h).
extern "C" RVQ_API int64_t rvq_set_stream_max_frames(int64_t max_frames) {
  if (max_frames < 0) return rvq::g_stream_max_frames.load();
  return rvq::g_stream_max_frames.exchange(max_frames);
}
