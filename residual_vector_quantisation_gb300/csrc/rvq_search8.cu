// Encode step 2 (the stage loop) for d = 8 codes: the small code space of the
// quantizer in moss-tts.cpp AGENTS.md, gotcha 9 ("argmin in 8-dim codebook
// space"), for either metric.
//
// Same re-associated form as the d = 64 kernel (rvq_encode_tc.cu): P0 =
// x.W_in^T + b_in of every stage comes from k_project_tc, and the query of
// stage q+1 is p = P0[n][q+1] - sum_{s<=q} G[q+1][s][code_s].  With d = 8 a
// chunk of 128 codewords is three tcgen05 MMAs (3xTF32: a_hi.b_lo, a_hi.b_hi,
// a_lo.b_hi, K = 8), so the limit is no longer the tensor core but the scan
// of the distances by the row threads.  The kernel is laid out for that:
//   * a stage's whole codebook image (K codewords of -2c, normalised for the
//     cosine metric, as TF32 hi and lo in 32-byte swizzled 128-codeword
//     blocks) and its norm operand (one 4 KB block per pair of chunks) come in
//     by one bulk copy each and stay in shared memory for the stage,
//     double-buffered by stage;
//   * three pipelines per CTA, each four row warps (one thread per frame of a
//     128-frame tile), one MMA issuer and 160 TMEM columns: query hi [0,8),
//     query lo [8,16), the norm MMA's A operands [16,32), distances [32,160);
//   * with more tiles than SMs each pipeline works on a tile of its own
//     (items of three tiles); otherwise (the SPLIT variant) the three share
//     one tile, pipeline p scanning the chunks c = p mod 3, and pipelines 1
//     and 2 hand their per-frame (value, index) minima to pipeline 0 at the
//     end of each stage.  Pipeline 0 alone then builds the query (all three
//     issuers read its TMEM columns) and gathers its terms.
// Query terms are copied per thread -- its own frame's 32-byte rows -- by
// 16-byte asynchronous copies into staging slots after the first distance
// chunk of a stage (all of them at once: one round trip a stage) and folded
// into an 8-float partial in registers at the stage boundary, in the order
// P0, G[.][0], G[.][1], ...; the boundary loads the row of the code just
// found straight into registers.  Deep stacks run in blocks of at most as
// many stages as a pipeline has staging slots (12 for a split tile, 4 for a
// tile of its own), the terms of earlier blocks subtracted from P0 by
// k_cross_terms between the launches.  The distance of codeword k is
// -2 (s p).c_k + ||c_k||^2 with s = 1 (plain metric) or 1 / max(||p||, 1e-12)
// (cosine metric, codebook normalised in the tables): the scale is applied to
// the query before it is split, and the norms are added by a fourth MMA per
// chunk -- A = [1 1 1 0 0 0 0 0] (or [0 0 0 0 1 1 1 0] for an odd chunk), a
// constant in TMEM, times a block holding the three exact TF32 parts of each
// ||c||^2 -- so the accumulator holds the distances themselves and the row
// threads' scan is a minimum tree only.  Ties go to the lowest index.  Every
// mbarrier wait is bounded.
#include <atomic>

#include "rvq_internal.cuh"
#include "sm103_ptx.cuh"

namespace rvq {
namespace {

using namespace ptx;

constexpr int S8_D = kCodeDimSmall;              // 8
constexpr int S8_KC = 128;                       // codewords per chunk (MMA N)
constexpr int S8_P = 3;                          // pipelines per CTA
constexpr int S8_THREADS = 512;                  // warp 0 producer, 1-3 issuers, 4-15 rows
constexpr uint32_t S8_TMEM_COLS = 512;
constexpr uint32_t S8_PIPE_COLS = 160;
constexpr uint32_t S8_A_HI = 0, S8_A_LO = 8, S8_A_NORM = 16, S8_ACC = 32;  // A_NORM: even chunk, +8 odd
constexpr uint32_t S8_IDESC = idesc_tf32(128, S8_KC);
constexpr uint32_t S8_HALF = 128 * S8_D * 4;     // 4 KB: the hi or the lo block of a chunk
constexpr int S8_TB = 4;                         // staging slots per pipeline
constexpr uint32_t S8_STG_BYTES = S8_P * S8_TB * 2 * 128 * 16;  // [pipe][slot][half][frame] x 16 B
constexpr uint32_t S8_XCH_BYTES = 2 * 2 * 128 * 4 * 2;  // values, indices
constexpr uint32_t S8_XROW_BYTES = 2 * 128 * S8_D * 4;  // pipelines 1, 2: their candidates' next-term rows

struct S8Bars {
  uint64_t img_full[2], img_free[2];
  uint64_t a_ready[S8_P], acc_full[S8_P], acc_empty[S8_P], drain[S8_P];
  uint64_t xch_full[2], xch_free[2];
  uint32_t tmem;
  uint32_t pad;
};

constexpr uint32_t S8_NBLOCK = 128 * S8_D * 4;  // 4 KB: the norm operand of a pair of chunks
__host__ __device__ constexpr uint32_t s8_buf_stride(int K) {
  return ((uint32_t)K * (2 * S8_D * 4) + (uint32_t)cn_img8_blocks(K) * S8_NBLOCK + 1023u) & ~1023u;
}
__host__ __device__ constexpr size_t s8_smem_bytes(int K) {
  return 1024 + 2 * (size_t)s8_buf_stride(K) + S8_STG_BYTES + S8_XCH_BYTES + S8_XROW_BYTES + sizeof(S8Bars);
}

__device__ __forceinline__ void record_error8(int *status, int code) { atomicCAS(status, 0, code); }

// Minimum of 64 values by a tree of three-input minima (32 instructions).
__device__ __forceinline__ float min64(const float (&v)[64]) {
  float a[22];
#pragma unroll
  for (int i = 0; i < 21; ++i) a[i] = fmin3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[21] = v[63];
  float b[8];
#pragma unroll
  for (int i = 0; i < 7; ++i) b[i] = fmin3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  b[7] = a[21];
  return fmin3(fmin3(b[0], b[1], b[2]), fmin3(b[3], b[4], b[5]), fminf(b[6], b[7]));
}

template <bool SPLIT>
__global__ void __launch_bounds__(S8_THREADS, 1)
    k_search8_tc(const float *__restrict__ P0, const float *__restrict__ G, const float *__restrict__ cb_img,
                 const float *__restrict__ cn_img, int32_t *__restrict__ codes, int64_t n_rows, int n_q, int q_begin,
                 int q_end, int K, int n_tiles, int metric, int *__restrict__ status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  constexpr int d = S8_D;
  constexpr int T = SPLIT ? 1 : S8_P;  // tiles per item
  const int nkc = K / S8_KC;
  const uint32_t img_bytes = (uint32_t)K * (2 * d * 4);
  const uint32_t cn_bytes = (uint32_t)cn_img8_blocks(K) * S8_NBLOCK;
  const uint32_t buf_stride = s8_buf_stride(K);
  unsigned char *bufs = smem;
  unsigned char *stg = smem + 2 * buf_stride;
  float *xv = reinterpret_cast<float *>(stg + S8_STG_BYTES);  // [2][2][128]
  int *xk = reinterpret_cast<int *>(xv + 2 * 2 * 128);         // [2][2][128]
  float4 *xr = reinterpret_cast<float4 *>(xk + 2 * 2 * 128);   // [2][128][2]: one buffer (see the exchange)
  S8Bars &bar = *reinterpret_cast<S8Bars *>(xr + 2 * 128 * 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = (n_tiles + T - 1) / T;
  // one tile per CTA in the SPLIT variant
  if (SPLIT && n_tiles > (int)gridDim.x) {
    if (tid == 0) record_error8(status, RVQ_DEVICE_BAD_LAUNCH);
    return;
  }

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar.img_full[b], 1);
      mbar_init(&bar.img_free[b], S8_P + S8_P * 128);  // every issuer's MMAs and every row thread's norm reads
      mbar_init(&bar.xch_full[b], 2 * 128);
      mbar_init(&bar.xch_free[b], 128);
    }
    for (int p = 0; p < S8_P; ++p) {
      mbar_init(&bar.a_ready[p], 128);
      mbar_init(&bar.acc_full[p], 1);
      mbar_init(&bar.acc_empty[p], 128);
      mbar_init(&bar.drain[p], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem, S8_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem;

  if (warp == 0) {
    // ---------------- producer: one stage image + norms per stage, double-buffered ----------------
    if (lane == 0) {
      uint32_t g = 0;  // stages gone through
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x)
        for (int q = q_begin; q < q_end && ok; ++q, ++g) {
          const int b = g & 1;
          if (g >= 2 && !mbar_wait(&bar.img_free[b], ((g >> 1) - 1) & 1)) {
            record_error8(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          unsigned char *dst = bufs + b * buf_stride;
          mbar_arrive_expect_tx(&bar.img_full[b], img_bytes + cn_bytes);
          bulk_g2s(dst, cb_img + (size_t)q * K * (2 * d), img_bytes, &bar.img_full[b]);
          bulk_g2s(dst + img_bytes, cn_img + (size_t)q * (cn_bytes / 4), cn_bytes, &bar.img_full[b]);
        }
      // the copies still in flight land before the CTA may exit
      for (uint32_t gg = g > 2 ? g - 2 : 0; gg < g; ++gg) mbar_wait(&bar.img_full[gg & 1], (gg >> 1) & 1);
    }
  } else if (warp <= S8_P) {
    // ---------------- MMA issuers: warp 1 + p for pipeline p ----------------
    // An issuer's wait stalls until its own queued MMAs have drained; with
    // three issuers the others' MMAs keep the tensor core busy meanwhile.
    const int p = warp - 1;
    if (lane == 0) {
      uint32_t g = 0, u = 0;
      bool ok = true;
      auto wait_or_fail = [&](uint64_t *b, uint32_t parity) {
        if (ok && !mbar_wait(b, parity)) {
          record_error8(status, RVQ_DEVICE_TIMEOUT);
          ok = false;
        }
        return ok;
      };
      const uint32_t acc = tmem + p * S8_PIPE_COLS + S8_ACC;
      const uint32_t ta = tmem + (SPLIT ? 0 : p) * S8_PIPE_COLS;  // the query's columns
      const uint32_t buf0 = smem_addr(bufs);
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x)
        for (int q = q_begin; q < q_end && ok; ++q, ++g) {
          const int b = g & 1;
          bool first = true;
          for (int c = SPLIT ? p : 0; c < nkc; c += SPLIT ? S8_P : 1) {
            if (u > 0 && !wait_or_fail(&bar.acc_empty[p], (u - 1) & 1)) break;
            if (first) {
              if (!wait_or_fail(&bar.a_ready[SPLIT ? 0 : p], g & 1)) break;
              if (!wait_or_fail(&bar.img_full[b], (g >> 1) & 1)) break;
              first = false;
            }
            tc_fence_after();
            const uint32_t chunk = buf0 + b * buf_stride + (uint32_t)c * (2 * S8_HALF);
            const uint64_t bhi = smem_desc(chunk, 16, 256, kSwizzle32B);
            const uint64_t blo = smem_desc(chunk + S8_HALF, 16, 256, kSwizzle32B);
            const uint64_t bnorm = smem_desc(buf0 + b * buf_stride + img_bytes + (uint32_t)(c >> 1) * S8_NBLOCK, 16,
                                             256, kSwizzle32B);
            mma_tf32_ta(acc, ta + S8_A_HI, blo, S8_IDESC, 0u);
            mma_tf32_ta(acc, ta + S8_A_HI, bhi, S8_IDESC, 1u);
            mma_tf32_ta(acc, ta + S8_A_LO, bhi, S8_IDESC, 1u);
            mma_tf32_ta(acc, ta + S8_A_NORM + 8u * (uint32_t)(c & 1), bnorm, S8_IDESC, 1u);
            mma_commit(&bar.acc_full[p]);
            ++u;
          }
          if (!ok) break;
          // an issuer with no chunk in the stage (split, fewer chunks than
          // pipelines) still keeps step: its commit for this stage must not
          // reach the buffer's barrier while an earlier stage is in use
          if (first && !wait_or_fail(&bar.a_ready[SPLIT ? 0 : p], g & 1)) break;
          mma_commit(&bar.img_free[b]);  // this stage's image is free once these MMAs are done
        }
      mma_commit(&bar.drain[p]);
      mbar_wait(&bar.drain[p], 0);
    }
  } else {
    // ---------------- one thread per frame row (warps 4-15) ----------------
    const int p = (warp - 1 - S8_P) >> 2;  // pipeline
    const int quarter = warp & 3;          // TMEM lane quarter of this warp
    const int f = quarter * 32 + lane;     // frame within the tile
    const uint32_t lane_base = tmem + p * S8_PIPE_COLS + ((uint32_t)(quarter * 32) << 16);
    const bool builder = !SPLIT || p == 0;  // builds the query, gathers its terms, writes codes
    constexpr int kSlots = SPLIT ? S8_P * S8_TB : S8_TB;
    const float4 *stg4 = reinterpret_cast<const float4 *>(stg) + (SPLIT ? 0 : p * S8_TB * 2 * 128);
    float4 *stg4w = reinterpret_cast<float4 *>(stg) + (SPLIT ? 0 : p * S8_TB * 2 * 128);
    const int64_t ld = (int64_t)n_q * d;
    const int n_own = SPLIT ? (nkc - p + S8_P - 1) / S8_P : nkc;  // chunks this pipeline scans per stage
    uint32_t g = 0, ua = 0, xu = 0;
    bool ok = true;
    int my_codes[kMaxStages];
    float part[d], gl[d];
#pragma unroll
    for (int j = 0; j < d; ++j) part[j] = gl[j] = 0.0f;
    {
      // the norm MMA's A operands, constant: the even and the odd chunk's slots
      const float a_even[d] = {1.f, 1.f, 1.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      const float a_odd[d] = {0.f, 0.f, 0.f, 0.f, 1.f, 1.f, 1.f, 0.f};
      tmem_st8(lane_base + S8_A_NORM, a_even);
      tmem_st8(lane_base + S8_A_NORM + 8, a_odd);
      // (made visible by the tmem_wait_st before the first query's a_ready)
    }

    // Term rows in flight: `npend` rows in staging slots 0.., the first one
    // added (the P0 row) when pend_p0, every other one subtracted.
    int npend = 0;
    bool pend_p0 = false;
    auto terms_finish = [&]() {
      if (npend == 0) return;
      cp_async_wait_all();
      for (int i = 0; i < npend; ++i) {
        const float4 a = stg4[(i * 2 + 0) * 128 + f], c4 = stg4[(i * 2 + 1) * 128 + f];
        const float r[d] = {a.x, a.y, a.z, a.w, c4.x, c4.y, c4.z, c4.w};
        if (i == 0 && pend_p0) {
#pragma unroll
          for (int j = 0; j < d; ++j) part[j] += r[j];
        } else {
#pragma unroll
          for (int j = 0; j < d; ++j) part[j] -= r[j];
        }
      }
      npend = 0;
      pend_p0 = false;
    };
    auto term_copy = [&](int slot, const float *row) {
      cp_async16_ca(stg4w + (slot * 2 + 0) * 128 + f, row);
      cp_async16_ca(stg4w + (slot * 2 + 1) * 128 + f, row + 4);
    };

    auto tile_of = [&](int item) { return SPLIT ? item : item * S8_P + p; };
    auto row_of = [&](int item) -> int64_t {  // this thread's frame of that item, clamped to a real row
      const int64_t nn = (int64_t)tile_of(item) * 128 + f;
      return (item < n_items && nn < n_rows) ? nn : 0;
    };
    if (builder) {  // the first query's first term: the projection row itself
      term_copy(0, P0 + row_of(blockIdx.x) * ld + q_begin * d);
      cp_async_commit();
      npend = 1;
      pend_p0 = true;
    }
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const int64_t n = (int64_t)tile_of(it) * 128 + f;
      const bool valid = tile_of(it) < n_tiles && n < n_rows;
      const int64_t n_row = row_of(it);
      const bool has_next = it + (int)gridDim.x < n_items;
      const int64_t n_next = row_of(it + gridDim.x);
#pragma unroll
      for (int j = 0; j < d; ++j) gl[j] = 0.0f;
      for (int q = q_begin; q < q_end && ok; ++q, ++g) {
        const int b = g & 1;
        if (builder) {
          // ---- stage boundary: query = partial - the row of the code just found
          terms_finish();
          float pq[d], ss = 0.0f;
#pragma unroll
          for (int j = 0; j < d; ++j) {
            pq[j] = part[j] - gl[j];
            ss = fmaf(pq[j], pq[j], ss);
            part[j] = 0.0f;
          }
          if (metric == RVQ_METRIC_COSINE) {  // the query scaled by 1 / n(p) before the split
            const float s_row = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
            for (int j = 0; j < d; ++j) pq[j] *= s_row;
          }
          tmem_st8(lane_base + S8_A_HI, pq);  // raw = hi after TF32 truncation
#pragma unroll
          for (int j = 0; j < d; ++j) pq[j] -= __uint_as_float(__float_as_uint(pq[j]) & 0xffffe000u);
          tmem_st8(lane_base + S8_A_LO, pq);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar.a_ready[p]);
        } else {
          // pipelines 1, 2 of a split tile: this stage's query is built
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.a_ready[0], g & 1))) {
            record_error8(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
        }
        // ---- terms of the next query known before this stage's code:
        //      next stage: P0[n][q+1], G[q+1][q_begin..q-1];  next item: P0[n'][q_begin]
        const int q_next = q + 1 < q_end ? q + 1 : q_begin;
        const int n_terms = !builder ? 0 : q + 1 < q_end ? q + 1 - q_begin : (has_next ? 1 : 0);
        const int64_t term_n = q + 1 < q_end ? n_row : n_next;
        int done = 0;
        // ---- scan this pipeline's chunks
        float best_v = __int_as_float(0x7f800000);
        int best_k = 0;
        int i_own = 0;
        for (int c = SPLIT ? p : 0; c < nkc; c += SPLIT ? S8_P : 1, ++i_own) {
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.acc_full[p], ua & 1))) {
            record_error8(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          ++ua;
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[64];
            tmem_ld32(lane_base + S8_ACC + 64 * h, *reinterpret_cast<float(*)[32]>(&v[0]));
            tmem_ld32(lane_base + S8_ACC + 64 * h + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
            tmem_wait_ld();
            if (h == 1) {
              tc_fence_before();
              mbar_arrive(&bar.acc_empty[p]);  // the accumulator is free: the values are in registers
            }
            const float m = min64(v);  // the distances themselves (norms added by the MMA)
            if (m <= best_v) {  // locate the first index holding m
              const int k = c * S8_KC + 64 * h + first_index_of(v, m);
              if (m < best_v || k < best_k) {
                best_v = m;
                best_k = k;
              }
            }
          }
          // ---- this chunk's share of the next query's known terms: all of
          //      them after the first chunk when the staging slots hold them
          //      (one round trip a stage), else spread over the chunks
          if (n_terms > 0) {
            const int target = n_terms <= kSlots ? n_terms : (n_terms * (i_own + 1) + n_own - 1) / n_own;
            while (done < target) {
              terms_finish();
              const int t1 = min(target, done + kSlots);
              for (int t = done; t < t1; ++t)
                term_copy(t - done, t == 0 ? P0 + term_n * ld + q_next * d
                                           : G + ((size_t)pair_index(q_next, q_begin + t - 1) * K +
                                                  my_codes[q_begin + t - 1]) * d);
              cp_async_commit();
              npend = t1 - done;
              pend_p0 = done == 0;
              done = t1;
            }
          }
        }
        if (!ok) break;
        mbar_arrive(&bar.img_free[b]);  // (kept in the count: every row thread is done with the stage)
        // the next query's last term for this pipeline's candidate code, loaded
        // before the exchange so that its latency overlaps it (the winner's row
        // is then at hand when the code is known)
        const bool next_term = q + 1 < q_end;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c4 = a;
        if (next_term) {
          const float4 *gr = reinterpret_cast<const float4 *>(G + ((size_t)pair_index(q + 1, q) * K + best_k) * d);
          a = __ldg(gr);
          c4 = __ldg(gr + 1);
        }
        if (SPLIT) {
          // ---- pipelines 1, 2 hand their minima (and candidate rows) to pipeline 0
          const int xb = xu & 1;
          const uint32_t use = xu >> 1;
          ++xu;
          if (p > 0) {
            if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(&bar.xch_free[xb], (use - 1) & 1))) {
              record_error8(status, RVQ_DEVICE_TIMEOUT);
              ok = false;
              break;
            }
            xv[(xb * 2 + p - 1) * 128 + f] = best_v;
            xk[(xb * 2 + p - 1) * 128 + f] = best_k;
            // one buffer: pipeline 0 reads it before it builds the next query,
            // which this pipeline waits for before its next write
            if (next_term) {
              xr[((p - 1) * 128 + f) * 2] = a;
              xr[((p - 1) * 128 + f) * 2 + 1] = c4;
            }
            mbar_arrive(&bar.xch_full[xb]);
            continue;
          }
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.xch_full[xb], use & 1))) {
            record_error8(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          int from = 0;  // the pipeline whose candidate won
#pragma unroll
          for (int pp = 0; pp < 2; ++pp) {
            const float ov = xv[(xb * 2 + pp) * 128 + f];
            const int ok_k = xk[(xb * 2 + pp) * 128 + f];
            if (ov < best_v || (ov == best_v && ok_k < best_k)) {
              best_v = ov;
              best_k = ok_k;
              from = pp + 1;
            }
          }
          if (next_term && from > 0) {
            a = xr[((from - 1) * 128 + f) * 2];
            c4 = xr[((from - 1) * 128 + f) * 2 + 1];
          }
          mbar_arrive(&bar.xch_free[xb]);
        }
        my_codes[q] = best_k;
        if (valid) codes[n * n_q + q] = best_k;
        if (next_term) {  // the next query's last term
          gl[0] = a.x;
          gl[1] = a.y;
          gl[2] = a.z;
          gl[3] = a.w;
          gl[4] = c4.x;
          gl[5] = c4.y;
          gl[6] = c4.z;
          gl[7] = c4.w;
        }
      }
    }
    if (npend > 0) cp_async_wait_all();  // nothing lands after the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S8_TMEM_COLS);
  }
}

std::atomic<unsigned long long> g_attr8_done{0};

cudaError_t ensure_attributes8() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (g_attr8_done.load() & bit) return cudaSuccess;
  const int smem = (int)s8_smem_bytes(kMaxKSmall);
  e = cudaFuncSetAttribute(k_search8_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_search8_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  g_attr8_done.fetch_or(bit);
  return cudaSuccess;
}

static_assert(s8_smem_bytes(kMaxKSmall) <= 227 * 1024, "d = 8 search kernel shared memory");

}  // namespace

int search8_block_stages(bool split) { return split ? S8_P * S8_TB : S8_TB; }

cudaError_t launch_search8(const rvq_dims &dm, const void *tables, const float *p0, int64_t n, int n_q, int q_begin,
                           int q_end, int32_t *codes, int *status, int sms, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  cudaError_t e = ensure_attributes8();
  if (e != cudaSuccess) return e;
  const int tiles = (int)((n + 127) / 128);
  // no more tiles than SMs: one tile per CTA, split between its three pipelines
  const bool split = search8_split(n, sms);
  const int items = split ? tiles : (tiles + S8_P - 1) / S8_P;
  const int grid = items < sms ? items : sms;
  const size_t smem = s8_smem_bytes(dm.K);
  auto kern = split ? k_search8_tc<true> : k_search8_tc<false>;
  kern<<<grid, S8_THREADS, smem, st>>>(p0, at<float>(tables, L.g), at<float>(tables, L.cb_img),
                                       at<float>(tables, L.cn_img8), codes, n, n_q, q_begin, q_end, dm.K, tiles,
                                       dm.metric, status);
  return cudaGetLastError();
}

}  // namespace rvq
