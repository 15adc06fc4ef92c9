// RVQ encode on the fifth-generation tensor cores (tcgen05 + TMEM + TMA).
//
// The encode loop of omnivoice.cpp ARCHITECTURE.md ("RVQ codec", Encode
// (residual loop)) in the re-associated form prepared by rvq_prepare:
//
//   step 1 (k_project_tc)  P0[n][q*d + j] = w_in[q][j] . x[n] + b_in[q][j]   for all q < n_q
//   step 2 (k_search_tc)   for q = 0 .. n_q-1, per frame:
//                            p_q    = P0[n][q] - sum_{s<q} G[q][s][code_s]
//                            code_q = argmin_k  ||c_k||^2 - 2 p_q . c_k   (lowest k on ties)
//
// Both contractions run as 3xTF32 on the tensor cores: a = a_hi + a_lo with
// a_hi the TF32 truncation (the tensor core truncates float32 operands to TF32,
// so a raw float32 tile serves as a_hi) and a_lo = a - a_hi exact in float32;
// a.b ~= a_hi.b_hi + a_hi.b_lo + a_lo.b_hi, accumulated in float32 in TMEM.
// That keeps the distances at about float32 accuracy; one TF32 pass (10-bit
// mantissa) would not (the pages keep the codec in F32 because reduced
// precision loses late-codebook matches: omnivoice.cpp ARCHITECTURE.md,
// "Model conversion").
//
// Every mbarrier wait is bounded; a timeout records RVQ_DEVICE_TIMEOUT in the
// scratch status word, the kernel drains its own copies and MMAs, frees TMEM
// and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "rvq_internal.cuh"
#include "sm103_ptx.cuh"

namespace rvq {
namespace {

using namespace ptx;

// ===========================================================================
// step 1: P0 = x . w_in^T + b_in
// CTA item: 256 frames (two M=128 tiles) x 256 output columns, K = D in
// slices of 16 floats (64-byte rows, 64-byte swizzle), 3-stage TMA ring.
// Warps: 0 TMA producer, 1 MMA issuer (+ TMEM owner), 2-5 lo-split + epilogue.
// ===========================================================================
constexpr int PJ_BK = 16;
constexpr int PJ_STAGES = 3;
constexpr uint32_t PJ_A_TILE = 128 * PJ_BK * 4;          // 8 KB: one tile's K-slice
constexpr uint32_t PJ_B = 256 * PJ_BK * 4;               // 16 KB
constexpr uint32_t PJ_STAGE = 4 * PJ_A_TILE + 2 * PJ_B;  // raw[2] lo[2] bhi blo = 64 KB
constexpr uint32_t PJ_TX = 2 * PJ_A_TILE + 2 * PJ_B;     // bytes TMA writes per stage
constexpr int PJ_THREADS = 192;
constexpr uint32_t PJ_IDESC = idesc_tf32(128, 256);

struct PjBars {
  uint64_t full[PJ_STAGES], conv[PJ_STAGES], empty[PJ_STAGES];
  uint64_t acc_full, acc_empty, drain;
  uint32_t tmem;
};
constexpr size_t PJ_SMEM = 1024 + PJ_STAGES * PJ_STAGE + sizeof(PjBars);

__device__ __forceinline__ void record_error(int *status, int code) { atomicCAS(status, 0, code); }

__global__ void __launch_bounds__(PJ_THREADS, 1)
    k_project_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_whi,
                 const __grid_constant__ CUtensorMap tm_wlo, const float *__restrict__ bias,
                 float *__restrict__ P0, int64_t n_rows, int n_cols, int D, int n_items, int n_cb,
                 int *__restrict__ status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  PjBars &bar = *reinterpret_cast<PjBars *>(smem + PJ_STAGES * PJ_STAGE);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nk = D / PJ_BK;
  auto a_raw = [&](int s, int t) { return smem + s * PJ_STAGE + t * PJ_A_TILE; };
  auto a_lo = [&](int s, int t) { return smem + s * PJ_STAGE + (2 + t) * PJ_A_TILE; };
  auto b_hi = [&](int s) { return smem + s * PJ_STAGE + 4 * PJ_A_TILE; };
  auto b_lo = [&](int s) { return smem + s * PJ_STAGE + 4 * PJ_A_TILE + PJ_B; };

  if (tid == 0) {
    for (int s = 0; s < PJ_STAGES; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.conv[s], 128);
      mbar_init(&bar.empty[s], 1);
    }
    mbar_init(&bar.acc_full, 1);
    mbar_init(&bar.acc_empty, 128);
    mbar_init(&bar.drain, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_whi);
    prefetch_tmap(&tm_wlo);
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int m0 = (item / n_cb) * 256, c0 = (item % n_cb) * 256;
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = it % PJ_STAGES;
          const uint32_t use = it / PJ_STAGES;
          if (use > 0 && !mbar_wait(&bar.empty[s], (use - 1) & 1)) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar.full[s], PJ_TX);
          tma_load_2d(a_raw(s, 0), &tm_x, ks * PJ_BK, m0, &bar.full[s]);
          tma_load_2d(a_raw(s, 1), &tm_x, ks * PJ_BK, m0 + 128, &bar.full[s]);
          tma_load_2d(b_hi(s), &tm_whi, ks * PJ_BK, c0, &bar.full[s]);
          tma_load_2d(b_lo(s), &tm_wlo, ks * PJ_BK, c0, &bar.full[s]);
        }
      }
      // drain: the last load issued into each stage has landed before exit
      for (uint32_t k = 0; k < PJ_STAGES && k < it; ++k) {
        const uint32_t j = it - 1 - k;
        mbar_wait(&bar.full[j % PJ_STAGES], (j / PJ_STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, n_done = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n_done) {
        if (n_done > 0 && !mbar_wait(&bar.acc_empty, (n_done - 1) & 1)) {
          record_error(status, RVQ_DEVICE_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = it % PJ_STAGES;
          if (!mbar_wait(&bar.conv[s], (it / PJ_STAGES) & 1)) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int j = 0; j < PJ_BK / 8; ++j) {
              const uint64_t ah = smem_desc(smem_addr(a_raw(s, t)) + j * 32, 16, 512, kSwizzle64B);
              const uint64_t al = smem_desc(smem_addr(a_lo(s, t)) + j * 32, 16, 512, kSwizzle64B);
              const uint64_t bh = smem_desc(smem_addr(b_hi(s)) + j * 32, 16, 512, kSwizzle64B);
              const uint64_t bl = smem_desc(smem_addr(b_lo(s)) + j * 32, 16, 512, kSwizzle64B);
              const uint32_t d = tmem + t * 256;
              mma_tf32(d, ah, bh, PJ_IDESC, (ks | j) ? 1u : 0u);
              mma_tf32(d, ah, bl, PJ_IDESC, 1u);
              mma_tf32(d, al, bh, PJ_IDESC, 1u);
            }
          mma_commit(&bar.empty[s]);
        }
        if (ok) mma_commit(&bar.acc_full);
      }
      // no MMA of this CTA may be in flight when TMEM is freed
      mma_commit(&bar.drain);
      mbar_wait(&bar.drain, 0);
    }
  } else {
    // ---------------- lo split + epilogue (warps 2..5) ----------------
    const int ct = tid - 64;                 // 0..127
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;       // row within each tile
    uint32_t it = 0, n_done = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n_done) {
      const int64_t m0 = (int64_t)(item / n_cb) * 256;
      const int c0 = (item % n_cb) * 256;
      for (int ks = 0; ks < nk; ++ks, ++it) {
        const int s = it % PJ_STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar.full[s], (it / PJ_STAGES) & 1))) {
          record_error(status, RVQ_DEVICE_TIMEOUT);
          ok = false;
          break;
        }
        // lo = a - trunc_tf32(a), element-wise over both tiles' raw slices
        const float4 *src = reinterpret_cast<const float4 *>(a_raw(s, 0));
        float4 *dst = reinterpret_cast<float4 *>(a_lo(s, 0));
#pragma unroll
        for (int u = 0; u < (2 * PJ_A_TILE / 16) / 128; ++u) {
          const float4 v = src[ct + u * 128];
          float4 l;
          l.x = v.x - __uint_as_float(__float_as_uint(v.x) & 0xffffe000u);
          l.y = v.y - __uint_as_float(__float_as_uint(v.y) & 0xffffe000u);
          l.z = v.z - __uint_as_float(__float_as_uint(v.z) & 0xffffe000u);
          l.w = v.w - __uint_as_float(__float_as_uint(v.w) & 0xffffe000u);
          dst[ct + u * 128] = l;
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar.conv[s]);
      }
      if (!ok) break;
      // warp-uniform decision before the warp-collective TMEM loads
      if (!__all_sync(0xffffffffu, mbar_wait(&bar.acc_full, n_done & 1))) {
        record_error(status, RVQ_DEVICE_TIMEOUT);
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        const int64_t n = m0 + t * 128 + r;
        float *out = P0 + n * n_cols + c0;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + t * 256 + c, v);
          tmem_wait_ld();
          if (n < n_rows && c0 + c < n_cols) {
            const float4 *b4 = reinterpret_cast<const float4 *>(bias + c0 + c);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 b = __ldg(b4 + u);
              reinterpret_cast<float4 *>(out + c)[u] =
                  make_float4(v[4 * u] + b.x, v[4 * u + 1] + b.y, v[4 * u + 2] + b.z, v[4 * u + 3] + b.w);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar.acc_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// step 2: the stage loop in code space.
// CTA item: one tile of 128 frames; two CTAs share each SM's tensor core, so
// one CTA's stage boundaries and distance scans overlap the other's MMAs.
// The query tile (A operand, hi and lo) lives in TMEM, written by the row
// threads with tcgen05.st; shared memory holds only a ring of codebook
// half-chunks: 128 codewords of -2*c, hi or lo, pre-swizzled, 32 KB per bulk
// copy.  TMEM (256 columns): [0,64) A hi, [64,128) A lo, [128,256) distances.
// Warps: 0 bulk-copy producer, 1 MMA issuer (+ TMEM owner), 2-5 one thread per
// frame row: build the stage's query, then scan the distances.
// ===========================================================================
constexpr int SR_KC = 128;
constexpr int SR_STAGES = 3;
constexpr uint32_t SR_ATOM = 128 * 128;      // 128 rows x 128 B
constexpr uint32_t SR_B_STAGE = 2 * SR_ATOM;  // [atom] = 32 KB
constexpr int SR_THREADS = 192;
constexpr uint32_t SR_TMEM_COLS = 256;
constexpr uint32_t SR_A_HI = 0, SR_A_LO = 64, SR_ACC = 128;
constexpr uint32_t SR_IDESC = idesc_tf32(128, SR_KC);

constexpr int SR_MAX_K = 1024;  // codewords whose norms fit the per-stage smem copy (larger K reads global)
struct SrBars {
  uint64_t b_full[SR_STAGES], b_empty[SR_STAGES];
  uint64_t a_ready, acc_full, acc_empty, drain;
  uint32_t tmem;
};
constexpr size_t SR_CN_BYTES = SR_MAX_K * 4;        // ||c||^2 of the current stage
constexpr int SR_XPOSE_LD = 20;                       // floats per row of a warp's transpose scratch (16 + pad)
constexpr size_t SR_XPOSE_BYTES = 4 * 32 * SR_XPOSE_LD * 4;  // 4 row warps x 32 frames
constexpr size_t SR_SMEM = 1024 + SR_STAGES * SR_B_STAGE + SR_CN_BYTES + SR_XPOSE_BYTES + sizeof(SrBars);

__global__ void __launch_bounds__(SR_THREADS, 2)
    k_search_tc(const float *__restrict__ P0, const float *__restrict__ G, const float *__restrict__ cb_img,
                const float *__restrict__ cnorm, int32_t *__restrict__ codes, int64_t n_rows, int n_q, int K,
                int n_items, int *__restrict__ status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  float *cn_smem = reinterpret_cast<float *>(smem + SR_STAGES * SR_B_STAGE);
  float *xpose = reinterpret_cast<float *>(smem + SR_STAGES * SR_B_STAGE + SR_CN_BYTES);
  SrBars &bar = *reinterpret_cast<SrBars *>(smem + SR_STAGES * SR_B_STAGE + SR_CN_BYTES + SR_XPOSE_BYTES);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkc = K / SR_KC;
  // Every CTA walks the same codebook chunks; starting each CTA at a different
  // chunk spreads the simultaneous bulk copies over nkc chunks of L2 instead
  // of one hot chunk.  The argmin merge below is order-independent.
  const int rot = blockIdx.x % nkc;
  constexpr int d = kCodeDim;

  if (tid == 0) {
    for (int s = 0; s < SR_STAGES; ++s) {
      mbar_init(&bar.b_full[s], 1);
      mbar_init(&bar.b_empty[s], 1);
    }
    mbar_init(&bar.a_ready, 128);
    mbar_init(&bar.acc_full, 1);
    mbar_init(&bar.acc_empty, 128);
    mbar_init(&bar.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem, SR_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem;

  if (warp == 0) {
    // ---------------- producer: codebook half-chunk images ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x)
        for (int q = 0; q < n_q && ok; ++q)
          for (int c = 0; c < nkc && ok; ++c)
            for (int h = 0; h < 2; ++h, ++it) {
              const int cr = (c + rot) % nkc;
              const int s = it % SR_STAGES;
              const uint32_t use = it / SR_STAGES;
              if (use > 0 && !mbar_wait(&bar.b_empty[s], (use - 1) & 1)) {
                record_error(status, RVQ_DEVICE_TIMEOUT);
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&bar.b_full[s], SR_B_STAGE);
              const float *src = cb_img + ((((size_t)q * nkc + cr) * 2 + h) * SR_B_STAGE) / 4;
              bulk_g2s(smem + s * SR_B_STAGE, src, SR_B_STAGE, &bar.b_full[s]);
            }
      for (uint32_t k = 0; k < SR_STAGES && k < it; ++k) {
        const uint32_t j = it - 1 - k;
        mbar_wait(&bar.b_full[j % SR_STAGES], (j / SR_STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, cc = 0, builds = 0;
      bool ok = true;
      auto wait_or_fail = [&](uint64_t *b, uint32_t parity) {
        if (!mbar_wait(b, parity)) {
          record_error(status, RVQ_DEVICE_TIMEOUT);
          ok = false;
        }
        return ok;
      };
      // descriptor of the smem base; operand descriptors add (byte offset >> 4)
      const uint64_t desc0 = smem_desc(smem_addr(smem), 16, 1024, kSwizzle128B);
      auto dB = [&](int s, int ks) {
        return desc0 + (uint64_t)((s * SR_B_STAGE + (ks >> 2) * SR_ATOM + (ks & 3) * 32) >> 4);
      };
      const uint32_t acc = tmem + SR_ACC;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x)
        for (int q = 0; q < n_q && ok; ++q, ++builds)
          for (int c = 0; c < nkc && ok; ++c, ++cc) {
            if (cc > 0 && !wait_or_fail(&bar.acc_empty, (cc - 1) & 1)) break;
            // hi half: a_hi . b_hi + a_lo . b_hi
            int s = it % SR_STAGES;
            if (!wait_or_fail(&bar.b_full[s], (it / SR_STAGES) & 1)) break;
            if (c == 0 && !wait_or_fail(&bar.a_ready, builds & 1)) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < d / 8; ++ks) {
              const uint64_t bh = dB(s, ks);
              mma_tf32_ta(acc, tmem + SR_A_HI + ks * 8, bh, SR_IDESC, ks ? 1u : 0u);
              mma_tf32_ta(acc, tmem + SR_A_LO + ks * 8, bh, SR_IDESC, 1u);
            }
            mma_commit(&bar.b_empty[s]);
            ++it;
            // lo half: a_hi . b_lo
            s = it % SR_STAGES;
            if (!wait_or_fail(&bar.b_full[s], (it / SR_STAGES) & 1)) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < d / 8; ++ks) mma_tf32_ta(acc, tmem + SR_A_HI + ks * 8, dB(s, ks), SR_IDESC, 1u);
            mma_commit(&bar.acc_full);
            mma_commit(&bar.b_empty[s]);
            ++it;
          }
      mma_commit(&bar.drain);
      mbar_wait(&bar.drain, 0);
    }
  } else {
    // ---------------- one thread per frame row (warps 2..5) ----------------
    // Stage q's query is p_q = P0[n][q] - sum_{s<q} G[q][s][code_s], built
    // between stages (the co-resident CTA keeps the tensor core busy meanwhile).
    const int quarter = warp & 3;       // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;  // row within the tile = TMEM lane
    const int rt = tid - 64;            // 0..127
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int64_t ld = (int64_t)n_q * d;
    const bool cn_in_smem = K <= SR_MAX_K;
    uint32_t cc = 0, stage_count = 0;
    bool ok = true;
    int my_codes[kMaxStages];
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int64_t n = (int64_t)item * 128 + r;
      const bool valid = n < n_rows;
      for (int q = 0; q < n_q && ok; ++q, ++stage_count) {
        // ---- query p_q = P0[n][q] - sum_{s<q} G[q][s][code_s], rows read cooperatively:
        //      four lanes read 64 contiguous bytes of one frame's row (8 rows per warp
        //      instruction), and a per-warp shared-memory transpose hands every lane
        //      its own frame's 64 values.  Terms are added in the same order as a
        //      plain per-thread sum.
        {
          float p[d];
#pragma unroll
          for (int u = 0; u < d; ++u) p[u] = 0.f;
          float *xs = xpose + (warp - 2) * 32 * SR_XPOSE_LD;
          auto coop_accumulate = [&](const float *row, bool add) {
            const unsigned long long mine = reinterpret_cast<unsigned long long>(row);
            const int j = lane & 3;
            // all 16 loads of this lane in flight at once: frames (lane/4) + 8i, dims 16b + 4j
            float4 vb[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float *src =
                  reinterpret_cast<const float *>(__shfl_sync(0xffffffffu, mine, (lane >> 2) + 8 * i));
#pragma unroll
              for (int b = 0; b < d / 16; ++b) vb[4 * b + i] = __ldg(reinterpret_cast<const float4 *>(src + 16 * b + 4 * j));
            }
#pragma unroll
            for (int b = 0; b < d / 16; ++b) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4 *>(xs + ((lane >> 2) + 8 * i) * SR_XPOSE_LD + 4 * j) = vb[4 * b + i];
              __syncwarp();
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float4 v = *reinterpret_cast<const float4 *>(xs + lane * SR_XPOSE_LD + 4 * u);
                if (add) {
                  p[16 * b + 4 * u] += v.x;
                  p[16 * b + 4 * u + 1] += v.y;
                  p[16 * b + 4 * u + 2] += v.z;
                  p[16 * b + 4 * u + 3] += v.w;
                } else {
                  p[16 * b + 4 * u] -= v.x;
                  p[16 * b + 4 * u + 1] -= v.y;
                  p[16 * b + 4 * u + 2] -= v.z;
                  p[16 * b + 4 * u + 3] -= v.w;
                }
              }
              __syncwarp();
            }
          };
          // invalid frames read a valid row and discard the result
          coop_accumulate(P0 + (valid ? n : 0) * ld + q * d, true);
          for (int s = 0; s < q; ++s)
            coop_accumulate(G + (pair_index(q, s) * K + (valid ? my_codes[s] : 0)) * d, false);
          if (!valid) {
#pragma unroll
            for (int u = 0; u < d; ++u) p[u] = 0.f;
          }
          // A operand: raw (= hi after TF32 truncation) and lo parts into this row's TMEM lane
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float lo[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float v = p[32 * h + i];
              lo[i] = v - __uint_as_float(__float_as_uint(v) & 0xffffe000u);
            }
            tmem_st32(lane_base + SR_A_HI + 32 * h, *reinterpret_cast<const float(*)[32]>(&p[32 * h]));
            tmem_st32(lane_base + SR_A_LO + 32 * h, lo);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar.a_ready);
        }
        // the next stage's projections do not depend on this stage's code: pull them into L2 now
        if (valid && q + 1 < n_q) {
          const float *nxt = P0 + n * ld + (q + 1) * d;
          prefetch_l2(nxt);
          prefetch_l2(nxt + 32);
        }
        // ---- this stage's squared norms into smem, between two barriers of the row
        //      threads (every row thread has finished the previous stage's scan)
        const float *cnq = cnorm + (int64_t)q * K;
        float *cns = cn_smem;
        if (cn_in_smem) {
          asm volatile("bar.sync 1, 128;" ::: "memory");
          for (int e = rt * 4; e < K; e += 128 * 4)
            *reinterpret_cast<float4 *>(cns + e) = __ldg(reinterpret_cast<const float4 *>(cnq + e));
          asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        const float *cnsrc = cn_in_smem ? cns : cnq;
        // ---- scan the K distances ||c||^2 - 2 p.c; keep the lexicographic (value, index) minimum
        float best_v = __int_as_float(0x7f800000);
        int best_k = 0;
        for (int c = 0; c < nkc; ++c, ++cc) {
          const int cr = (c + rot) % nkc;
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.acc_full, cc & 1))) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          float v[SR_KC];
#pragma unroll
          for (int g = 0; g < SR_KC / 32; ++g)
            tmem_ld32(lane_base + SR_ACC + g * 32, *reinterpret_cast<float(*)[32]>(&v[32 * g]));
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bar.acc_empty);  // the accumulator is free: the values are in registers
          const float4 *cn4 = reinterpret_cast<const float4 *>(cnsrc + cr * SR_KC);
#pragma unroll
          for (int u = 0; u < SR_KC / 4; ++u) {
            const float4 cn = cn4[u];
            v[4 * u] += cn.x;
            v[4 * u + 1] += cn.y;
            v[4 * u + 2] += cn.z;
            v[4 * u + 3] += cn.w;
          }
          float mm[SR_KC / 2];
#pragma unroll
          for (int i = 0; i < SR_KC / 2; ++i) mm[i] = fminf(v[2 * i], v[2 * i + 1]);
#pragma unroll
          for (int w2 = SR_KC / 4; w2 >= 1; w2 >>= 1)
#pragma unroll
            for (int i = 0; i < w2; ++i) mm[i] = fminf(mm[i], mm[i + w2]);
          const float m = mm[0];
          if (m <= best_v) {  // rare after the first chunks: locate the first index holding m
            int first = SR_KC - 1;
#pragma unroll
            for (int i = SR_KC - 1; i >= 0; --i)
              if (v[i] == m) first = i;
            const int k = cr * SR_KC + first;
            if (m < best_v || k < best_k) {
              best_v = m;
              best_k = k;
            }
          }
        }
        if (!ok) break;
        my_codes[q] = best_k;
        if (valid) codes[n * n_q + q] = best_k;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, SR_TMEM_COLS);
  }
}

// ===========================================================================
// host side
// ===========================================================================
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::once_flag g_encode_once;

cudaError_t tensor_map_2d(CUtensorMap *map, const float *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                          uint32_t box_outer, CUtensorMapSwizzle sw) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode_tiled) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * sizeof(float)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
                              es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

std::atomic<unsigned long long> g_attr_done{0};

cudaError_t ensure_attributes() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (g_attr_done.load() & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(k_project_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PJ_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_search_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SR_SMEM);
  if (e != cudaSuccess) return e;
  g_attr_done.fetch_or(bit);
  return cudaSuccess;
}

int sm_count() {
  static std::atomic<int> cached{0};
  int v = cached.load();
  if (v) return v;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
  cached.store(v);
  return v;
}

}  // namespace

cudaError_t launch_encode_chunk(const rvq_dims &dm, const void *tables, const float *x, int64_t n0, int64_t n,
                                int n_q, int32_t *codes, float *p0, int *status, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  const int D = dm.D, d = dm.d, K = dm.K, Q = dm.Q;
  const int n_cols = n_q * d;
  cudaError_t e = ensure_attributes();
  if (e != cudaSuccess) return e;
  CUtensorMap tm_x, tm_whi, tm_wlo;
  if ((e = tensor_map_2d(&tm_x, x + n0 * D, (uint64_t)D, (uint64_t)n, PJ_BK, 128, CU_TENSOR_MAP_SWIZZLE_64B)) !=
      cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&tm_whi, at<float>(tables, L.w_in_hi), (uint64_t)D, (uint64_t)Q * d, PJ_BK, 256,
                         CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&tm_wlo, at<float>(tables, L.w_in_lo), (uint64_t)D, (uint64_t)Q * d, PJ_BK, 256,
                         CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess)
    return e;
  const int n_pairs_rows = (int)((n + 255) / 256);
  const int n_cb = (n_cols + 255) / 256;
  const int items1 = n_pairs_rows * n_cb;
  const int sms = sm_count();
  k_project_tc<<<items1 < sms ? items1 : sms, PJ_THREADS, PJ_SMEM, st>>>(
      tm_x, tm_whi, tm_wlo, at<float>(tables, L.b_in), p0, n, n_cols, D, items1, n_cb, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int tiles = (int)((n + 127) / 128);
  k_search_tc<<<tiles < 2 * sms ? tiles : 2 * sms, SR_THREADS, SR_SMEM, st>>>(
      p0, at<float>(tables, L.g), at<float>(tables, L.cb_img), at<float>(tables, L.cnorm), codes + n0 * n_q, n, n_q,
      K, tiles, status);
  return cudaGetLastError();
}

}  // namespace rvq
