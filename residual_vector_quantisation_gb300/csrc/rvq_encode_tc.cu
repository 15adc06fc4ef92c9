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
// mantissa) would not (the codec is kept in F32 because reduced
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
// CTA item: NT tiles of 128 frames x NC output columns (NT = 2, NC = 256 for
// large calls; one tile and 128 or 64 columns when a call has too few such
// items to fill the GPU), K = D in slices of 16 floats (64-byte rows, 64-byte
// swizzle), 3-stage TMA ring.  The smaller items keep two accumulators in
// TMEM, so an item's epilogue overlaps the next item's MMAs (moss_lfq encode
// 268 -> 259 us).
// Warps: 0 and 6 TMA producers (x tiles; w_in hi and lo tiles -- a thread's
// copies are carried out one after another, so two threads issue them),
// 1 MMA issuer (+ TMEM owner), 2-5 lo-split + epilogue, and for the 256 x 256
// items, whose one accumulator makes the next item's MMAs wait for the
// epilogue, 7-10 a second epilogue crew that takes the second tile's steps
// (large_batch encode 1.406 -> 1.381 ms).
// ===========================================================================
constexpr int PJ_BK = 16;
constexpr int PJ_STAGES = 3;
constexpr uint32_t PJ_A_TILE = 128 * PJ_BK * 4;  // 8 KB: one tile's K-slice
constexpr uint32_t PJ_BLK = 32 * 32 * 4;       // a 32 x 32 block per epilogue warp

template <int NT, int NC>
struct PjShape {
  static constexpr uint32_t B = NC * PJ_BK * 4;                      // one w_in part's K-slice
  static constexpr uint32_t STAGE = 2 * NT * PJ_A_TILE + 2 * B;      // raw[NT] lo[NT] bhi blo
  static constexpr uint32_t TX_X = NT * PJ_A_TILE;                   // bytes each producer's TMA writes per stage
  static constexpr uint32_t TX_W = 2 * B;
  static constexpr uint32_t ACC_COLS = NT * NC;                      // one item's accumulators
  // two accumulators when they fit TMEM, so an item's epilogue overlaps the
  // next item's MMAs
  static constexpr uint32_t ACC_BUFS = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr uint32_t TMEM_COLS = ACC_BUFS * ACC_COLS;
  static constexpr uint32_t IDESC = idesc_tf32(128, NC);
  static constexpr int ROWS = 128 * NT;                              // frames per item
  // one-accumulator items: four more warps share the epilogue
  static constexpr int HELP = ACC_BUFS == 1 ? 4 : 0;
  static constexpr int THREADS = 224 + 32 * HELP;
  static constexpr uint32_t EPI = (4 + HELP) * PJ_BLK;
};

struct PjBars {
  uint64_t full[PJ_STAGES], conv[PJ_STAGES], empty[PJ_STAGES];
  uint64_t acc_full[2], acc_empty[2], drain;
  uint32_t tmem;
};
template <int NT, int NC>
constexpr size_t pj_smem() { return 1024 + PJ_STAGES * PjShape<NT, NC>::STAGE + PjShape<NT, NC>::EPI + sizeof(PjBars); }

__device__ __forceinline__ void record_error(int *status, int code) { atomicCAS(status, 0, code); }

// zero_status: clear the status word first (a call whose first kernel this
// is); the kernel also lets a dependent launch start at once (programmatic
// dependent launch; no effect on a plain launch after it).
template <int NT, int NC>
__global__ void __launch_bounds__(PjShape<NT, NC>::THREADS, 1)
    k_project_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_whi,
                 const __grid_constant__ CUtensorMap tm_wlo, const float *__restrict__ bias,
                 float *__restrict__ P0, int64_t n_rows, int n_cols, int D, int n_items, int n_cb,
                 int *__restrict__ status, int zero_status) {
  using S = PjShape<NT, NC>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  PjBars &bar = *reinterpret_cast<PjBars *>(smem + PJ_STAGES * S::STAGE + S::EPI);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_launch_dependents();
  if (zero_status && blockIdx.x == 0 && tid == 0) *status = 0;
  const int nk = D / PJ_BK;
  auto a_raw = [&](int s, int t) { return smem + s * S::STAGE + t * PJ_A_TILE; };
  auto a_lo = [&](int s, int t) { return smem + s * S::STAGE + (NT + t) * PJ_A_TILE; };
  auto b_hi = [&](int s) { return smem + s * S::STAGE + 2 * NT * PJ_A_TILE; };
  auto b_lo = [&](int s) { return smem + s * S::STAGE + 2 * NT * PJ_A_TILE + S::B; };

  if (tid == 0) {
    for (int s = 0; s < PJ_STAGES; ++s) {
      mbar_init(&bar.full[s], 2);  // one arrival per producer
      mbar_init(&bar.conv[s], 128);
      mbar_init(&bar.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar.acc_full[b], 1);
      mbar_init(&bar.acc_empty[b], S::HELP ? 256 : 128);
    }
    mbar_init(&bar.drain, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_whi);
    prefetch_tmap(&tm_wlo);
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem, S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem;

  // this warp's 32 x 32 block: row i's 16-byte piece j at i * 8 + (j ^ (i & 7)),
  // so both the row-wise writes and the column-wise reads below are free of
  // bank conflicts
  const int quarter = warp & 3;  // TMEM lanes this warp may access (epilogue warps)
  const int ew = warp >= 2 && warp <= 5 ? warp - 2 : warp >= 7 ? warp - 3 : 0;  // epilogue warp index
  float4 *blk = reinterpret_cast<float4 *>(smem + PJ_STAGES * S::STAGE) + ew * 256;
  // One epilogue step: 32 columns of one tile of an item's accumulator,
  // + bias, to P0 (e < NT * NC / 32).  Lane i holds row i of the warp's 32
  // rows; the block goes through shared memory so that each store
  // instruction writes four whole 128-byte row pieces (lane i: row
  // 4u + i / 8, piece i % 8) instead of 32 pieces of 16 bytes in 32 lines.
  // A 256 x 256 item keeps one accumulator, so the next item's MMAs wait
  // for its epilogue: large_batch encode 1.465 -> 1.416 ms with the block
  // transpose, -> 1.394 ms with the bias loads out of the steps' dependency
  // chain.  (A TMA store of each block, the bias added before the block is
  // written, measured the same: 1.403-1.405 against 1.405-1.412 ms.)
  constexpr int NE = NT * NC / 32, NCS = NC / 32;
  const int pc = lane & 7;
  // this lane's four bias values of step e (zero past the last column; n_cols
  // is a multiple of 8, n_q * d, so a step may end inside the row)
  auto bias4 = [&](int item_e, int e) {
    const int cc = (item_e % n_cb) * NC + (e % NCS) * 32;
    return cc < n_cols && pc < min(8, (n_cols - cc) / 4) ? __ldg(reinterpret_cast<const float4 *>(bias + cc) + pc)
                                                         : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  auto epi_load = [&](uint32_t ab, int e, float (&v)[32]) {
    tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + ab * S::ACC_COLS + (e / NCS) * NC + (e % NCS) * 32, v);
  };
  // v (loaded and waited for) + b to P0
  auto epi_put = [&](int item_e, int e, const float (&v)[32], float4 b) {
    const int64_t n0 = (int64_t)(item_e / n_cb) * S::ROWS + (e / NCS) * 128 + quarter * 32;
    const int c0 = (item_e % n_cb) * NC, c = (e % NCS) * 32;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      blk[lane * 8 + (j ^ (lane & 7))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    if (c0 + c < n_cols && pc < min(8, (n_cols - (c0 + c)) / 4)) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = 4 * u + (lane >> 3);
        if (n0 + i < n_rows) {
          const float4 a = blk[i * 8 + (pc ^ (i & 7))];
          reinterpret_cast<float4 *>(P0 + (n0 + i) * n_cols + c0 + c)[pc] =
              make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
        }
      }
    }
    __syncwarp();  // the block is read before the next step writes it
  };
  // a single step (two-accumulator items, between lo splits), its bias load
  // overlapping the TMEM load
  auto epi_step = [&](int item_e, uint32_t ab, int e) {
    float v[32];
    epi_load(ab, e, v);
    const float4 b = bias4(item_e, e);
    tmem_wait_ld();
    epi_put(item_e, e, v, b);
  };
  if (warp == 0 || warp == 6) {
    // ---------------- TMA producers ----------------
    const bool px = warp == 0;
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int m0 = (item / n_cb) * S::ROWS, c0 = (item % n_cb) * NC;
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = it % PJ_STAGES;
          const uint32_t use = it / PJ_STAGES;
          if (use > 0 && !mbar_wait(&bar.empty[s], (use - 1) & 1)) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          if (px) {
            mbar_arrive_expect_tx(&bar.full[s], S::TX_X);
#pragma unroll
            for (int t = 0; t < NT; ++t) tma_load_2d(a_raw(s, t), &tm_x, ks * PJ_BK, m0 + 128 * t, &bar.full[s]);
          } else {
            mbar_arrive_expect_tx(&bar.full[s], S::TX_W);
            tma_load_2d(b_hi(s), &tm_whi, ks * PJ_BK, c0, &bar.full[s]);
            tma_load_2d(b_lo(s), &tm_wlo, ks * PJ_BK, c0, &bar.full[s]);
          }
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
        const uint32_t ab = n_done % S::ACC_BUFS, au = n_done / S::ACC_BUFS;  // accumulator, its use
        if (au > 0 && !mbar_wait(&bar.acc_empty[ab], (au - 1) & 1)) {
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
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int j = 0; j < PJ_BK / 8; ++j) {
              const uint64_t ah = smem_desc(smem_addr(a_raw(s, t)) + j * 32, 16, 512, kSwizzle64B);
              const uint64_t al = smem_desc(smem_addr(a_lo(s, t)) + j * 32, 16, 512, kSwizzle64B);
              const uint64_t bh = smem_desc(smem_addr(b_hi(s)) + j * 32, 16, 512, kSwizzle64B);
              const uint64_t bl = smem_desc(smem_addr(b_lo(s)) + j * 32, 16, 512, kSwizzle64B);
              const uint32_t d = tmem + ab * S::ACC_COLS + t * NC;
              mma_tf32(d, ah, bh, S::IDESC, (ks | j) ? 1u : 0u);
              mma_tf32(d, ah, bl, S::IDESC, 1u);
              mma_tf32(d, al, bh, S::IDESC, 1u);
            }
          mma_commit(&bar.empty[s]);
        }
        if (ok) mma_commit(&bar.acc_full[ab]);
      }
      // no MMA of this CTA may be in flight when TMEM is freed
      mma_commit(&bar.drain);
      mbar_wait(&bar.drain, 0);
    }
  } else if (warp <= 5) {
    // ---------------- lo split + epilogue (warps 2..5) ----------------
    const int ct = tid - 64;                 // 0..127
    // With two accumulators, an item's epilogue is done a step at a time
    // between the lo splits of the next item (once its MMAs are seen
    // complete), so the tensor core does not wait for it; with one, the
    // next item's MMAs need the accumulator, and it is done at once.
    int pend = -1, pend_done = 0;        // the item whose epilogue is pending, steps done
    uint32_t pend_ab = 0, pend_au = 0;   // its accumulator and that accumulator's use
    bool pend_ready = false;             // its MMAs are seen complete
    auto finish_pending = [&]() -> bool {
      if (pend < 0) return true;
      // warp-uniform decision before the warp-collective TMEM loads
      if (!pend_ready) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bar.acc_full[pend_ab], pend_au & 1))) {
          record_error(status, RVQ_DEVICE_TIMEOUT);
          return false;
        }
        tc_fence_after();
      }
      // the remaining steps, with the item's bias loaded beforehand (one
      // dependent bias load per step cost 1.3 % of a large_batch encode)
      float4 bq[NCS];
#pragma unroll
      for (int k = 0; k < NCS; ++k) bq[k] = bias4(pend, k);
#pragma unroll
      for (int e = 0; e < (S::HELP ? NE / 2 : NE); ++e) {
        if (e < pend_done) continue;
        float v[32];
        epi_load(pend_ab, e, v);
        tmem_wait_ld();
        epi_put(pend, e, v, bq[e % NCS]);
      }
      pend_done = NE;
      tc_fence_before();
      mbar_arrive(&bar.acc_empty[pend_ab]);
      pend = -1;
      return true;
    };
    uint32_t it = 0, n_done = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n_done) {
      for (int ks = 0; ks < nk; ++ks, ++it) {
        const int s = it % PJ_STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&bar.full[s], (it / PJ_STAGES) & 1))) {
          record_error(status, RVQ_DEVICE_TIMEOUT);
          ok = false;
          break;
        }
        // lo = a - trunc_tf32(a), element-wise over the tiles' raw slices
        const float4 *src = reinterpret_cast<const float4 *>(a_raw(s, 0));
        float4 *dst = reinterpret_cast<float4 *>(a_lo(s, 0));
#pragma unroll
        for (int u = 0; u < (NT * PJ_A_TILE / 16) / 128; ++u) {
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
        if (S::ACC_BUFS == 2 && pend >= 0 && pend_done < NE) {
          if (!pend_ready) {
            pend_ready = __all_sync(0xffffffffu, mbar_test_wait(&bar.acc_full[pend_ab], pend_au & 1));
            if (pend_ready) tc_fence_after();
          }
          if (pend_ready) epi_step(pend, pend_ab, pend_done++);
        }
      }
      if (!ok) break;
      if (!finish_pending()) {  // the previous item's epilogue (two accumulators)
        ok = false;
        break;
      }
      pend = item;
      pend_ab = n_done % S::ACC_BUFS;
      pend_au = n_done / S::ACC_BUFS;
      pend_done = 0;
      pend_ready = false;
      if (S::ACC_BUFS == 1 && !finish_pending()) {  // one accumulator: this item's epilogue now
        ok = false;
        break;
      }
    }
    if (ok) finish_pending();  // the last item's
  } else if (S::HELP) {
    // ---------------- epilogue helpers (warps 7..10): the second half of each
    // one-accumulator item's steps
    uint32_t n_done = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++n_done) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bar.acc_full[0], n_done & 1))) {
        record_error(status, RVQ_DEVICE_TIMEOUT);
        break;
      }
      tc_fence_after();
      float4 bq[NCS];
#pragma unroll
      for (int k = 0; k < NCS; ++k) bq[k] = bias4(item, k);
#pragma unroll
      for (int e = NE / 2; e < NE; ++e) {
        float v[32];
        epi_load(0, e, v);
        tmem_wait_ld();
        epi_put(item, e, v, bq[e % NCS]);
      }
      tc_fence_before();
      mbar_arrive(&bar.acc_empty[0]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

// ===========================================================================
// step 2: the stage loop in code space.
// CTA item: two tiles of 128 frames that walk the same codebook chunks, so
// every chunk brought into shared memory feeds both (half the L2 traffic of
// one tile per copy).  The two tiles' MMA issuers take turns chunk by chunk,
// so the tensor core works on one tile's chunk while the other tile scans its
// distances.
//   * a ring of three (split: five) 32 KB half-chunks, each brought in by two
//     16 KB bulk copies from two threads (a thread's copies run one after
//     another, each in about the same time whatever its size): a chunk is
//     128 codewords of -2*c as four atoms of 128 rows x 128 B, pre-swizzled --
//     hi dims 0-31, hi 32-63 (hi half), lo 0-31, lo 32-63 (lo half); the lo
//     half is copied and used first;
//   * per tile: the partial sum of the next query (32 KB) and a staging area
//     for one row per frame (32 KB);
//   * ||c||^2 of the last three chunks (512 B each, one bulk copy per chunk);
//   * TMEM, 256 columns per tile: [0,64) query hi, [64,128) query lo,
//     [128,256) distances;
//   * warps: 0 and 11 producers (bulk copies), 1 and 10 MMA issuers of tiles 0
//     and 1, 2-5 rows of tile 0, 6-9 rows of tile 1 (one thread per frame:
//     build the query, scan the distances).
// The query of stage q+1 is p = P0[n][q+1] - sum_{s<=q} G[q+1][s][code_s].
// All of it but the last term is known while stage q is being scanned, so
// the row warps gather those rows between distance chunks: 16-byte
// asynchronous copies (four lanes per 64-byte row segment) into the staging
// area, subtracted from the partial sum one chunk later (the P0 row is copied
// straight into the partial); at the stage boundary the staging area takes
// the one row of the code just found, copied the same way, and the query is
// formed in registers.
// Terms are added in the order s = 0, 1, ..., q.  A launch over a block of
// stages [q_begin, q_end) of a deep stack finds the terms of the earlier
// blocks already subtracted from P0 (k_cross_terms) and sums from q_begin.
// A launch with no more tiles than SMs (the SPLIT variant, for a stage of an
// even number of chunks) gives each CTA one tile and splits it: both
// pipelines work on that tile, pipeline t taking the chunks c = t mod 2, so
// the issuers still take turns.
// Only pipeline 0 builds the query; both MMA issuers read it from pipeline
// 0's TMEM columns, and tile 1's shared-memory areas become two more ring
// slots.  At the end of a stage pipeline 1 hands its per-frame (value,
// index) minimum to pipeline 0 through TMEM (two of its own query columns,
// unused when split), and pipeline 0 keeps the lexicographic minimum of the
// two.  (Otherwise a CTA's last item may hold one tile alone; it runs on
// pipeline 0 with no turns.  It ends no later than the two-tile items of the
// other CTAs, so splitting it would not shorten the launch.)
// A launch with no more tiles than the GPU holds clusters of two CTAs (and
// a multiple of four chunks a stage) runs each tile on a CTA pair instead:
// the same split item on both SMs of a cluster, each taking half the chunks,
// so a call of up to about 76 tiles uses all the SMs' tensor cores.
// ===========================================================================
constexpr int SR_KC = 128;                    // codewords per chunk (MMA N)
constexpr uint32_t SR_ATOM = 128 * 128;       // 128 codewords x 128 B
constexpr uint32_t SR_HALF = 2 * SR_ATOM;     // hi or lo part of a chunk
constexpr int SR_COPY_PIECES = 2;             // bulk copies (and producer threads) per half-chunk
constexpr int SR_SLOTS = 3;                   // half-chunks in the ring
constexpr int SR_SLOTS_SPLIT = 5;             // ... when every item is split: plus tile 1's two areas
constexpr int SR_SLOTS_CPAIR = 4;             // ... split across a CTA pair: tile 1's staging area holds the pair's minima
constexpr int SR_THREADS = 384;
constexpr uint32_t SR_TMEM_COLS = 512;        // 256 per tile
constexpr uint32_t SR_TILE_COLS = 256;
constexpr uint32_t SR_A_HI = 0, SR_A_LO = 64, SR_ACC = 128;
constexpr uint32_t SR_IDESC = idesc_tf32(128, SR_KC);
constexpr uint32_t SR_RING_BYTES = SR_SLOTS * SR_HALF;
constexpr uint32_t SR_PART_BYTES = 128 * kCodeDim * 4;  // per tile: [128 rows][16 float4 slots], slot ^ (row & 7)
constexpr int SR_CN_SLOTS = 3;
constexpr uint32_t SR_CN_BYTES = SR_KC * 4;              // ||c||^2 of one chunk

struct SrBars {
  uint64_t b_full[SR_SLOTS_SPLIT], b_empty[SR_SLOTS_SPLIT];
  uint64_t cn_full[SR_CN_SLOTS], cn_free[SR_CN_SLOTS];
  uint64_t a_ready[2], acc_full[2], acc_empty[2];
  uint64_t turn[2];  // turn[t]: the other tile's issuer has issued most of its chunk
  uint64_t drain[2];
  uint64_t xch_full[2], xch_free[2];  // split items: pipeline 1's stage minima (in TMEM), double-buffered
  uint64_t px_full[2];                // CTA pairs: the other CTA's stage minima have landed, double-buffered
  uint64_t p1t_full;                  // split items: pipeline 1's share of the next query's terms is in TMEM
  uint32_t tmem;
  uint32_t pad;
};
// ring, tile 1's partial and staging (the ring's slots 3 and 4 when every item
// is split), tile 0's partial and staging, norms, barriers
static_assert(SR_RING_BYTES + 2 * SR_PART_BYTES == SR_SLOTS_SPLIT * SR_HALF, "split ring");
constexpr size_t SR_SMEM = 1024 + SR_RING_BYTES + 4 * SR_PART_BYTES + SR_CN_SLOTS * SR_CN_BYTES + sizeof(SrBars);
static_assert(SR_SMEM <= 227 * 1024, "search kernel shared memory");

// MODE 0: items of two tiles; 1: one tile per CTA, split between its two
// pipelines; 2: one tile per cluster of two CTAs (CPAIR), CTA r scanning the
// chunks c = r mod 2 of each stage with its two pipelines (c / 2 = t mod 2
// on pipeline t); at the end of a stage each CTA's pipeline 0 sends its
// per-frame (value, index) minimum to the other CTA's shared memory and both
// keep the lexicographic minimum of the two, so both hold the same codes and
// build the same next query.
// SHARE (split items only): pipeline 1 fetches half of the next query's
// terms into a partial of its own in TMEM (deep stacks; see the row threads).
template <int MODE, bool SHARE = false>
__global__ void __launch_bounds__(SR_THREADS, 1)
    k_search_tc(const float *__restrict__ P0, const float *__restrict__ G, const float *__restrict__ cb_img,
                const float *__restrict__ cnorm, int32_t *__restrict__ codes, int64_t n_rows, int n_q, int q_begin,
                int q_end, int K, int n_tiles, int metric, int *__restrict__ status) {
  constexpr bool SPLIT = MODE >= 1, CPAIR = MODE == 2;
  // this CTA's item index and the number of such (a CTA pair counts once);
  // unsigned, like blockIdx.x itself (signed forms measured 2.5 % slower:
  // more registers spilled in the row threads)
#define CTA_ID (CPAIR ? (blockIdx.x >> 1) : blockIdx.x)
#define N_CTA (CPAIR ? (gridDim.x >> 1) : gridDim.x)
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  unsigned char *ring = smem;
  float *cn_buf = reinterpret_cast<float *>(smem + SR_RING_BYTES + 4 * SR_PART_BYTES);
  SrBars &bar = *reinterpret_cast<SrBars *>(smem + SR_RING_BYTES + 4 * SR_PART_BYTES + SR_CN_SLOTS * SR_CN_BYTES);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkc = K / SR_KC;
  // tiles of this CTA: b + 2Bk as tile 0 and b + B + 2Bk as tile 1
  // (b = blockIdx.x, B = gridDim.x); a launch with no more tiles than CTAs
  // thus puts one tile on each SM, split between the CTA's two pipelines
  const int sweep = 2 * N_CTA;
  // Every CTA walks the same codebook chunks; starting each at a different
  // chunk spreads the simultaneous bulk copies over nkc chunks of L2 instead
  // of one hot chunk.  The argmin merge below is order-independent.
  const int rot = CTA_ID % nkc;
  constexpr int d = kCodeDim;
  constexpr int SLOTS = CPAIR ? SR_SLOTS_CPAIR : SPLIT ? SR_SLOTS_SPLIT : SR_SLOTS;
  // CTA pairs: this CTA's rank in its cluster; its chunks are c = rank,
  // rank + 2, ... (in a split item pipeline t takes those with c / 2 = t mod 2)
  const uint32_t prank = CPAIR ? cluster_ctarank() : 0u;
  constexpr int C_STEP = CPAIR ? 2 : 1;
  // the split ring takes tile 1's areas: only for launches of one tile per CTA
  if ((SPLIT && (n_tiles > (int)N_CTA || nkc % (CPAIR ? 4 : 2) != 0)) ||
      (CPAIR && (cluster_nctarank() != 2u || (gridDim.x & 1u) != 0u))) {
    if (threadIdx.x == 0) record_error(status, RVQ_DEVICE_BAD_LAUNCH);
    return;  // uniform over the cluster: no CTA reaches a cluster barrier
  }
  // CTA pairs: the other CTA's minima, [2][128] (value bits, index)
  uint2 *px = reinterpret_cast<uint2 *>(smem + SR_RING_BYTES + SR_PART_BYTES);

  if (tid == 0) {
    for (int s = 0; s < SLOTS; ++s) {
      mbar_init(&bar.b_full[s], SR_COPY_PIECES);
      mbar_init(&bar.b_empty[s], 2);  // one commit per tile's MMA issuer
    }
    for (int s = 0; s < SR_CN_SLOTS; ++s) {
      mbar_init(&bar.cn_full[s], 1);
      mbar_init(&bar.cn_free[s], 256);  // every row thread of both tiles has scanned the chunk
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar.a_ready[t], 128);
      mbar_init(&bar.acc_full[t], 1);
      mbar_init(&bar.acc_empty[t], 128);
      mbar_init(&bar.drain[t], 1);
      mbar_init(&bar.turn[t], 1);
      mbar_init(&bar.xch_full[t], 128);
      mbar_init(&bar.xch_free[t], 128);
      mbar_init(&bar.px_full[t], 128);  // one remote arrive per frame
    }
    mbar_init(&bar.p1t_full, 128);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem, SR_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (CPAIR) cluster_sync_all();  // the other CTA's barriers are initialised before any remote arrive
  const uint32_t tmem = bar.tmem;

  if (warp == 0 || warp == 11) {
    // ---------------- producers: warp 0 lanes 0-1 the lo halves, lane 2 the norms; warp 11 lanes 0-1 the hi halves ----------------
    // A thread's bulk copies are carried out one after another (about a third
    // of a microsecond each, whatever their size), so each kind of copy gets
    // threads of its own, each half-chunk copied in SR_COPY_PIECES pieces by
    // as many threads: with one tile per CTA the tensor core needs a chunk
    // every 0.8 us, about the time of two copies in a row (two pieces: mid-size
    // encodes 1-2 % faster than whole halves, four: no better).
    const int role = warp == 11 ? (lane < SR_COPY_PIECES ? 0 : -1)
                                : (lane < SR_COPY_PIECES ? 1 : lane == SR_COPY_PIECES ? 2 : -1);  // hi, lo, norms
    const int piece = lane;                                                // of a half-chunk
    const int h = role == 0 ? 0 : 1;  // the half of a chunk image (hi, lo)
    if (role >= 0) {
      uint32_t ch = 0;  // chunks gone through
      bool ok = true;
      for (int t0 = CTA_ID; t0 < n_tiles && ok; t0 += sweep)
        for (int q = q_begin; q < q_end && ok; ++q)
          for (int c = (int)prank; c < nkc && ok; c += C_STEP, ++ch) {
            const int cr = (c + rot) % nkc;
            if (role == 2) {
              // the chunk's squared norms; the slot last held chunk ch - 3
              const int sn = ch % SR_CN_SLOTS;
              if (ch >= SR_CN_SLOTS && !mbar_wait(&bar.cn_free[sn], (ch / SR_CN_SLOTS - 1) & 1)) {
                record_error(status, RVQ_DEVICE_TIMEOUT);
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&bar.cn_full[sn], SR_CN_BYTES);
              bulk_g2s(cn_buf + sn * SR_KC, cnorm + (size_t)q * K + cr * SR_KC, SR_CN_BYTES, &bar.cn_full[sn]);
              continue;
            }
            const uint32_t j = 2 * ch + (1 - h);
            const int s = j % SLOTS;
            const uint32_t use = j / SLOTS;
            if (use > 0 && !mbar_wait(&bar.b_empty[s], (use - 1) & 1)) {
              record_error(status, RVQ_DEVICE_TIMEOUT);
              ok = false;
              break;
            }
            constexpr uint32_t PB = SR_HALF / SR_COPY_PIECES;
            mbar_arrive_expect_tx(&bar.b_full[s], PB);
            bulk_g2s(ring + s * SR_HALF + piece * PB,
                     cb_img + (((size_t)q * nkc + cr) * 2 + h) * (SR_HALF / 4) + piece * (PB / 4), PB, &bar.b_full[s]);
          }
      // Every copy is waited for by the threads that use it before the final
      // barrier; after an error, the last copy of this thread (whose slot no
      // later copy can have reused) still lands before the CTA may exit.
      if (ch > 0) {
        if (role == 2) {
          mbar_wait(&bar.cn_full[(ch - 1) % SR_CN_SLOTS], ((ch - 1) / SR_CN_SLOTS) & 1);
        } else {
          const uint32_t jj = 2 * (ch - 1) + (1 - h);
          mbar_wait(&bar.b_full[jj % SLOTS], (jj / SLOTS) & 1);
        }
      }
    }
  } else if (warp == 1 || warp == 10) {
    // ---------------- MMA issuers: warp 1 for tile 0, warp 10 for tile 1 ----------------
    // An issuing thread that waits on an mbarrier stalls until its queued MMAs
    // have drained, which would leave the tensor core idle; with one issuer per
    // tile, each does its waits while the other tile's MMAs are queued.  The
    // two take turns chunk by chunk (tile 0, tile 1, tile 0, ...; in a split
    // item, the even and the odd chunks): an issuer hands over the turn after
    // 18 of its 24 MMAs, so the next chunk's MMAs queue up behind the last
    // ones without a gap, and the pipeline that has just finished scans its
    // distances while the tensor core works on the other.  The 24 MMAs of a
    // chunk are issued straight-line (compile-time operand offsets and
    // accumulate flags) so that one thread keeps pace with the tensor core.
    // Each user of a half-chunk commits once to its empty barrier (count 2); a
    // sole user (a tile alone, or a split chunk) commits twice.  A tile 0
    // alone takes no turns.
    const int t = warp == 1 ? 0 : 1;
    if (lane == 0) {
      uint32_t ch = 0, u = 0, builds = 0;  // chunks gone through, chunks issued, queries
      bool ok = true;
      auto wait_or_fail = [&](uint64_t *b, uint32_t parity) {
        if (ok && !mbar_wait(b, parity)) {
          record_error(status, RVQ_DEVICE_TIMEOUT);
          ok = false;
        }
        return ok;
      };
      auto wait_hot_or_fail = [&](uint64_t *b, uint32_t parity) {
        if (ok && !mbar_wait_hot(b, parity)) {
          record_error(status, RVQ_DEVICE_TIMEOUT);
          ok = false;
        }
        return ok;
      };
      // descriptor of the ring base; an operand adds (byte offset >> 4)
      const uint64_t desc0 = smem_desc(smem_addr(ring), 16, 1024, kSwizzle128B);
      const uint32_t tb = tmem + t * SR_TILE_COLS;
      const uint32_t ta = SPLIT ? tmem : tb;  // the query's columns
      for (int t0 = CTA_ID; t0 < n_tiles && ok; t0 += sweep) {
        const bool pair = !SPLIT && t0 + (int)N_CTA < n_tiles;  // tile 1 present in this item
        if (t == 1 && !pair && !SPLIT) break;
        const bool turns = SPLIT || pair;
        const bool twice = !pair;  // sole user of each half-chunk
        for (int q = q_begin; q < q_end && ok; ++q, ++builds)
          for (int c = (int)prank; c < nkc && ok; c += C_STEP, ++ch) {
            if (SPLIT && ((CPAIR ? c >> 1 : c) & 1) != t) continue;
            const uint32_t j0 = 2 * ch, j1 = j0 + 1;  // the chunk's lo and hi half-chunks
            const int s0 = j0 % SLOTS, s1 = j1 % SLOTS;
            // the accumulator free, the query built, the lo half in, the turn: issuer
            // 1's n-th chunk follows issuer 0's n-th, issuer 0's follows issuer 1's (n-1)-th
            if (u > 0 && !wait_or_fail(&bar.acc_empty[t], (u - 1) & 1)) break;
            if (c == (CPAIR ? (int)prank + 2 * t : SPLIT ? t : 0) && !wait_or_fail(&bar.a_ready[SPLIT ? 0 : t], builds & 1)) break;
            if (!wait_or_fail(&bar.b_full[s0], (j0 / SLOTS) & 1)) break;
            // (the turn is polled: its wait is the one the tensor core idles on)
            if (turns && (t == 1 || u > 0) && !wait_hot_or_fail(&bar.turn[t], (t == 1 ? u : u - 1) & 1)) break;
            ++u;
            tc_fence_after();
            // lo half first (a_hi.b_lo, 8 MMAs), then hi (a_hi.b_hi + a_lo.b_hi, 16): the
            // lo half's slot is freed early, and the next chunk's hi half, copied
            // into it, is needed only a third of the way into that chunk
            const uint64_t bd_lo = desc0 + (uint64_t)((s0 * SR_HALF) >> 4);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const uint64_t b = bd_lo + (uint64_t)((((m >> 2) * SR_ATOM) + (m & 3) * 32) >> 4);
              mma_tf32_ta(tb + SR_ACC, ta + SR_A_HI + (uint32_t)m * 8, b, SR_IDESC, m == 0 ? 0u : 1u);
            }
            mma_commit(&bar.b_empty[s0]);  // the lo half is free once these MMAs are done
            if (twice) mma_commit(&bar.b_empty[s0]);
            if (!wait_or_fail(&bar.b_full[s1], (j1 / SLOTS) & 1)) break;
            tc_fence_after();
            const uint64_t bd_hi = desc0 + (uint64_t)((s1 * SR_HALF) >> 4);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              if (m == 5) mbar_arrive(&bar.turn[1 - t]);  // 18 of 24 issued: hand over
              const uint64_t b = bd_hi + (uint64_t)((((m >> 2) * SR_ATOM) + (m & 3) * 32) >> 4);
              mma_tf32_ta(tb + SR_ACC, ta + SR_A_HI + (uint32_t)m * 8, b, SR_IDESC, 1u);
              mma_tf32_ta(tb + SR_ACC, ta + SR_A_LO + (uint32_t)m * 8, b, SR_IDESC, 1u);
            }
            mma_commit(&bar.acc_full[t]);
            mma_commit(&bar.b_empty[s1]);
            if (twice) mma_commit(&bar.b_empty[s1]);
          }
      }
      mma_commit(&bar.drain[t]);
      mbar_wait(&bar.drain[t], 0);
    }
  } else {
    // ---------------- one thread per frame row (warps 2-9) ----------------
    const int tile = (warp - 2) >> 2;  // 0 or 1
    const int quarter = warp & 3;      // TMEM lane quarter of this warp
    const uint32_t lane_base = tmem + tile * SR_TILE_COLS + ((uint32_t)(quarter * 32) << 16);
    const int64_t ld = (int64_t)n_q * d;
    unsigned char *tile_area = smem + SR_RING_BYTES + (1 - tile) * 2 * SR_PART_BYTES;
    float4 *wpart = reinterpret_cast<float4 *>(tile_area) + quarter * 32 * (d / 4);
    float4 *wstage = reinterpret_cast<float4 *>(tile_area + SR_PART_BYTES) + quarter * 32 * (d / 4);
    const int f0 = lane >> 2, j = lane & 3;       // cooperative layout: frames f0 + 8i, slots 4b + j
    uint64_t *acc_full = &bar.acc_full[tile], *acc_empty = &bar.acc_empty[tile], *a_ready = &bar.a_ready[tile];
    uint32_t cc = 0;
    bool ok = true;
    int my_codes[kMaxStages];

    // Term rows: one 64-float row per frame of this warp (`mine` is this
    // thread's frame's row), copied asynchronously in the cooperative layout;
    // each lane later reads back only the pieces it copied itself.  A first
    // term lands straight in the partial sum, any other in the staging area.
    bool pending = false, pending_first = false;
    auto term_issue = [&](const float *mine, bool first) {
      const unsigned long long m = reinterpret_cast<unsigned long long>(mine);
      float4 *dst = first ? wpart : wstage;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 *src = reinterpret_cast<const float4 *>(__shfl_sync(0xffffffffu, m, f0 + 8 * i));
#pragma unroll
        for (int b = 0; b < 4; ++b) cp_async16(dst + (f0 + 8 * i) * (d / 4) + ((4 * b + j) ^ f0), src + 4 * b + j);
      }
      cp_async_commit();
      pending = true;
      pending_first = first;
    };
    // wait for this thread's copies; partial -= staged rows
    auto term_finish = [&]() {
      cp_async_wait_all();
      if (!pending_first) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int idx = (f0 + 8 * i) * (d / 4) + ((4 * b + j) ^ f0);
            float4 t = wpart[idx];
            const float4 v = wstage[idx];
            t.x -= v.x;
            t.y -= v.y;
            t.z -= v.z;
            t.w -= v.w;
            wpart[idx] = t;
          }
      }
      pending = false;
    };

    const int n_cta = N_CTA;
    // split items: pipeline 1's (value, index) per frame, two column pairs of
    // its query columns (unused in a split item), in this frame's TMEM lane
    const uint32_t xch = tmem + SR_TILE_COLS + ((uint32_t)(quarter * 32) << 16) + SR_A_HI;
    uint32_t ua = 0, xu = 0, nb = 0;  // accumulator uses, stage minima handed over, queries seen
    uint32_t p1u = 0;                  // split items: pipeline 1 partials taken
    // split items: pipeline 1's partial of the next query's terms, TMEM
    // columns [SR_A_LO, SR_A_LO + 64) of tile 1 (its query columns, unused when split)
    const uint32_t p1part = tmem + SR_TILE_COLS + SR_A_LO + ((uint32_t)(quarter * 32) << 16);
    float s_row = 1.0f;               // this frame's distance scale (1 / n(p) for the cosine metric)
    // the first query's partial: the projection row itself (tile 1 only if the first item has one)
    if (tile == 0 || (!SPLIT && CTA_ID + n_cta < n_tiles)) {
      const int64_t n = (int64_t)(CTA_ID + tile * n_cta) * 128 + quarter * 32 + lane;
      term_issue(P0 + (n < n_rows ? n : 0) * ld + q_begin * d, true);
    }
    uint32_t xs = 0;  // CTA pairs: stage minima exchanged
    for (int t0 = CTA_ID; t0 < n_tiles && ok; t0 += sweep) {
      const bool pair = !SPLIT && t0 + n_cta < n_tiles;
      constexpr bool split = SPLIT;
      if (tile == 1 && !pair && !split) break;
      const bool scan_only = tile == 1 && split;  // half the chunks; no query, no codes
      const int my_tile = tile == 1 && pair ? t0 + n_cta : t0;
      const int64_t n = (int64_t)my_tile * 128 + quarter * 32 + lane;
      const bool valid = n < n_rows;
      const int64_t n_next = n + (int64_t)sweep * 128;
      const bool has_next = my_tile + sweep < n_tiles;
      // a tile 0 without a partner tile or split releases the norm blocks for both
      const bool alone = !pair && !split;
      const int n_own = CPAIR ? nkc / 4 : split ? nkc / 2 : nkc;  // chunks scanned per stage
      constexpr bool share_terms = SPLIT && SHARE;
      for (int q = q_begin; q < q_end && ok; ++q) {
        if (!scan_only) {
          // ---- stage boundary: the query = partial - the last known term (if
          //      still staged) - the row of the code just found (none at the
          //      block's first stage).  The partial minus the staged term is read
          //      into registers; the staging area then takes the rows of the codes
          //      just found, copied cooperatively like every term (a row per
          //      thread would take one L1 wavefront per lane and load), and the
          //      query is formed in registers: the boundary writes no shared
          //      memory.
          const bool sub_staged = pending && !pending_first;
          if (pending) {
            cp_async_wait_all();
            pending = false;
          }
          __syncwarp();  // the warp's copies (this frame's staged row among them) have landed
          float4 pq[d / 4];
#pragma unroll
          for (int u = 0; u < d / 4; ++u) {
            const int idx = lane * (d / 4) + (u ^ (lane & 7));
            pq[u] = wpart[idx];
            if (sub_staged) {
              const float4 v = wstage[idx];
              pq[u].x -= v.x;
              pq[u].y -= v.y;
              pq[u].z -= v.z;
              pq[u].w -= v.w;
            }
          }
          if (q > q_begin) {
            __syncwarp();  // every lane has read its staged row before the code rows overwrite it
            term_issue(G + ((size_t)pair_index(q, q - 1) * K + my_codes[q - 1]) * d, false);
            cp_async_wait_all();
            pending = false;
            __syncwarp();
#pragma unroll
            for (int u = 0; u < d / 4; ++u) {
              const float4 v = wstage[lane * (d / 4) + (u ^ (lane & 7))];
              pq[u].x -= v.x;
              pq[u].y -= v.y;
              pq[u].z -= v.z;
              pq[u].w -= v.w;
            }
          }
          // split items: pipeline 1's partial of this query's terms (q - (q + 1) / 2
          // of the q fetched during the last stage), in this frame's TMEM lane
          const int q_rel = q - q_begin;
          const bool sub_p1 = share_terms && q_rel > 0 && q_rel - (q_rel + 1) / 2 > 0;
          if (sub_p1) {
            if (!__all_sync(0xffffffffu, mbar_wait(&bar.p1t_full, p1u & 1))) {
              record_error(status, RVQ_DEVICE_TIMEOUT);
              ok = false;
              break;
            }
            ++p1u;
            tc_fence_after();
          }
          // raw (= hi after TF32 truncation) and lo parts into this row's TMEM lane
          float ss = 0.0f;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float p[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 t = pq[8 * h + u];
              p[4 * u] = t.x;
              p[4 * u + 1] = t.y;
              p[4 * u + 2] = t.z;
              p[4 * u + 3] = t.w;
            }
            if (sub_p1) {
              float p1v[32];
              tmem_ld32(p1part + 32 * h, p1v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) p[i] -= p1v[i];
            }
            tmem_st32(lane_base + SR_A_HI + 32 * h, p);
#pragma unroll
            for (int i = 0; i < 32; ++i) ss = fmaf(p[i], p[i], ss);
#pragma unroll
            for (int i = 0; i < 32; ++i) p[i] -= __uint_as_float(__float_as_uint(p[i]) & 0xffffe000u);
            tmem_st32(lane_base + SR_A_LO + 32 * h, p);
          }
          // cosine metric: the query stays raw in TMEM and its distances are
          // scaled by 1 / max(||p||, 1e-12) in the scan
          s_row = metric == RVQ_METRIC_COSINE ? 1.0f / fmaxf(sqrtf(ss), 1e-12f) : 1.0f;
          // for pipeline 1: the distance scale, and the code just found (its terms need it)
          if (split) tmem_st2(xch + 4, __float_as_uint(s_row), share_terms && q > q_begin ? (uint32_t)my_codes[q - 1] : 0u);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(a_ready);
          __syncwarp();  // every lane has read its row before the next query's terms overwrite it
        } else {
          // pipeline 1 of a split item: this stage's query is built; its distance scale
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.a_ready[0], nb & 1))) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          ++nb;
          tc_fence_after();
          uint32_t sv, code_prev;
          tmem_ld2(xch + 4, sv, code_prev);
          tmem_wait_ld();
          s_row = __uint_as_float(sv);
          if (share_terms && q > q_begin) my_codes[q - 1] = (int)code_prev;
        }
        // ---- terms of the next query known before this stage's code:
        //      next stage: P0[n][q+1], G[q+1][q_begin..q-1];  next tile: P0[n'][q_begin]
        const int q_next = q + 1 < q_end ? q + 1 : q_begin;
        const int n_terms_all = q + 1 < q_end ? q + 1 - q_begin : (has_next ? 1 : 0);
        // split items of deep stacks: pipeline 0 fetches the first half of the
        // terms (P0 first) into its partial in shared memory, pipeline 1 the
        // rest into a partial of its own in TMEM, subtracted at the stage
        // boundary, so each has half the fetch round trips
        const int n_half = share_terms ? (n_terms_all + 1) / 2 : n_terms_all;
        const int n_terms = scan_only ? 0 : n_half;
        const int n_p1 = share_terms && q + 1 < q_end ? n_terms_all - n_half : 0;
        const int64_t n_row = q + 1 < q_end ? (valid ? n : 0) : (n_next < n_rows ? n_next : 0);
        auto term_row = [&](int t) -> const float * {
          return t == 0 ? P0 + n_row * ld + q_next * d
                        : G + ((size_t)pair_index(q_next, q_begin + t - 1) * K + my_codes[q_begin + t - 1]) * d;
        };
        int done = 0, done1 = 0;
        // ---- scan the K distances ||c||^2 - 2 p.c; keep the lexicographic (value, index) minimum
        float best_v = __int_as_float(0x7f800000);
        int best_k = 0;
        for (int c = (int)prank; c < nkc; c += C_STEP, ++cc) {
          const int sn = cc % SR_CN_SLOTS;
          if (split && ((CPAIR ? c >> 1 : c) & 1) != tile) {
            // the other pipeline's chunk: its norm block is released by both, in order
            if (!__all_sync(0xffffffffu, mbar_wait(&bar.cn_full[sn], (cc / SR_CN_SLOTS) & 1))) {
              record_error(status, RVQ_DEVICE_TIMEOUT);
              ok = false;
              break;
            }
            mbar_arrive(&bar.cn_free[sn]);
            continue;
          }
          const int cr = (c + rot) % nkc;
          if (!__all_sync(0xffffffffu, mbar_wait(acc_full, (SPLIT ? ua : cc) & 1))) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          if (SPLIT) ++ua;
          tc_fence_after();
          float v[SR_KC];
#pragma unroll
          for (int g = 0; g < SR_KC / 32; ++g)
            tmem_ld32(lane_base + SR_ACC + g * 32, *reinterpret_cast<float(*)[32]>(&v[32 * g]));
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(acc_empty);  // the accumulator is free: the values are in registers
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.cn_full[sn], (cc / SR_CN_SLOTS) & 1))) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          // distance (up to this frame's constant): s * (-2 p.c) + ||c||^2, with
          // s = 1 for the plain metric (exact) and 1 / n(p) for the cosine one
          const float4 *cn4 = reinterpret_cast<const float4 *>(cn_buf + sn * SR_KC);
#pragma unroll
          for (int u = 0; u < SR_KC / 4; ++u) {
            const float4 cn = cn4[u];
            fma2(v[4 * u], v[4 * u + 1], s_row, cn.x, cn.y);
            fma2(v[4 * u + 2], v[4 * u + 3], s_row, cn.z, cn.w);
          }
          const float m = min128(v);
          mbar_arrive(&bar.cn_free[sn]);  // the norms are in registers
          if (alone) mbar_arrive(&bar.cn_free[sn]);
          if (m <= best_v) {  // rare after the first chunks: locate the first index holding m
            const int k = cr * SR_KC + first_index_of(v, m);
            if (m < best_v || k < best_k) {
              best_v = m;
              best_k = k;
            }
          }
          // ---- this chunk's share of the next query's known terms, in order:
          //      the previous one is added now, the new one stays in flight
          //      until after the next chunk's scan
          const int target = (n_terms * ((CPAIR ? c >> 2 : split ? c >> 1 : c) + 1) + n_own - 1) / n_own;
          for (; done < target; ++done) {
            if (pending) term_finish();
            term_issue(term_row(done), done == 0);
          }
          if (scan_only && n_p1 > 0) {
            // pipeline 1: its terms (G rows n_half ..), this frame's row straight
            // into registers, summed into its TMEM partial
            const int target1 = (n_p1 * ((CPAIR ? c >> 2 : c >> 1) + 1) + n_own - 1) / n_own;
            for (; done1 < target1; ++done1) {
              const float4 *row = reinterpret_cast<const float4 *>(term_row(n_half + done1));
              float4 r[d / 4];
#pragma unroll
              for (int u = 0; u < d / 4; ++u) r[u] = __ldg(row + u);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float a[32];
                if (done1 > 0) {
                  tmem_wait_st();  // this thread's previous sum is written before it is read back
                  tmem_ld32(p1part + 32 * h, a);
                  tmem_wait_ld();
                } else {
#pragma unroll
                  for (int i = 0; i < 32; ++i) a[i] = 0.0f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  a[4 * u] += r[8 * h + u].x;
                  a[4 * u + 1] += r[8 * h + u].y;
                  a[4 * u + 2] += r[8 * h + u].z;
                  a[4 * u + 3] += r[8 * h + u].w;
                }
                tmem_st32(p1part + 32 * h, a);
              }
            }
          }
        }
        if (!ok) break;
        if (scan_only && n_p1 > 0) {  // pipeline 1's share of the next query is in TMEM
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar.p1t_full);
        }
        if (split) {
          // ---- pipeline 1's minimum of the stage to pipeline 0
          const uint32_t xb = xch + (xu & 1) * 2;
          const uint32_t use = xu >> 1;
          if (scan_only) {
            if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(&bar.xch_free[xu & 1], (use - 1) & 1))) {
              record_error(status, RVQ_DEVICE_TIMEOUT);
              ok = false;
              break;
            }
            tmem_st2(xb, __float_as_uint(best_v), (uint32_t)best_k);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bar.xch_full[xu & 1]);
            ++xu;
            continue;
          }
          if (!__all_sync(0xffffffffu, mbar_wait(&bar.xch_full[xu & 1], use & 1))) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t o_v, o_k;
          tmem_ld2(xb, o_v, o_k);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bar.xch_free[xu & 1]);
          ++xu;
          const float ov = __uint_as_float(o_v);
          if (ov < best_v || (ov == best_v && (int)o_k < best_k)) {
            best_v = ov;
            best_k = (int)o_k;
          }
        }
        if (CPAIR) {
          // ---- the pair's exchange: this CTA's minimum into the other CTA's
          //      shared memory (a store, then a release arrive on its barrier),
          //      then the lexicographic minimum of the two -- the same in both
          const uint32_t b = xs & 1, other = prank ^ 1u;
          const int f = quarter * 32 + lane;
          st_cluster_v2u32(cluster_map(smem_addr(px + b * 128 + f), other), __float_as_uint(best_v), (uint32_t)best_k);
          mbar_arrive_cluster(cluster_map(smem_addr(&bar.px_full[b]), other));
          if (!__all_sync(0xffffffffu, mbar_wait_cluster(&bar.px_full[b], (xs >> 1) & 1))) {
            record_error(status, RVQ_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          ++xs;
          // (buffer b is written again two exchanges later, after the other
          // CTA has had this CTA's next minimum, sent after this read)
          const uint2 o = px[b * 128 + f];
          const float ov = __uint_as_float(o.x);
          if (ov < best_v || (ov == best_v && (int)o.y < best_k)) {
            best_v = ov;
            best_k = (int)o.y;
          }
        }
        my_codes[q] = best_k;
        if (valid && prank == 0) codes[n * n_q + q] = best_k;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CPAIR) cluster_sync_all();  // no CTA leaves while the other may still write into it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, SR_TMEM_COLS);
  }
#undef CTA_ID
#undef N_CTA
}

// ===========================================================================
// Stage blocks of deep stacks.  The query of stage t is
//   p_t = P0[n][t] - sum_{s<t} G[t][s][code_s],
// t terms of which a search launch over all stages would gather t - 1 (one
// 256-byte row each) between the distance chunks of stage t - 1: 496 rows a
// frame at 32 stages, with one or two in flight per row thread.  A deep stack
// therefore runs as a few search launches over blocks of stages [q_begin,
// q_end), each gathering only the terms of its own block (s >= q_begin); the
// terms of the earlier stages are all known once the previous blocks are
// done, and this kernel subtracts them from P0[n][q_begin..q_end) first, with
// many rows in flight on every SM.  The order is the search kernel's own:
// s = 0, 1, ..., q_begin - 1 here, then q_begin, ... in the search.
// d/4 lanes per (frame, stage t), one float4 column each (d = 64 or 8); a
// code outside [0, K) (an earlier launch that gave up) reads row 0.
// ===========================================================================
constexpr int CT_THREADS = 256;
constexpr int CT_UNROLL = 8;

template <int d>
__global__ void __launch_bounds__(CT_THREADS)
    k_cross_terms(float *__restrict__ P0, const float *__restrict__ G, const int32_t *__restrict__ codes,
                  int64_t n_rows, int n_q, int q_begin, int q_end, int K) {
  constexpr int LPI = d / 4;  // lanes per item
  const int nt = q_end - q_begin;
  const int64_t item = ((int64_t)blockIdx.x * CT_THREADS + threadIdx.x) / LPI;
  if (item >= n_rows * nt) return;
  const int l = threadIdx.x % LPI;
  const int64_t n = item / nt;
  const int t = q_begin + (int)(item - n * nt);
  const int32_t *cr = codes + n * n_q;
  float4 *dst = reinterpret_cast<float4 *>(P0 + (n * n_q + t) * d) + l;
  const float4 *g = reinterpret_cast<const float4 *>(G + (size_t)pair_index(t, 0) * K * d) + l;
  float4 acc = *dst;
  for (int s0 = 0; s0 < q_begin; s0 += CT_UNROLL) {
    int c[CT_UNROLL];
#pragma unroll
    for (int u = 0; u < CT_UNROLL; ++u) {
      const int v = s0 + u < q_begin ? __ldg(cr + s0 + u) : 0;
      c[u] = (unsigned)v < (unsigned)K ? v : 0;
    }
    float4 r[CT_UNROLL];
#pragma unroll
    for (int u = 0; u < CT_UNROLL; ++u)
      if (s0 + u < q_begin) r[u] = __ldg(g + ((size_t)(s0 + u) * K + c[u]) * (d / 4));
#pragma unroll
    for (int u = 0; u < CT_UNROLL; ++u)
      if (s0 + u < q_begin) {
        acc.x -= r[u].x;
        acc.y -= r[u].y;
        acc.z -= r[u].z;
        acc.w -= r[u].w;
      }
  }
  *dst = acc;
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
  e = cudaFuncSetAttribute(k_project_tc<2, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pj_smem<2, 256>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_project_tc<1, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pj_smem<1, 128>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_project_tc<1, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pj_smem<1, 64>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_search_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SR_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_search_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SR_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_search_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SR_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_search_tc<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SR_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_search_tc<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SR_SMEM);
  if (e != cudaSuccess) return e;
  g_attr_done.fetch_or(bit);
  return cudaSuccess;
}

// Clusters of CS (here 2) search CTAs the device holds at once (0 if the
// query fails).
template <int CS>
int max_search_clusters() {
  static std::atomic<int> cached{-1};
  int v = cached.load();
  if (v >= 0) return v;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)CS, 1, 1);
  cfg.blockDim = dim3(SR_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SR_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  v = 0;
  if (cudaOccupancyMaxActiveClusters(&v, k_search_tc<CS>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();  // the query's error is not the caller's
    v = 0;
  }
  cached.store(v);
  return v;
}

// Whether a split item's pipeline 1 should fetch half of the next query's
// terms: once pipeline 0 alone would fetch more than one a chunk on average
// (n_q^2 / 2 terms over n_q stages of its own chunks), i.e. deep stacks.
// Measured: 32 stages 15 % faster; 8 and 10 stages 5 % slower.
bool share_terms(int n_q, int own_chunks) { return n_q > 2 * own_chunks; }

// Stage blocks of a call (k_cross_terms): a stack deeper than kStageBlock
// whose row threads would fetch more than two terms a chunk at its last
// stage runs in the fewest blocks of at most kStageBlock stages (sizes as
// equal as they go).
constexpr int kStageBlock = 6;
int stage_blocks(int n_q, int own_chunks) {
  return n_q > kStageBlock && n_q > 2 * own_chunks ? (n_q + kStageBlock - 1) / kStageBlock : 1;
}

// One tile per cluster of CS CTAs, stages [q0, q1).
template <int CS>
cudaError_t launch_search_clusters(const float *p0, const float *G, const float *cb_img, const float *cn,
                                   int32_t *codes, int64_t n, int n_q, int q0, int q1, int K, int tiles, int metric,
                                   int *status, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(CS * tiles), 1, 1);
  cfg.blockDim = dim3(SR_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SR_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kern = share_terms(q1 - q0, K / SR_KC / 4) ? k_search_tc<CS, true> : k_search_tc<CS, false>;
  return cudaLaunchKernelEx(&cfg, kern, p0, G, cb_img, cn, codes, n, n_q, q0, q1, K, tiles, metric, status);
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

// The item shape of the projection: 256 frames x 256 columns, or a smaller
// item (128 x 128 or 128 x 64) that spreads a call with few frames over more
// SMs, whichever needs the fewest MMA cycles on the busiest SM (waves x the
// cycles of an item's K-slice: 12 MMAs of 128 x 256 x 8 at 128 cycles, 6 of
// 128 x 128 x 8 at 64, 6 of 128 x 64 x 8 at 48), small items in at most two
// waves: more re-read x and w_in from L2 more often than they save (three
// waves measured 470 against 443 us for 9728 frames of ten 4096-entry
// stages).  (Items of 256 x 128, two accumulators in TMEM, measured slower
// wherever this count favoured them: moss_deep encode 704 against 686 us;
// forced onto large_batch, 1.70 against 1.46 ms.)
int projection_shape(int64_t n, int n_cols, int sms) {
  const int64_t t128 = (n + 127) / 128;
  const int64_t items[3] = {((n + 255) / 256) * ((n_cols + 255) / 256), t128 * ((n_cols + 127) / 128),
                            t128 * ((n_cols + 63) / 64)};
  const int64_t slice_cycles[3] = {12 * 128, 6 * 64, 6 * 48};
  int best = 0;
  int64_t best_cost = ((items[0] + sms - 1) / sms) * slice_cycles[0];
  for (int i = 1; i < 3; ++i) {
    const int64_t waves = (items[i] + sms - 1) / sms;
    if (waves <= 2 && waves * slice_cycles[i] < best_cost) {
      best = i;
      best_cost = waves * slice_cycles[i];
    }
  }
  return best;
}

}  // namespace

cudaError_t launch_project_tc(const rvq_dims &dm, const void *tables, const float *x, int64_t n, int n_q, float *p0,
                              int *status, bool zero_status, cudaStream_t st, int shape) {
  const TablesLayout L = tables_layout(dm);
  const int D = dim_in(dm), d = dm.d, Q = dm.Q;  // frames are D_in wide (fc folded into w_in)
  const int n_cols = n_q * d;
  cudaError_t e = ensure_attributes();
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (shape < 0) shape = projection_shape(n, n_cols, sms);
  const uint32_t nc = shape == 0 ? 256 : shape == 1 ? 128 : 64, rows = shape == 0 ? 256 : 128;
  CUtensorMap tm_x, tm_whi, tm_wlo;
  if ((e = tensor_map_2d(&tm_x, x, (uint64_t)D, (uint64_t)n, PJ_BK, 128, CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&tm_whi, at<float>(tables, L.w_in_hi), (uint64_t)D, (uint64_t)Q * d, PJ_BK, nc,
                         CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess)
    return e;
  if ((e = tensor_map_2d(&tm_wlo, at<float>(tables, L.w_in_lo), (uint64_t)D, (uint64_t)Q * d, PJ_BK, nc,
                         CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess)
    return e;
  const int n_cb = (int)((n_cols + nc - 1) / nc);
  const int items = (int)((n + rows - 1) / rows) * n_cb;
  const int grid = items < sms ? items : sms;
  const float *b_in = at<float>(tables, L.b_in);
  const int zs = zero_status ? 1 : 0;
  if (shape == 0)
    k_project_tc<2, 256><<<grid, PjShape<2, 256>::THREADS, pj_smem<2, 256>(), st>>>(tm_x, tm_whi, tm_wlo, b_in, p0, n, n_cols, D,
                                                                      items, n_cb, status, zs);
  else if (shape == 1)
    k_project_tc<1, 128><<<grid, PjShape<1, 128>::THREADS, pj_smem<1, 128>(), st>>>(tm_x, tm_whi, tm_wlo, b_in, p0, n, n_cols, D,
                                                                      items, n_cb, status, zs);
  else
    k_project_tc<1, 64><<<grid, PjShape<1, 64>::THREADS, pj_smem<1, 64>(), st>>>(tm_x, tm_whi, tm_wlo, b_in, p0, n, n_cols, D,
                                                                    items, n_cb, status, zs);
  return cudaGetLastError();
}

cudaError_t launch_encode_chunk(const rvq_dims &dm, const void *tables, const float *x, int64_t n0, int64_t n,
                                int n_q, int32_t *codes, float *p0, int *status, cudaStream_t st) {
  if (stream_supported(dm, n_q, n))  // a small batch: the low-latency cluster kernels
    return launch_encode_stream(dm, tables, x + n0 * dim_in(dm), n, n_q, codes + n0 * n_q, p0, status, false, st);
  const TablesLayout L = tables_layout(dm);
  const int d = dm.d, K = dm.K;
  cudaError_t e = launch_project_tc(dm, tables, x + n0 * dim_in(dm), n, n_q, p0, status, false, st, -1);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  const float *G = at<float>(tables, L.g), *cb_img = at<float>(tables, L.cb_img), *cn = at<float>(tables, L.cnorm);
  int32_t *codes_c = codes + n0 * n_q;
  // the terms of stages [0, q0) subtracted from P0[.][q0, q1)
  auto cross_terms = [&](int q0, int q1) {
    const int64_t threads = n * (q1 - q0) * (d / 4);
    const unsigned blocks = (unsigned)((threads + CT_THREADS - 1) / CT_THREADS);
    if (d == kCodeDimSmall)
      k_cross_terms<kCodeDimSmall><<<blocks, CT_THREADS, 0, st>>>(p0, G, codes_c, n, n_q, q0, q1, K);
    else
      k_cross_terms<kCodeDim><<<blocks, CT_THREADS, 0, st>>>(p0, G, codes_c, n, n_q, q0, q1, K);
    return cudaGetLastError();
  };
  if (d == kCodeDimSmall) {
    const int bs = search8_block_stages(search8_split(n, sms));
    const int nb = (n_q + bs - 1) / bs;
    for (int b = 0; b < nb; ++b) {
      const int q0 = (int)((int64_t)n_q * b / nb), q1 = (int)((int64_t)n_q * (b + 1) / nb);
      if (q0 > 0 && (e = cross_terms(q0, q1)) != cudaSuccess) return e;
      if ((e = launch_search8(dm, tables, p0, n, n_q, q0, q1, codes_c, status, sms, st)) != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  const int tiles = (int)((n + 127) / 128);
  const int nkc = K / SR_KC;
  // one wave of CTA pairs: each tile's chunks split over two SMs; else, with
  // no more tiles than SMs, every item is split and the ring takes tile 1's areas
  const bool pairs = nkc % 4 == 0 && tiles <= max_search_clusters<2>();
  const bool split = !pairs && tiles <= sms && nkc % 2 == 0;
  const int own = pairs ? nkc / 4 : split ? nkc / 2 : nkc;  // chunks a pipeline scans per stage
  const int nb = stage_blocks(n_q, own);
  for (int b = 0; b < nb; ++b) {
    const int q0 = (int)((int64_t)n_q * b / nb), q1 = (int)((int64_t)n_q * (b + 1) / nb);
    if (q0 > 0 && (e = cross_terms(q0, q1)) != cudaSuccess) return e;
    if (pairs) {
      e = launch_search_clusters<2>(p0, G, cb_img, cn, codes_c, n, n_q, q0, q1, K, tiles, dm.metric, status, st);
    } else {
      auto search = split ? (share_terms(q1 - q0, nkc / 2) ? k_search_tc<1, true> : k_search_tc<1, false>)
                          : k_search_tc<0>;
      search<<<tiles < sms ? tiles : sms, SR_THREADS, SR_SMEM, st>>>(p0, G, cb_img, cn, codes_c, n, n_q, q0, q1, K,
                                                                     tiles, dm.metric, status);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace rvq
