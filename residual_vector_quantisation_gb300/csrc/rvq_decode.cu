// RVQ decode: y[n] = b_dec + sum_{q < n_q} Z[q][codes[n][q]]
//
// The decode graph of omnivoice.cpp ARCHITECTURE.md ("RVQ codec": per stage
// gather the codeword, project_out, add the bias, accumulate) with the
// projection and bias folded into the prepared table Z[q][k] = w_out[q] .
// codebook[q][k] + b_out[q].  Per frame the work is n_q codes in and D floats
// out, but each output float needs n_q table reads: the on-chip gathers, not
// HBM, set the pace.  The table (33.6 MB at D=1024, Q=8) stays in L2; the
// threads of a frame sum their float4 columns of the n_q rows in stage order,
// so each warp instruction reads 512 contiguous bytes of one table row.
// With the codec's fc2 folded into Z (Z = fc2_w . stage output, D_out wide)
// the sum starts at fc2_b; without it, at zero.
//
// (Reading the table from shared memory measured slower on the 192 000-frame
// workload.  A CTA holds at most a 4-column slice of the table (128 KB at
// Q = 8, K = 1024), so it writes 16 bytes per frame.  With each codeword's 8
// stage pieces laid side by side and the lanes of a quarter-warp reading
// stages (lane + step) mod 8, the gather is free of bank conflicts and runs at
// 56 % of the HBM roofline without stores; the 16-byte stores then cost as
// much again -- 514 us as scattered stores, 600 us as TMA stores of 16-byte
// wide boxes -- against about 300 us for the L2 gather here.)
#include "rvq_internal.cuh"

namespace rvq {
namespace {

// One CTA per frame, one thread per float4 column group (the frame index is
// the CTA index, so the frame's codes and the rows they select are the same
// for every thread of a warp).  A code outside [0, K) is read as row 0 and
// weighted by 0, so every stage's load is issued without a branch and the
// rows of all stages can be in flight at once; the sum is taken in stage
// order, starting at the decode bias when the tables hold one (*b_used, set
// by rvq_prepare) and at zero otherwise.  What limits the kernel is the L2:
// each output float is the sum of n_q table reads, and the gathers run at
// about 22 TB/s of L2 reads on the GB300.

// n_q, K and D/4 fixed at compile time: the compiler then keeps the row
// loads of a thread in flight, about 1.4x faster than the general kernel
// below on the OmniVoice codec's 8 x 1024 x 1024 shape.  Instantiated for the
// shapes of the codecs on the source pages (OmniVoice: 8 stages of 1024
// entries into 1024; MOSS: 32 stages into 768, 9-10 % faster than the general
// kernel; Audio8: 10 stages of 4096, 21 % faster).  (OmniVoice with fc2, 256
// wide, measured the same either way and takes the general kernel.)
template <int NQ, int KC, int DC>
__global__ void __launch_bounds__(DC) k_decode_fixed(const float4 *__restrict__ Z4, const float4 *__restrict__ b4,
                                                     const int *__restrict__ b_used, const int32_t *__restrict__ codes,
                                                     float4 *__restrict__ y4, unsigned long long *__restrict__ bad) {
  const int64_t n = blockIdx.x;
  const int c = threadIdx.x;
  float4 acc = __ldg(b_used) != 0 ? __ldg(b4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  int n_bad = 0;
  const auto add = [&](int q, int code) {
    const bool ok = (unsigned)code < (unsigned)KC;
    const float w = ok ? 1.f : 0.f;
    code = ok ? code : 0;
    const float4 z = __ldg(Z4 + ((int64_t)q * KC + code) * DC + c);
    acc.x = fmaf(z.x, w, acc.x);
    acc.y = fmaf(z.y, w, acc.y);
    acc.z = fmaf(z.z, w, acc.z);
    acc.w = fmaf(z.w, w, acc.w);
    n_bad += !ok;
  };
  if constexpr (NQ % 4 == 0) {
    // the codes four at a time (16-byte aligned, checked by the launcher):
    // each warp load is one L1 wavefront, and the kernel is bound
    // by the L1's wavefront rate and the L2's sector rate, so one load per
    // four stages instead of one per stage took 1.5 % (307 -> 302 us for
    // 192 000 frames; 65 -> 63 us for 12 000 MOSS frames).  Deep stacks are
    // unrolled by 8 stages, not fully: at 32 stages the full unroll kept
    // fewer loads in flight (71.6 against 63.4 us for 12 000 MOSS frames).
    constexpr int UNROLL = NQ > 16 ? 2 : NQ / 4;
    const int4 *c4 = reinterpret_cast<const int4 *>(codes + n * NQ);
#pragma unroll UNROLL
    for (int g = 0; g < NQ / 4; ++g) {
      const int4 cv = __ldg(c4 + g);
      add(4 * g, cv.x);
      add(4 * g + 1, cv.y);
      add(4 * g + 2, cv.z);
      add(4 * g + 3, cv.w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < NQ; ++q) add(q, __ldg(codes + n * NQ + q));
  }
  __stcs(y4 + n * DC + c, acc);
  if (c == 0 && bad && n_bad) atomicAdd(bad, (unsigned long long)n_bad);
}

// R stages starting at the codes cq and the column pointer zq (stage 0 of the group).
template <int R>
__device__ __forceinline__ void add_stages(float4 &acc, const int32_t *__restrict__ cq, const float4 *__restrict__ zq,
                                           int64_t stage, int K, int D4, int &n_bad) {
#pragma unroll
  for (int j = 0; j < R; ++j) {
    int code = __ldg(cq + j);
    const bool ok = (unsigned)code < (unsigned)K;
    const float w = ok ? 1.f : 0.f;
    code = ok ? code : 0;
    const float4 z = __ldg(zq + j * stage + (int64_t)code * D4);
    acc.x = fmaf(z.x, w, acc.x);
    acc.y = fmaf(z.y, w, acc.y);
    acc.z = fmaf(z.z, w, acc.z);
    acc.w = fmaf(z.w, w, acc.w);
    n_bad += !ok;
  }
}

// Any shape: the stages in groups of 8, then TAIL = n_q % 8 more.
template <int TAIL>
__global__ void __launch_bounds__(256) k_decode_any(const float4 *__restrict__ Z4, const float4 *__restrict__ b4,
                                                    const int *__restrict__ b_used, const int32_t *__restrict__ codes,
                                                    float4 *__restrict__ y4, int n_q, int K, int D4,
                                                    unsigned long long *__restrict__ bad) {
  const int64_t n = blockIdx.x;
  const int32_t *cn = codes + n * n_q;
  const int64_t stage = (int64_t)K * D4;
  const bool with_bias = __ldg(b_used) != 0;
  const int n_full = n_q >> 3;
  int n_bad = 0, iters = 0;
  for (int c = threadIdx.x; c < D4; c += blockDim.x, ++iters) {
    float4 acc = with_bias ? __ldg(b4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 *zq = Z4 + c;
    const int32_t *cq = cn;
    for (int g = 0; g < n_full; ++g, cq += 8, zq += 8 * stage) add_stages<8>(acc, cq, zq, stage, K, D4, n_bad);
    if constexpr (TAIL > 0) add_stages<TAIL>(acc, cq, zq, stage, K, D4, n_bad);
    __stcs(y4 + n * D4 + c, acc);
  }
  // every column pass saw the same codes
  if (threadIdx.x == 0 && bad && n_bad) atomicAdd(bad, (unsigned long long)(n_bad / iters));
}

template <int TAIL>
cudaError_t launch_any(dim3 grid, int threads, cudaStream_t st, const float4 *Z4, const float4 *b4, const int *b_used,
                       const int32_t *codes, float4 *y4, int n_q, int K, int D4, unsigned long long *bad) {
  k_decode_any<TAIL><<<grid, threads, 0, st>>>(Z4, b4, b_used, codes, y4, n_q, K, D4, bad);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const rvq_dims &dm, const void *tables, const int32_t *codes, int64_t n, int n_q, float *y,
                          int64_t *bad, cudaStream_t st) {
  const TablesLayout L = tables_layout(dm);
  unsigned long long *bad_u = reinterpret_cast<unsigned long long *>(bad);
  const int D4 = dim_out(dm) / 4;
  const float4 *Z4 = at<float4>(tables, L.z), *b4 = at<float4>(tables, L.b_dec);
  const int *b_used = at<int>(tables, L.b_dec_used);
  float4 *y4 = reinterpret_cast<float4 *>(y);
  if (n > 0x7fffffffLL) return cudaErrorInvalidValue;  // one CTA per frame
  const dim3 grid((unsigned)n);
  // The fixed kernels of 8 and 32 stages read the codes as int4.  rvq_decode
  // refuses codes that are not 16-byte aligned and a frame's codes are 32 or
  // 128 bytes, so every frame is aligned there; the check guards the library's
  // own callers, which pass chunks of a codes buffer.
  const bool codes16 = (reinterpret_cast<uintptr_t>(codes) & 15) == 0;
  if (codes16 && dm.K == 1024 && n_q == 8 && D4 == 256) {
    k_decode_fixed<8, 1024, 256><<<grid, 256, 0, st>>>(Z4, b4, b_used, codes, y4, bad_u);
    return cudaGetLastError();
  }
  if (codes16 && dm.K == 1024 && n_q == 32 && D4 == 192) {
    k_decode_fixed<32, 1024, 192><<<grid, 192, 0, st>>>(Z4, b4, b_used, codes, y4, bad_u);
    return cudaGetLastError();
  }
  if (dm.K == 4096 && n_q == 10 && D4 == 256) {
    k_decode_fixed<10, 4096, 256><<<grid, 256, 0, st>>>(Z4, b4, b_used, codes, y4, bad_u);
    return cudaGetLastError();
  }
  const int threads = D4 >= 256 ? 256 : (D4 + 31) / 32 * 32;
  switch (n_q & 7) {
    case 0: return launch_any<0>(grid, threads, st, Z4, b4, b_used, codes, y4, n_q, dm.K, D4, bad_u);
    case 1: return launch_any<1>(grid, threads, st, Z4, b4, b_used, codes, y4, n_q, dm.K, D4, bad_u);
    case 2: return launch_any<2>(grid, threads, st, Z4, b4, b_used, codes, y4, n_q, dm.K, D4, bad_u);
    case 3: return launch_any<3>(grid, threads, st, Z4, b4, b_used, codes, y4, n_q, dm.K, D4, bad_u);
    case 4: return launch_any<4>(grid, threads, st, Z4, b4, b_used, codes, y4, n_q, dm.K, D4, bad_u);
    case 5: return launch_any<5>(grid, threads, st, Z4, b4, b_used, codes, y4, n_q, dm.K, D4, bad_u);
    case 6: return launch_any<6>(grid, threads, st, Z4, b4, b_used, codes, y4, n_q, dm.K, D4, bad_u);
    default: return launch_any<7>(grid, threads, st, Z4, b4, b_used, codes, y4, n_q, dm.K, D4, bad_u);
  }
}

}  // namespace rvq
