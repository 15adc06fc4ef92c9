// Internal declarations shared by the RVQ CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "rvq.h"

namespace rvq {

constexpr int kCodeDim = 64;            // d of the main kernels
constexpr int kCodeDimSmall = 8;        // d of the small-code-space kernels
constexpr int kMaxKSmall = 1024;        // K limit at d = 8 (two stages' codebooks on chip)
constexpr int kChunkCodes = 128;        // codewords per tensor-core distance chunk
constexpr size_t kScratchHeader = 256;  // status word at the head of encode scratch
constexpr int RVQ_DEVICE_TIMEOUT = 5;   // status word value: a bounded device wait gave up
constexpr int RVQ_DEVICE_BAD_LAUNCH = 6;  // status word value: a kernel refused its launch shape
constexpr int kMaxStages = 64;         // Q limit
constexpr size_t kAlign = 256;

inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// Number of (q, s) stage pairs with s < q, and the pair index of (q, s).
__host__ __device__ inline int64_t n_pairs(int Q) { return (int64_t)Q * (Q - 1) / 2; }
__host__ __device__ inline int64_t pair_index(int q, int s) { return (int64_t)q * (q - 1) / 2 + s; }

// Widths of encode's frames and decode's output (D without fc / fc2).
inline int dim_in(const rvq_dims &dm) { return dm.D_in > 0 ? dm.D_in : dm.D; }
inline int dim_out(const rvq_dims &dm) { return dm.D_out > 0 ? dm.D_out : dm.D; }

// Whether the shape can take the small-batch (streaming) kernels at all, i.e.
// whether the tables include their copies (w_in_f, cb_stream): d = 8, or
// d = 64 with slices of at most 512 codewords (K <= 4096).
inline bool stream_tables(const rvq_dims &dm) { return dm.d != kCodeDim || dm.K <= 4096; }

// Blocks of the d = 8 norm operand per stage: one per pair of 128-codeword chunks.
__host__ __device__ constexpr size_t cn_img8_blocks(int K) { return (size_t)(K / 128 + 1) / 2; }

// Byte offsets of the prepared tables inside the caller's tables buffer.
struct TablesLayout {
  size_t w_in_hi;  // [Q*d][D_in]  f32, TF32-truncated high part of w_in (. fc_w)
  size_t w_in_lo;  // [Q*d][D_in]  f32, the exact remainder
  size_t b_in;     // [Q*d]     f32 (zeros when absent)
  size_t cnorm;    // [Q][K]    f32 squared norms (float64 sums)
  size_t cb_img;   // [Q][K/128][hi,lo][2][128 x 32] f32: -2*codebook split in TF32 hi/lo,
                   //   each 128-codeword chunk as two 128-byte-swizzled K-major atoms
  size_t z;        // [Q][K][D_out] f32 decode table (fc2 folded in)
  size_t b_dec;    // [D_out]   f32 decode bias (fc2_b, zeros without fc2)
  size_t b_dec_used;  // int32: 1 if the decode bias holds fc2_b, 0 if it is all zeros
  size_t g;        // [P][K][d] f32 cross-stage table, P = Q(Q-1)/2
  size_t m64;      // [P][d][d] f64 w_in[q] . w_out[s]   (prepare temporary)
  size_t vb64;     // [P][d]    f64 w_in[q] . b_out[s]   (prepare temporary)
  size_t m2_64;    // [Q][D_out][d] f64 fc2_w . w_out[q], then [Q][D_out] fc2_w . b_out[q]  (prepare temporary)
  size_t w_in_f;   // [Q*d][D_in] f32 w_in (. fc_w) (hi + lo): the streaming path's projection
  size_t cb_stream;  // [Q][CS][d/4][K/CS] float4: the codebook (each codeword divided by n(c) for the
                     //   cosine metric) cut into the streaming path's CS = stream_cluster_size(K) slices,
                     //   each slice column-block major so one bulk copy stages it
  size_t cn_img8;  // d = 8 only: [Q][ceil(K/256)][sw32(128 rows x 8)] f32: the squared norms as the
                   //   B operand of one more MMA -- row k % 128 of the block of chunks 2i, 2i+1 holds
                   //   the exact TF32 parts (n1, n2, n3) of ||c||^2 in slots 0-2 (even chunk) or 4-6
  size_t total;
};

inline TablesLayout tables_layout(const rvq_dims &dm) {
  const size_t d = dm.d, K = dm.K, Q = dm.Q, P = (size_t)n_pairs(dm.Q);
  const size_t Di = dim_in(dm), Do = dim_out(dm);
  TablesLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  L.w_in_hi = take(Q * d * Di * 4);
  L.w_in_lo = take(Q * d * Di * 4);
  L.b_in = take(Q * d * 4);
  L.cnorm = take(Q * K * 4);
  L.cb_img = take(Q * K * d * 2 * 4);
  L.z = take(Q * K * Do * 4);
  L.b_dec = take(Do * 4);
  L.b_dec_used = take(4);
  L.g = take((P ? P : 1) * K * d * 4);
  L.m64 = take((P ? P : 1) * d * d * 8);
  L.vb64 = take((P ? P : 1) * d * 8);
  L.m2_64 = take(Q * Do * (d + 1) * 8);
  const bool st = stream_tables(dm);  // the streaming copies, else empty
  L.w_in_f = take(st ? Q * d * Di * 4 : 0);
  L.cb_stream = take(st ? Q * K * d * 4 : 0);
  L.cn_img8 = take(d == (size_t)kCodeDimSmall ? Q * cn_img8_blocks(dm.K) * 128 * 8 * 4 : 0);
  L.total = o;
  return L;
}

template <class T>
inline T *at(void *base, size_t off) { return reinterpret_cast<T *>(static_cast<char *>(base) + off); }
template <class T>
inline const T *at(const void *base, size_t off) {
  return reinterpret_cast<const T *>(static_cast<const char *>(base) + off);
}

// Launchers (each returns cudaSuccess or the launch error).
cudaError_t launch_prepare(const rvq_dims &dm, const rvq_weights &w, void *tables, cudaStream_t s);
// P0 = x . w_in'^T + b_in' on the tensor cores (3xTF32) for n frames at depth
// n_q; shape: the item shape (0: 256 frames x 256 columns, 1: 128 x 128,
// 2: 128 x 64; -1: chosen for n); zero_status clears the status word first.
cudaError_t launch_project_tc(const rvq_dims &dm, const void *tables, const float *x, int64_t n, int n_q, float *p0,
                              int *status, bool zero_status, cudaStream_t st, int shape);
cudaError_t launch_encode_chunk(const rvq_dims &dm, const void *tables, const float *x, int64_t n0,
                                int64_t n, int n_q, int32_t *codes, float *p0, int *status, cudaStream_t s);
// The streaming path (rvq_stream.cu): groups of up to kStreamFrames frames
// run on clusters of stream_cluster_size(K) CTAs (one or more groups a
// cluster), each CTA owning K/CS
// codewords of every stage.  stream_supported: true if it takes a call of
// n_frames frames at depth n_q (else the tile path does).
constexpr int kStreamFrames = 16;
constexpr int kStreamMaxFramesDefault = 512;
__host__ __device__ inline int stream_cluster_size(int K) { return K / 128 < 8 ? K / 128 : 8; }
bool stream_supported(const rvq_dims &dm, int n_q, int64_t n_frames);
// The streaming plan of a call (rvq_stream_plan's six values).
cudaError_t stream_plan(const rvq_dims &dm, int n_q, int64_t n_frames, int64_t plan[6]);
// p0: scratch for the stage projections ([n][n_q*d] f32); zero_status: the
// first kernel clears the status word (the caller has not).
cudaError_t launch_encode_stream(const rvq_dims &dm, const void *tables, const float *x, int64_t n, int n_q,
                                 int32_t *codes, float *p0, int *status, bool zero_status, cudaStream_t s);
// The d = 8 stage loop over stages [q_begin, q_end) of n_q (a stage block;
// the terms of earlier stages already subtracted from p0).
cudaError_t launch_search8(const rvq_dims &dm, const void *tables, const float *p0, int64_t n, int n_q, int q_begin,
                           int q_end, int32_t *codes, int *status, int sms, cudaStream_t s);
// Whether the d = 8 search puts one tile on each CTA, split over its three
// pipelines (no more tiles than SMs).
inline bool search8_split(int64_t n, int sms) { return (n + 127) / 128 <= sms; }
// The most stages a block of the d = 8 search spans: one stage's query terms
// fit its pipeline's staging slots.
int search8_block_stages(bool split);
cudaError_t launch_decode(const rvq_dims &dm, const void *tables, const int32_t *codes, int64_t n,
                          int n_q, float *y, int64_t *bad, cudaStream_t s);

// The status a device status word stands for (0: RVQ_OK, RVQ_DEVICE_TIMEOUT:
// RVQ_ERR_TIMEOUT, anything else: RVQ_ERR_INTERNAL).
inline rvq_status status_from_word(int word) {
  if (word == 0) return RVQ_OK;
  return word == RVQ_DEVICE_TIMEOUT ? RVQ_ERR_TIMEOUT : RVQ_ERR_INTERNAL;
}
// Device address, in the current context, of the library's own encode scratch
// (rvq_encode_noalloc.cu).
cudaError_t static_scratch_address(void **out);

}  // namespace rvq
