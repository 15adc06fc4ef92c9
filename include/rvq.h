/*
 * rvq.h -- C ABI for residual vector quantisation (RVQ) encode and decode on
 * one NVIDIA GB300 GPU (sm_103a).
 *
 * Plain C99, extern "C", only rvq_* symbols exported.  Conventions follow the
 * plain-C ABI discipline of omnivoice.cpp ARCHITECTURE.md, sections "Public
 * API" and "ABI guarantee": a status enum where 0 is success and negative
 * values are errors, and a header that C, C++ and ctypes consume alike.  The
 * operation set (encode, decode, reconstruct, prefix depth) follows the codec
 * API of moss-tts.cpp AGENTS.md ("Layout": moss::Codec encode / decode /
 * reconstruct) and its bitrate control (gotcha 12: use the first k stages).
 *
 * What is computed (omnivoice.cpp ARCHITECTURE.md, section "RVQ codec"):
 *   encode, per frame, for stage q = 0 .. n_q-1:
 *     p_q       = w_in[q] . residual + b_in[q]
 *     code_q    = argmin_k || p_q - codebook[q][k] ||^2   (lowest k on ties)
 *     residual -= w_out[q] . codebook[q][code_q] + b_out[q]
 *   decode:  y = sum_{q < n_q} ( w_out[q] . codebook[q][code_q] + b_out[q] )
 *   with residual = x on entry.
 * With metric RVQ_METRIC_COSINE the argmin is taken between L2-normalised
 * vectors, || p_q/n(p_q) - codebook[q][k]/n(codebook[q][k]) ||^2 with
 * n(v) = max(||v||_2, 1e-12) (moss-tts.cpp AGENTS.md, gotcha 9: the quantizer
 * L2-normalises the projected encoding and the codebook before the argmin in
 * code space); the residual update and decode still use the stored codeword.
 * Optionally the Linear layers around the quantizer in that codec
 * (omnivoice.cpp ARCHITECTURE.md, "Audio tokenizer" data flow: fc 1024 -> 1024
 * before the RVQ encode, fc2 1024 -> 256 after the RVQ decode) are folded
 * into the tables: encode then takes frames of width D_in and maps each by
 * fc (x' = fc_w . x + fc_b) before the loop, and decode returns
 * fc2_w . y + fc2_b, of width D_out.
 *
 * Shapes and layouts (all float32 row-major, PyTorch (out, in) layouts as in
 * that section's tensor table):
 *   w_in     [Q][d][D]      b_in  [Q][d]  (nullable: zero)
 *   codebook [Q][K][d]
 *   w_out    [Q][D][d]      b_out [Q][D]  (nullable: zero)
 *   fc_w [D][D_in], fc_b [D]; fc2_w [D_out][D], fc2_b [D_out]   (all nullable)
 *   x [N][D_in], y and x_hat [N][D_out]   frame-major: one contiguous vector per frame
 *   codes    [N][n_q] int32 frame-major (moss-tts.cpp AGENTS.md, gotcha 8)
 *
 * Memory and ownership.  Every pointer except the struct pointers is DEVICE
 * memory owned by the caller.  The library allocates nothing, frees nothing
 * and never synchronises the stream (except rvq_read_status,
 * rvq_read_error_count and the synchronous host pipeline): each call
 * validates its arguments on the host, enqueues kernels on `stream` and
 * returns.  Results are ready when the stream reaches that point.
 *   tables  -- written by rvq_prepare, read-only afterwards; the weights are
 *              not read again, so they may be freed after rvq_prepare's work
 *              has completed on its stream.  One tables buffer may serve
 *              concurrent calls on several streams.
 *   scratch -- per-call working memory of rvq_encode / rvq_reconstruct.
 *              Calls that may overlap on the GPU need separate scratch.
 *
 * Errors.  Arguments are checked before any launch:
 *   RVQ_ERR_INVALID_ARG  null pointer, n_frames < 0, n_q outside [1, Q], a
 *                        tables or scratch buffer smaller than required, a
 *                        device pointer not 16-byte aligned;
 *   RVQ_ERR_UNSUPPORTED  shapes the kernels do not handle (see
 *                        rvq_dims_supported);
 *   RVQ_ERR_CUDA         a launch failed (cudaGetLastError after launch).
 * Failures found on the device after a call has returned (a bounded device
 * wait that gave up: RVQ_ERR_TIMEOUT; a kernel that refused its launch shape:
 * RVQ_ERR_INTERNAL) are recorded in the status word at the head of the encode
 * scratch and read with rvq_read_status; the host pipeline reads them itself.
 * n_frames == 0 is valid and enqueues nothing.  Inputs must be finite; the
 * result for NaN or Inf inputs is unspecified.  Codes given to rvq_decode
 * outside [0, K) contribute nothing and are counted (see rvq_decode).
 */
#ifndef RVQ_H
#define RVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(_WIN32)
#define RVQ_API
#else
#define RVQ_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define RVQ_VERSION_MAJOR 0
#define RVQ_VERSION_MINOR 4
#define RVQ_VERSION_PATCH 0

/* Distance of the argmin (rvq_dims.metric). */
#define RVQ_METRIC_L2 0     /* squared L2 between p and the codeword */
#define RVQ_METRIC_COSINE 1 /* squared L2 between the L2-normalised vectors */

typedef enum rvq_status {
  RVQ_OK = 0,
  RVQ_ERR_INVALID_ARG = -1,
  RVQ_ERR_UNSUPPORTED = -2,
  RVQ_ERR_WORKSPACE = -3,
  RVQ_ERR_CUDA = -4,
  RVQ_ERR_TIMEOUT = -5,
  RVQ_ERR_CANCELLED = -6,
  RVQ_ERR_INTERNAL = -7
} rvq_status;

/* D: the quantizer's input (residual) dimension; d: code-space dimension;
 * K: entries per codebook; Q: number of stages held in the tables; metric:
 * RVQ_METRIC_L2 or RVQ_METRIC_COSINE; D_in: width of the frames given to
 * encode (with fc; 0 or D without); D_out: width of decode's output (with
 * fc2; 0 or D without).  An initialiser that leaves out the last three gives
 * RVQ_METRIC_L2 and no fc or fc2.  Tables prepared for one set of dims serve
 * only those dims. */
typedef struct rvq_dims {
  int32_t D;
  int32_t d;
  int32_t K;
  int32_t Q;
  int32_t metric;
  int32_t D_in;
  int32_t D_out;
} rvq_dims;

/* Device pointers to the per-stage tensors and the optional Linear layers
 * (layouts above).  fc_w must be given when dims.D_in is neither 0 nor D,
 * and fc2_w when dims.D_out is neither 0 nor D; when given they are used
 * (even at D_in == D or D_out == D). */
typedef struct rvq_weights {
  const float *w_in;
  const float *b_in;
  const float *codebook;
  const float *w_out;
  const float *b_out;
  const float *fc_w;
  const float *fc_b;
  const float *fc2_w;
  const float *fc2_b;
} rvq_weights;

/* Same type as cudaStream_t; the header needs no CUDA include.  NULL is the
 * legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *rvq_stream_t;

/* RVQ_OK if the kernels handle these dims, else RVQ_ERR_UNSUPPORTED (or
 * RVQ_ERR_INVALID_ARG for non-positive values or an unknown metric).
 * Supported: d == 64 with K a multiple of 128, K <= 65536; or d == 8 with K
 * a multiple of 128, K <= 1024 (two stages' codebooks stay on chip);
 * D, and D_in and D_out when non-zero, multiples of 16 up to 16384;
 * 1 <= Q <= 64; either metric. */
RVQ_API rvq_status rvq_dims_supported(rvq_dims dims);

/* Bytes of the tables buffer for these dims (0 if unsupported). */
RVQ_API size_t rvq_tables_bytes(rvq_dims dims);

/* Fill `tables` (tables_bytes >= rvq_tables_bytes(dims), 256-byte aligned)
 * from the weights.  The tables hold, computed in float64 and rounded once to
 * float32: squared codebook norms (of the normalised codewords for
 * RVQ_METRIC_COSINE); the decode table
 *   Z[q][k] = w_out[q] . codebook[q][k] + b_out[q]           ([Q][K][D]);
 * and the cross-stage table
 *   G[q][s][k] = w_in[q] . Z[s][k]   for s < q               ([Q(Q-1)/2][K][d]),
 * which lets encode update every stage's projection without materialising the
 * D-dimensional residual:  w_in[q] . residual_q = w_in[q] . x - sum_{s<q} G[q][s][code_s].
 * Both are exact re-associations of the sums in the "RVQ codec" section.
 * With fc, the projections read fc_w-mapped frames: w_in[q] . fc_w (and
 * w_in[q] . fc_b + b_in[q]) replace w_in[q] (and b_in[q]); with fc2, Z holds
 * fc2_w . Z[q][k] ([Q][K][D_out]) and fc2_b is added once per frame.
 * Also a copy of w_in (with fc folded in) split into TF32 high and low parts, and -2 x the
 * codebook (normalised first for RVQ_METRIC_COSINE) split the same way, in the
 * layouts the kernels read.  Asynchronous on `stream`. */
RVQ_API rvq_status rvq_prepare(rvq_dims dims, const rvq_weights *weights, void *tables,
                               size_t tables_bytes, rvq_stream_t stream);

/* Scratch bytes rvq_encode / rvq_reconstruct need for n_frames frames at
 * depth n_q.  Scratch starts with a 256-byte header whose first int32 is a
 * device status word: each call sets it to 0, and a kernel sets it to 5 if
 * one of its bounded device waits gave up, or to 6 if it was launched in a
 * shape it does not accept (an internal error); either way that call's codes
 * are invalid (read it after the stream reaches the call).  The rest holds the
 * per-frame stage projections ([chunk][n_q*d] float32) of one chunk of
 * frames; encode works through the frames chunk by chunk.  This returns the
 * size for chunks of up to about 512 MiB of projections.  A larger scratch is
 * accepted and used for larger chunks; a smaller one (at least
 * rvq_encode_min_scratch_bytes) gives smaller chunks. */
RVQ_API size_t rvq_encode_scratch_bytes(rvq_dims dims, int64_t n_frames, int32_t n_q);
RVQ_API size_t rvq_encode_min_scratch_bytes(rvq_dims dims, int32_t n_q);

/* Encode n_frames frames x [N][D_in] with the first n_q stages (1 <= n_q <= Q)
 * into codes [N][n_q].  Each code is the argmin of the squared L2 distance,
 * lowest index on ties.  The distances are computed to about float32
 * accuracy; where two entries' distances differ by less than that, either
 * may be returned. */
RVQ_API rvq_status rvq_encode(rvq_dims dims, const void *tables, const float *x, int64_t n_frames,
                              int32_t n_q, int32_t *codes, void *scratch, size_t scratch_bytes,
                              rvq_stream_t stream);

/* Decode codes [N][n_q] into y [N][D_out]:
 *   y[n] = fc2_b + sum_{q < n_q} Z[q][codes[n][q]]   (summed in stage order,
 *   float32; fc2_b is zero without fc2).
 * A code outside [0, K) contributes nothing; if bad_codes (device, int64) is
 * not NULL, the number of such codes is added to *bad_codes (atomically; the
 * caller zeroes it). */
RVQ_API rvq_status rvq_decode(rvq_dims dims, const void *tables, const int32_t *codes,
                              int64_t n_frames, int32_t n_q, float *y, int64_t *bad_codes,
                              rvq_stream_t stream);

/* Encode then decode: codes [N][n_q] (required) and x_hat [N][D_out] =
 * decode(codes), the quantised reconstruction of x (without fc and fc2,
 * x - x_hat is the final residual). */
RVQ_API rvq_status rvq_reconstruct(rvq_dims dims, const void *tables, const float *x,
                                   int64_t n_frames, int32_t n_q, int32_t *codes, float *x_hat,
                                   void *scratch, size_t scratch_bytes, rvq_stream_t stream);

/* Status of the encode work last enqueued with `scratch` (the scratch buffer
 * given to rvq_encode or rvq_reconstruct; NULL reads the library's own scratch
 * on the current device, the one rvq_encode_static uses).  Synchronises
 * `stream` (the stream of that call), then reads the status word at the head
 * of the scratch: RVQ_OK when that call's kernels ran cleanly,
 * RVQ_ERR_TIMEOUT when one of their bounded device waits gave up and
 * RVQ_ERR_INTERNAL when a kernel refused its launch shape -- either way the
 * call's codes are invalid.  RVQ_ERR_INVALID_ARG for a scratch pointer that
 * is not 16-byte aligned, RVQ_ERR_CUDA if synchronising or reading fails.
 * This is the one entry point besides the host pipeline that waits for the
 * GPU.  (Omnivoice.cpp ARCHITECTURE.md, "Status codes": every failure is
 * reported as a status value, none is left to be inferred.) */
RVQ_API rvq_status rvq_read_status(const void *scratch, rvq_stream_t stream);

/* Read the bad-code counter of rvq_decode (`bad_codes`, device int64,
 * 8-byte aligned) into *n_bad_codes (host) after synchronising `stream`.
 * RVQ_ERR_INVALID_ARG for a null or misaligned pointer, RVQ_ERR_CUDA if the
 * synchronisation or the copy fails. */
RVQ_API rvq_status rvq_read_error_count(const int64_t *bad_codes, int64_t *n_bad_codes, rvq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Host-memory pipeline: frames in host memory in, codes and reconstruction in
 * host memory out.  The frames are processed in chunks of chunk_frames
 * through three device buffer slots carved from a caller-owned workspace;
 * three streams overlap the host-to-device copy of one chunk, the encode +
 * decode of the previous one and the device-to-host copy of the one before
 * (pinned host memory lets the copies run at full speed).  The pipeline owns
 * three CUDA streams and nine events on the device that was current at
 * creation; it allocates no memory.  One pipeline serves one call at a time.
 * The first 256 bytes of the workspace hold the pipeline's status word: each
 * chunk's device status is folded into it, and rvq_pipeline_reconstruct
 * returns RVQ_ERR_TIMEOUT or RVQ_ERR_INTERNAL if any chunk's kernels recorded
 * a failure (see rvq_read_status).
 * --------------------------------------------------------------------------- */
typedef struct rvq_pipeline rvq_pipeline;

/* Workspace bytes for a pipeline (0 for unsupported arguments). */
RVQ_API size_t rvq_pipeline_workspace_bytes(rvq_dims dims, int32_t n_q, int64_t chunk_frames);

/* Create a pipeline for depth n_q over `workspace` (device memory, 256-byte
 * aligned, at least rvq_pipeline_workspace_bytes, caller-owned and reserved
 * until rvq_pipeline_destroy).  *out receives the pipeline. */
RVQ_API rvq_status rvq_pipeline_create(rvq_dims dims, int32_t n_q, int64_t chunk_frames, void *workspace,
                                       size_t workspace_bytes, rvq_pipeline **out);

/* Wait for the pipeline's work, release its streams and events, free it. */
RVQ_API rvq_status rvq_pipeline_destroy(rvq_pipeline *pipeline);

/* Encode and decode n_frames host frames x_host [N][D_in] with the tables of
 * rvq_prepare: codes_host [N][n_q] (required) and x_hat_host [N][D_out]
 * (nullable).  Synchronous: returns when every output is in host memory.
 * Returns RVQ_ERR_TIMEOUT / RVQ_ERR_INTERNAL if a chunk's kernels recorded a
 * device failure (its outputs are then invalid), and RVQ_ERR_CANCELLED if the
 * cancel callback asked to stop. */
RVQ_API rvq_status rvq_pipeline_reconstruct(rvq_pipeline *pipeline, const void *tables, const float *x_host,
                                            int64_t n_frames, int32_t *codes_host, float *x_hat_host);

/* Cancel callback of a pipeline: returns non-zero to stop.  As in the public
 * API of omnivoice.cpp ARCHITECTURE.md ("Public API": a cancel callback the
 * library polls between chunks), rvq_pipeline_reconstruct calls it on the
 * calling thread before it enqueues each chunk.  When it returns non-zero, no
 * further chunk is enqueued: the call waits for the chunks already enqueued
 * (their codes and reconstructions are written in full), leaves the outputs
 * of the later frames untouched and returns RVQ_ERR_CANCELLED.  `user` is
 * passed through. */
typedef int (*rvq_cancel_fn)(void *user);

/* Install (fn non-NULL) or remove (fn NULL) the pipeline's cancel callback.
 * RVQ_ERR_INVALID_ARG for a null pipeline.  Not to be called while a
 * rvq_pipeline_reconstruct on the same pipeline is running. */
RVQ_API rvq_status rvq_pipeline_set_cancel(rvq_pipeline *pipeline, rvq_cancel_fn fn, void *user);

/* Encode like rvq_encode, but with no scratch argument: for callers that
 * cannot allocate device memory when they encode (a real-time audio callback,
 * where cudaMalloc may stall on device-wide synchronisation, or an application
 * whose device memory all belongs to its own pool).  Neither omnivoice.cpp
 * ARCHITECTURE.md nor moss-tts.cpp AGENTS.md has a counterpart to this entry
 * point.
 * Scratch is a fixed RVQ_STATIC_SCRATCH_BYTES array inside the library, held
 * on every GPU that loads it until the process exits.  A call needs
 * 256 + n_frames * n_q * d * 4 bytes of it; a larger call returns RVQ_ERR_WORKSPACE
 * before launching anything (split the frames over several calls).  The
 * first call on each device (and the first after the device's context
 * changes, e.g. after cudaDeviceReset) looks up the array's device address,
 * so make it before any stream capture.  All calls share the array: calls
 * that can overlap on the GPU race and must not be issued.  The status word
 * of the last call (a device wait that gave up, say) is read with
 * rvq_read_status(NULL, stream).  Allocates nothing. */
#define RVQ_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
RVQ_API rvq_status rvq_encode_static(rvq_dims dims, const void *tables, const float *x,
                                     int64_t n_frames, int32_t n_q, int32_t *codes,
                                     rvq_stream_t stream);

/* Small batches.  A call of at most `max_frames` frames (rvq_encode,
 * rvq_reconstruct, rvq_encode_static, and each chunk of a larger call) runs on
 * low-latency kernels: the stage projections spread over many CTAs, then
 * groups of up to 16 frames on clusters of min(8, K/128) CTAs that each own
 * a slice of every codebook and exchange their best (distance, index) per
 * frame through distributed shared memory, so a call of a few frames
 * finishes in microseconds instead of walking every codeword of every stage
 * on one SM.  A cluster takes one group, or, for calls of more than 16
 * frames, as many groups (up to 8) as put the whole call in one wave of
 * clusters on the GPU, fewer where its shared memory runs out.  It computes the same
 * codes (distances in float32 FMA; ties to the lowest index) and takes
 * d = 8, or d = 64 with K <= 4096 (and n_q <= 42 when K = 128); other shapes
 * use the tile kernels.  Sets the process-wide threshold (0 turns the small-batch kernel
 * off) and returns the previous one; a negative argument only returns the
 * current value.  The default is 512 frames.  Thread-safe; a change applies to
 * calls made after it. */
RVQ_API int64_t rvq_set_stream_max_frames(int64_t max_frames);

/* How one call (or one chunk) of n_frames frames at depth n_q would run, for
 * the current device; launches nothing.  plan (host memory, 6 values):
 * [0] 1 if the call takes the small-batch kernels, else 0 and the rest 0;
 * [1] CTAs per cluster; [2] frames per group; [3] groups per cluster;
 * [4] clusters; [5] codebook slice buffers per CTA.  The first call on a
 * device asks the CUDA runtime how many clusters fit on it at once; if that
 * fails, RVQ_ERR_CUDA.  RVQ_ERR_INVALID_ARG (plan untouched) for bad dims,
 * n_q outside 1..Q, n_frames < 0 or a null plan. */
RVQ_API rvq_status rvq_stream_plan(rvq_dims dims, int32_t n_q, int64_t n_frames, int64_t *plan);

/* Static strings. */
RVQ_API const char *rvq_status_string(rvq_status status);
RVQ_API const char *rvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RVQ_H */
