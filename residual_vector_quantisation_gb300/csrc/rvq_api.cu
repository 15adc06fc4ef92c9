// Host entry points of the C ABI declared in include/rvq.h.
//
// Every entry point validates its arguments on the host before touching the
// CUDA runtime, so the early-return paths work on a machine with no GPU.
// Nothing here allocates or frees; only the two readers (rvq_read_status,
// rvq_read_error_count) synchronise a stream.
#include <stdint.h>

#include "rvq_internal.cuh"


namespace {

using rvq::TablesLayout;

// projections per encode chunk: large enough that a call of a few hundred
// thousand frames runs in one chunk (one launch of each kernel: on 192 000
// frames 1.544 ms against 1.601 ms in five chunks of 38 912)
constexpr size_t kChunkTargetBytes = size_t(512) << 20;
constexpr int64_t kChunkQuantum = 128;                   // frames

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

rvq_status check_dims(const rvq_dims &dm) {
  if (dm.D <= 0 || dm.d <= 0 || dm.K <= 0 || dm.Q <= 0) return RVQ_ERR_INVALID_ARG;
  if (dm.metric != RVQ_METRIC_L2 && dm.metric != RVQ_METRIC_COSINE) return RVQ_ERR_INVALID_ARG;
  if (dm.d != rvq::kCodeDim && dm.d != rvq::kCodeDimSmall) return RVQ_ERR_UNSUPPORTED;
  if (dm.K % 128 != 0 || dm.K > (dm.d == rvq::kCodeDim ? 65536 : rvq::kMaxKSmall)) return RVQ_ERR_UNSUPPORTED;
  if (dm.D % 16 != 0 || dm.D > 16384) return RVQ_ERR_UNSUPPORTED;
  if (dm.D_in < 0 || dm.D_out < 0) return RVQ_ERR_INVALID_ARG;
  if (dm.D_in % 16 != 0 || dm.D_in > 16384 || dm.D_out % 16 != 0 || dm.D_out > 16384) return RVQ_ERR_UNSUPPORTED;
  if (dm.Q > rvq::kMaxStages) return RVQ_ERR_UNSUPPORTED;
  return RVQ_OK;
}

size_t row_bytes(const rvq_dims &dm, int32_t n_q) { return (size_t)n_q * dm.d * sizeof(float); }

// Frames per encode chunk for a given scratch size (0 if the scratch is too small).
int64_t chunk_frames(const rvq_dims &dm, int32_t n_q, int64_t n_frames, size_t scratch_bytes) {
  const size_t rb = row_bytes(dm, n_q);
  if (scratch_bytes <= rvq::kScratchHeader) return 0;
  int64_t fit = (int64_t)((scratch_bytes - rvq::kScratchHeader) / rb);
  if (fit >= n_frames) return n_frames;
  fit = fit / kChunkQuantum * kChunkQuantum;
  return fit;
}

rvq_status launch_status(cudaError_t e) { return e == cudaSuccess ? RVQ_OK : RVQ_ERR_CUDA; }

int device_sms() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      v <= 0)
    return 1;
  return v;
}

rvq_status encode_impl(const rvq_dims &dm, const void *tables, const float *x, int64_t n_frames, int32_t n_q,
                       int32_t *codes, void *scratch, size_t scratch_bytes, cudaStream_t st) {
  int64_t chunk = chunk_frames(dm, n_q, n_frames, scratch_bytes);
  // a chunk of whole waves: one 256-frame search item per SM
  const int64_t wave = 256 * (int64_t)device_sms();
  if (chunk < n_frames && chunk >= wave) chunk = chunk / wave * wave;
  int *status = static_cast<int *>(scratch);
  float *p0 = reinterpret_cast<float *>(static_cast<char *>(scratch) + rvq::kScratchHeader);
  if (chunk >= n_frames && rvq::stream_supported(dm, n_q, n_frames))  // one small batch: its first kernel
    return launch_status(                                              // clears the status word
        rvq::launch_encode_stream(dm, tables, x, n_frames, n_q, codes, p0, status, true, st));
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return RVQ_ERR_CUDA;
  for (int64_t n0 = 0; n0 < n_frames; n0 += chunk) {
    const int64_t n = (n_frames - n0 < chunk) ? n_frames - n0 : chunk;
    cudaError_t e = rvq::launch_encode_chunk(dm, tables, x, n0, n, n_q, codes, p0, status, st);
    if (e != cudaSuccess) return RVQ_ERR_CUDA;
  }
  return RVQ_OK;
}

rvq_status check_encode_args(const rvq_dims &dm, const void *tables, const float *x, int64_t n_frames, int32_t n_q,
                             const int32_t *codes, const void *scratch, size_t scratch_bytes) {
  rvq_status s = check_dims(dm);
  if (s != RVQ_OK) return s;
  if (n_frames < 0 || n_q < 1 || n_q > dm.Q) return RVQ_ERR_INVALID_ARG;
  if (n_frames == 0) return RVQ_OK;
  if (!tables || !x || !codes || !scratch) return RVQ_ERR_INVALID_ARG;
  if (!aligned256(tables) || !aligned16(x) || !aligned16(scratch) || !aligned16(codes)) return RVQ_ERR_INVALID_ARG;
  if (chunk_frames(dm, n_q, n_frames, scratch_bytes) <= 0) return RVQ_ERR_INVALID_ARG;
  return RVQ_OK;
}

}  // namespace

extern "C" {

RVQ_API rvq_status rvq_dims_supported(rvq_dims dims) { return check_dims(dims); }

RVQ_API size_t rvq_tables_bytes(rvq_dims dims) {
  if (check_dims(dims) != RVQ_OK) return 0;
  return rvq::tables_layout(dims).total;
}

RVQ_API rvq_status rvq_prepare(rvq_dims dims, const rvq_weights *weights, void *tables, size_t tables_bytes,
                               rvq_stream_t stream) {
  rvq_status s = check_dims(dims);
  if (s != RVQ_OK) return s;
  if (!weights || !weights->w_in || !weights->codebook || !weights->w_out || !tables) return RVQ_ERR_INVALID_ARG;
  if (!aligned256(tables) || !aligned16(weights->w_in) || !aligned16(weights->codebook) ||
      !aligned16(weights->w_out))
    return RVQ_ERR_INVALID_ARG;
  // frames of another width need fc; an output of another width needs fc2
  if (!weights->fc_w && rvq::dim_in(dims) != dims.D) return RVQ_ERR_INVALID_ARG;
  if (!weights->fc2_w && rvq::dim_out(dims) != dims.D) return RVQ_ERR_INVALID_ARG;
  if ((weights->fc_b && !weights->fc_w) || (weights->fc2_b && !weights->fc2_w)) return RVQ_ERR_INVALID_ARG;
  if (tables_bytes < rvq::tables_layout(dims).total) return RVQ_ERR_INVALID_ARG;
  return launch_status(rvq::launch_prepare(dims, *weights, tables, reinterpret_cast<cudaStream_t>(stream)));
}

RVQ_API size_t rvq_encode_min_scratch_bytes(rvq_dims dims, int32_t n_q) {
  if (check_dims(dims) != RVQ_OK || n_q < 1 || n_q > dims.Q) return 0;
  return rvq::kScratchHeader + (size_t)kChunkQuantum * row_bytes(dims, n_q);
}

RVQ_API size_t rvq_encode_scratch_bytes(rvq_dims dims, int64_t n_frames, int32_t n_q) {
  if (check_dims(dims) != RVQ_OK || n_q < 1 || n_q > dims.Q || n_frames < 0) return 0;
  const size_t rb = row_bytes(dims, n_q);
  int64_t target = (int64_t)(kChunkTargetBytes / rb) / kChunkQuantum * kChunkQuantum;
  if (target < kChunkQuantum) target = kChunkQuantum;
  const int64_t frames = n_frames < target ? (n_frames > 0 ? n_frames : 1) : target;
  return rvq::kScratchHeader + (size_t)frames * rb;
}

RVQ_API rvq_status rvq_encode(rvq_dims dims, const void *tables, const float *x, int64_t n_frames, int32_t n_q,
                              int32_t *codes, void *scratch, size_t scratch_bytes, rvq_stream_t stream) {
  rvq_status s = check_encode_args(dims, tables, x, n_frames, n_q, codes, scratch, scratch_bytes);
  if (s != RVQ_OK || n_frames == 0) return s;
  return encode_impl(dims, tables, x, n_frames, n_q, codes, scratch, scratch_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

RVQ_API rvq_status rvq_decode(rvq_dims dims, const void *tables, const int32_t *codes, int64_t n_frames, int32_t n_q,
                              float *y, int64_t *bad_codes, rvq_stream_t stream) {
  rvq_status s = check_dims(dims);
  if (s != RVQ_OK) return s;
  if (n_frames < 0 || n_q < 1 || n_q > dims.Q) return RVQ_ERR_INVALID_ARG;
  if (n_frames == 0) return RVQ_OK;
  if (!tables || !codes || !y) return RVQ_ERR_INVALID_ARG;
  if (!aligned256(tables) || !aligned16(y) || !aligned16(codes)) return RVQ_ERR_INVALID_ARG;
  if (bad_codes && (reinterpret_cast<uintptr_t>(bad_codes) & 7u)) return RVQ_ERR_INVALID_ARG;
  return launch_status(
      rvq::launch_decode(dims, tables, codes, n_frames, n_q, y, bad_codes, reinterpret_cast<cudaStream_t>(stream)));
}

RVQ_API rvq_status rvq_reconstruct(rvq_dims dims, const void *tables, const float *x, int64_t n_frames, int32_t n_q,
                                   int32_t *codes, float *x_hat, void *scratch, size_t scratch_bytes,
                                   rvq_stream_t stream) {
  rvq_status s = check_encode_args(dims, tables, x, n_frames, n_q, codes, scratch, scratch_bytes);
  if (s != RVQ_OK) return s;
  if (n_frames == 0) return RVQ_OK;
  if (!x_hat || !aligned16(x_hat)) return RVQ_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  s = encode_impl(dims, tables, x, n_frames, n_q, codes, scratch, scratch_bytes, st);
  if (s != RVQ_OK) return s;
  return launch_status(rvq::launch_decode(dims, tables, codes, n_frames, n_q, x_hat, nullptr, st));
}

RVQ_API const char *rvq_status_string(rvq_status status) {
  switch (status) {
    case RVQ_OK: return "ok";
    case RVQ_ERR_INVALID_ARG: return "invalid argument";
    case RVQ_ERR_UNSUPPORTED: return "unsupported shape";
    case RVQ_ERR_WORKSPACE: return "workspace too small";
    case RVQ_ERR_CUDA: return "CUDA launch failed";
    case RVQ_ERR_TIMEOUT: return "device wait timed out";
    case RVQ_ERR_CANCELLED: return "cancelled";
    case RVQ_ERR_INTERNAL: return "internal error (a kernel refused its launch shape)";
  }
  return "unknown status";
}

RVQ_API rvq_status rvq_stream_plan(rvq_dims dims, int32_t n_q, int64_t n_frames, int64_t *plan) {
  const rvq_status s = check_dims(dims);
  if (s != RVQ_OK) return s;
  if (n_q < 1 || n_q > dims.Q || n_frames < 0 || plan == nullptr) return RVQ_ERR_INVALID_ARG;
  return rvq::stream_plan(dims, n_q, n_frames, plan) == cudaSuccess ? RVQ_OK : RVQ_ERR_CUDA;
}

RVQ_API rvq_status rvq_read_status(const void *scratch, rvq_stream_t stream) {
  if (scratch && !aligned16(scratch)) return RVQ_ERR_INVALID_ARG;
  const void *word_at = scratch;
  if (!word_at) {
    void *p = nullptr;
    if (rvq::static_scratch_address(&p) != cudaSuccess) return RVQ_ERR_CUDA;
    word_at = p;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  // ordered after the encode on its stream, then waited for
  if (cudaMemcpyAsync(&word, word_at, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return RVQ_ERR_CUDA;
  return rvq::status_from_word(word);
}

RVQ_API rvq_status rvq_read_error_count(const int64_t *bad_codes, int64_t *n_bad_codes, rvq_stream_t stream) {
  if (!bad_codes || !n_bad_codes || (reinterpret_cast<uintptr_t>(bad_codes) & 7u)) return RVQ_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int64_t v = 0;
  if (cudaMemcpyAsync(&v, bad_codes, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return RVQ_ERR_CUDA;
  *n_bad_codes = v;
  return RVQ_OK;
}

RVQ_API const char *rvq_version(void) { return "rvq-gb300 0.4.0 (sm_103a)"; }

}  // extern "C"
