// rvq_encode_static: RVQ encode for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at the point where they encode: a
// real-time audio callback, where an allocation can stall on device-wide
// synchronisation for an unbounded time, or an application whose device
// memory is all owned by its own pool allocator or was fixed at start-up.
// rvq_encode needs a caller-provided scratch buffer for its per-frame stage
// projections; this entry point uses a fixed buffer that lives in the
// library itself instead, so the caller supplies only the tables (from
// rvq_prepare), the frames and the codes.
//
// The buffer is a file-scope __device__ array of RVQ_STATIC_SCRATCH_BYTES
// (16 MiB, declared in rvq.h).
// Every GPU that loads the library holds one copy until the process exits.
// A call needs 256 + n_frames * n_q * d * 4 bytes of it (a status word, then
// the stage projections); larger calls are refused with RVQ_ERR_WORKSPACE
// before anything is launched.
//
// The array's address is looked up with cudaGetSymbolAddress once per device
// (with that device current), on the first call made on that device; make
// that first call before any stream capture begins.  Every call shares the
// one array and it keeps the previous call's contents (nothing in it needs
// to start at zero: each call writes every element it later reads).  Calls
// that can overlap on the GPU -- on different streams, or on one stream from
// several threads without ordering -- race on the array and must be avoided.
#include <atomic>
#include <mutex>

#include "rvq_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = RVQ_STATIC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of g_static_scratch on the current device (looked up once).
cudaError_t static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" RVQ_API rvq_status rvq_encode_static(rvq_dims dims, const void *tables, const float *x,
                                                int64_t n_frames, int32_t n_q, int32_t *codes,
                                                rvq_stream_t stream) {
  rvq_status s = rvq_dims_supported(dims);
  if (s != RVQ_OK) return s;
  if (n_frames < 0 || n_q < 1 || n_q > dims.Q) return RVQ_ERR_INVALID_ARG;
  if (n_frames == 0) return RVQ_OK;
  if (!tables || !x || !codes) return RVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(tables) & 255u) || (reinterpret_cast<uintptr_t>(x) & 15u) ||
      (reinterpret_cast<uintptr_t>(codes) & 15u))
    return RVQ_ERR_INVALID_ARG;
  const size_t need = rvq::kScratchHeader + (size_t)n_frames * (size_t)n_q * (size_t)dims.d * sizeof(float);
  if (need > kStaticScratchBytes) return RVQ_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return RVQ_ERR_CUDA;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int *status = static_cast<int *>(scratch);
  float *p0 = reinterpret_cast<float *>(static_cast<char *>(scratch) + rvq::kScratchHeader);
  cudaError_t e;
  if (rvq::stream_supported(dims, n_q, n_frames)) {  // its first kernel clears the status word
    e = rvq::launch_encode_stream(dims, tables, x, n_frames, n_q, codes, p0, status, true, st);
  } else {
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return RVQ_ERR_CUDA;
    e = rvq::launch_encode_chunk(dims, tables, x, 0, n_frames, n_q, codes, p0, status, st);
  }
  return e == cudaSuccess ? RVQ_OK : RVQ_ERR_CUDA;
}
