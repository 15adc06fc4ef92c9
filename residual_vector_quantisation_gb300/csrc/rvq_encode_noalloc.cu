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
// context (with that device current), on the first call made in it: the
// first call on each device, and again after the device's context has
// changed (a cudaDeviceReset, or a driver-API caller that made another context
// current), since the array then lives at another address.  Make that first
// call before any stream capture begins.  Every call shares the one array and
// it keeps the previous call's contents (the status word at its head is
// cleared by each call; nothing else needs to start at zero: each call writes
// every element it later reads).  Calls that can overlap on the GPU -- on
// different streams, or on one stream from several threads without ordering
// -- race on the array and must be avoided.  rvq_read_status(NULL, stream)
// reads the last call's status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "rvq_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = RVQ_STATIC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Per device index: the context the address was looked up in (its unique id)
// and the address.
constexpr int kMaxDevices = 64;
struct CachedAddress {
  unsigned long long ctx_id;
  void *ptr;
};
CachedAddress g_cache[kMaxDevices];
std::mutex g_cache_mutex;

PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;
std::once_flag g_driver_once;

void load_driver_entry_points() {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

// Unique id of the current context (0 if there is none yet).
cudaError_t current_context_id(unsigned long long *id) {
  std::call_once(g_driver_once, load_driver_entry_points);
  if (!g_ctx_get_current || !g_ctx_get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return cudaErrorContextIsDestroyed;
  *id = 0;
  if (ctx && g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorContextIsDestroyed;
  return cudaSuccess;
}

}  // namespace

namespace rvq {

// Device address of g_static_scratch in the current context.
cudaError_t static_scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  if ((e = current_context_id(&id)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cache_mutex);
  if (id != 0 && g_cache[dev].ctx_id == id && g_cache[dev].ptr) {
    *out = g_cache[dev].ptr;
    return cudaSuccess;
  }
  void *p = nullptr;
  // also makes the device's primary context current when no context was yet
  if ((e = cudaGetSymbolAddress(&p, g_static_scratch)) != cudaSuccess) return e;
  if (id == 0 && (e = current_context_id(&id)) != cudaSuccess) return e;
  g_cache[dev] = {id, p};
  *out = p;
  return cudaSuccess;
}

}  // namespace rvq

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
  if (rvq::static_scratch_address(&scratch) != cudaSuccess) return RVQ_ERR_CUDA;
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
