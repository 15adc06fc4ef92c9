// Host-memory pipeline: encode + decode frames that live in host memory.
//
// Frames are processed in chunks through three device buffer slots carved
// from a caller-owned workspace.  Three streams overlap the host-to-device
// copy of one chunk, the encode + decode of the previous one, and the
// device-to-host copy of the one before that; events order the slots.  The
// pipeline object owns only those streams and events; it allocates no memory.
//
// Failures: each chunk's encode clears and may set the status word of its
// slot's scratch; a one-thread kernel on the compute stream folds it into the
// pipeline's own status word (the head of the workspace) before the slot is
// reused, so a device wait that gave up in any chunk is reported when the
// call returns.  A cancel callback is polled between chunks (omnivoice.cpp
// ARCHITECTURE.md, "Public API": generation takes a cancel callback that the
// library polls, so a long job can be stopped between steps).
#include <new>

#include "rvq_internal.cuh"

namespace {

constexpr int kSlots = 3;
constexpr size_t kPipeHeader = 256;  // the pipeline's status word

// Keep the first failure: *acc = *chunk_status unless *acc already holds one.
__global__ void k_fold_status(int *acc, const int *chunk_status) {
  const int w = *chunk_status;
  if (w != 0 && *acc == 0) *acc = w;
}

struct SlotLayout {
  size_t x, y, codes, scratch, scratch_bytes, stride;
};

SlotLayout slot_layout(const rvq_dims &dm, int32_t n_q, int64_t chunk) {
  SlotLayout s{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = rvq::align_up(o + bytes); return at; };
  s.x = take((size_t)chunk * rvq::dim_in(dm) * sizeof(float));
  s.y = take((size_t)chunk * rvq::dim_out(dm) * sizeof(float));
  s.codes = take((size_t)chunk * n_q * sizeof(int32_t));
  s.scratch_bytes = rvq::kScratchHeader + (size_t)chunk * n_q * dm.d * sizeof(float);
  s.scratch = take(s.scratch_bytes);
  s.stride = o;
  return s;
}

}  // namespace

struct rvq_pipeline {
  rvq_dims dims;
  int32_t n_q;
  int64_t chunk;
  int device;
  unsigned char *workspace;
  SlotLayout layout;
  cudaStream_t s_in, s_comp, s_out;
  cudaEvent_t ev_in[kSlots], ev_comp[kSlots], ev_out[kSlots];
  rvq_cancel_fn cancel;
  void *cancel_user;
};

extern "C" {

RVQ_API size_t rvq_pipeline_workspace_bytes(rvq_dims dims, int32_t n_q, int64_t chunk_frames) {
  if (rvq_dims_supported(dims) != RVQ_OK || n_q < 1 || n_q > dims.Q || chunk_frames < 1) return 0;
  return kPipeHeader + kSlots * slot_layout(dims, n_q, chunk_frames).stride;
}

RVQ_API rvq_status rvq_pipeline_create(rvq_dims dims, int32_t n_q, int64_t chunk_frames, void *workspace,
                                       size_t workspace_bytes, rvq_pipeline **out) {
  if (!out) return RVQ_ERR_INVALID_ARG;
  *out = nullptr;
  rvq_status st = rvq_dims_supported(dims);
  if (st != RVQ_OK) return st;
  if (n_q < 1 || n_q > dims.Q || chunk_frames < 1 || !workspace) return RVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RVQ_ERR_INVALID_ARG;
  if (workspace_bytes < rvq_pipeline_workspace_bytes(dims, n_q, chunk_frames)) return RVQ_ERR_INVALID_ARG;
  rvq_pipeline *p = new (std::nothrow) rvq_pipeline();
  if (!p) return RVQ_ERR_WORKSPACE;
  p->dims = dims;
  p->n_q = n_q;
  p->chunk = chunk_frames;
  p->workspace = static_cast<unsigned char *>(workspace);
  p->layout = slot_layout(dims, n_q, chunk_frames);
  bool ok = cudaGetDevice(&p->device) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&p->s_comp, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < kSlots; ++i) {
    ok = ok && cudaEventCreateWithFlags(&p->ev_in[i], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&p->ev_comp[i], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&p->ev_out[i], cudaEventDisableTiming) == cudaSuccess;
  }
  if (!ok) {
    rvq_pipeline_destroy(p);
    return RVQ_ERR_CUDA;
  }
  *out = p;
  return RVQ_OK;
}

RVQ_API rvq_status rvq_pipeline_destroy(rvq_pipeline *p) {
  if (!p) return RVQ_ERR_INVALID_ARG;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(p->device);
  if (p->s_in) cudaStreamSynchronize(p->s_in);
  if (p->s_comp) cudaStreamSynchronize(p->s_comp);
  if (p->s_out) cudaStreamSynchronize(p->s_out);
  for (int i = 0; i < kSlots; ++i) {
    if (p->ev_in[i]) cudaEventDestroy(p->ev_in[i]);
    if (p->ev_comp[i]) cudaEventDestroy(p->ev_comp[i]);
    if (p->ev_out[i]) cudaEventDestroy(p->ev_out[i]);
  }
  if (p->s_in) cudaStreamDestroy(p->s_in);
  if (p->s_comp) cudaStreamDestroy(p->s_comp);
  if (p->s_out) cudaStreamDestroy(p->s_out);
  if (prev >= 0) cudaSetDevice(prev);
  delete p;
  return RVQ_OK;
}

RVQ_API rvq_status rvq_pipeline_reconstruct(rvq_pipeline *p, const void *tables, const float *x_host,
                                            int64_t n_frames, int32_t *codes_host, float *x_hat_host) {
  if (!p || n_frames < 0) return RVQ_ERR_INVALID_ARG;
  if (n_frames == 0) return RVQ_OK;
  if (!tables || !x_host || !codes_host) return RVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(tables) & 255u) != 0) return RVQ_ERR_INVALID_ARG;
  const rvq_dims dm = p->dims;
  const int32_t n_q = p->n_q;
  const SlotLayout &L = p->layout;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(p->device) != cudaSuccess) return RVQ_ERR_CUDA;
  int *fold = reinterpret_cast<int *>(p->workspace);
  rvq_status status = cudaMemsetAsync(fold, 0, sizeof(int), p->s_comp) == cudaSuccess ? RVQ_OK : RVQ_ERR_CUDA;
  const int64_t n_chunks = (n_frames + p->chunk - 1) / p->chunk;
  for (int64_t i = 0; i < n_chunks && status == RVQ_OK; ++i) {
    const int slot = (int)(i % kSlots);
    const int64_t n0 = i * p->chunk;
    const int64_t n = (n_frames - n0 < p->chunk) ? n_frames - n0 : p->chunk;
    if (p->cancel && p->cancel(p->cancel_user)) {
      status = RVQ_ERR_CANCELLED;
      break;
    }
    unsigned char *base = p->workspace + kPipeHeader + slot * L.stride;
    float *x_d = reinterpret_cast<float *>(base + L.x);
    float *y_d = reinterpret_cast<float *>(base + L.y);
    int32_t *c_d = reinterpret_cast<int32_t *>(base + L.codes);
    void *scratch = base + L.scratch;
    bool ok = true;
    // slot reuse: the copy-out of chunk i - kSlots has finished with this slot
    if (i >= kSlots) ok = ok && cudaStreamWaitEvent(p->s_in, p->ev_out[slot], 0) == cudaSuccess;
    const int64_t Di = rvq::dim_in(dm), Do = rvq::dim_out(dm);
    ok = ok && cudaMemcpyAsync(x_d, x_host + n0 * Di, (size_t)n * Di * sizeof(float), cudaMemcpyHostToDevice,
                               p->s_in) == cudaSuccess;
    ok = ok && cudaEventRecord(p->ev_in[slot], p->s_in) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(p->s_comp, p->ev_in[slot], 0) == cudaSuccess;
    if (!ok) {
      status = RVQ_ERR_CUDA;
      break;
    }
    status = rvq_reconstruct(dm, tables, x_d, n, n_q, c_d, y_d, scratch, L.scratch_bytes,
                             reinterpret_cast<rvq_stream_t>(p->s_comp));
    if (status != RVQ_OK) break;
    k_fold_status<<<1, 1, 0, p->s_comp>>>(fold, static_cast<const int *>(scratch));
    ok = cudaGetLastError() == cudaSuccess;
    ok = ok && cudaEventRecord(p->ev_comp[slot], p->s_comp) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(p->s_out, p->ev_comp[slot], 0) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(codes_host + n0 * n_q, c_d, (size_t)n * n_q * sizeof(int32_t), cudaMemcpyDeviceToHost,
                               p->s_out) == cudaSuccess;
    if (x_hat_host)
      ok = ok && cudaMemcpyAsync(x_hat_host + n0 * Do, y_d, (size_t)n * Do * sizeof(float),
                                 cudaMemcpyDeviceToHost, p->s_out) == cudaSuccess;
    ok = ok && cudaEventRecord(p->ev_out[slot], p->s_out) == cudaSuccess;
    if (!ok) status = RVQ_ERR_CUDA;
  }
  // the outputs are in host memory when the call returns
  if (cudaStreamSynchronize(p->s_in) != cudaSuccess || cudaStreamSynchronize(p->s_comp) != cudaSuccess ||
      cudaStreamSynchronize(p->s_out) != cudaSuccess) {
    status = RVQ_ERR_CUDA;
  } else if (status == RVQ_OK || status == RVQ_ERR_CANCELLED) {
    // a device failure in any enqueued chunk outranks a cancel
    int word = 0;
    if (cudaMemcpy(&word, fold, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
      status = RVQ_ERR_CUDA;
    else if (word != 0)
      status = rvq::status_from_word(word);
  }
  if (prev >= 0) cudaSetDevice(prev);
  return status;
}

RVQ_API rvq_status rvq_pipeline_set_cancel(rvq_pipeline *p, rvq_cancel_fn fn, void *user) {
  if (!p) return RVQ_ERR_INVALID_ARG;
  p->cancel = fn;
  p->cancel_user = fn ? user : nullptr;
  return RVQ_OK;
}

}  // extern "C"
