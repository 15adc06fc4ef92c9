// Plain float64 CPU oracle for residual vector quantisation (RVQ).
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg may load this code.  It shares no source with
// the CUDA path and the CUDA path never calls it.
//
// What it computes follows omnivoice.cpp ARCHITECTURE.md, section "RVQ codec":
//
//   Encode (residual loop), per frame, for stage k = 0 .. n_q-1:
//     e_k        = project_in[k](residual)              (W_in[k] residual + b_in[k])
//     codes_k    = argmin_i || e_k - codebook[k].embed[i] ||^2
//     quantized  = project_out[k](codebook[k].embed[codes_k])
//     residual  -= quantized
//
//   Decode graph, per stage k, accumulated:
//     acc += project_out_w[k] . embed[k][codes_k] + project_out_b[k]
//
// with the PyTorch (out, in) weight layouts of that section's tensor table:
//   w_in [Q][d][D], b_in [Q][d], codebook [Q][K][d], w_out [Q][D][d], b_out [Q][D].
// Frames x are [N][D] and codes are frame-major [N][n_q] (moss-tts.cpp
// AGENTS.md, gotcha 8).  Using the first n_q of Q stages is the bitrate
// control of moss-tts.cpp AGENTS.md, gotcha 12.
//
// Readings where omnivoice.cpp ARCHITECTURE.md and moss-tts.cpp AGENTS.md are silent:
//   * ties in the argmin go to the lowest index (strict '<' in an ascending scan);
//   * biases are optional (a null pointer means zero);
//   * distances are taken in direct form, sum_j (e_j - c_j)^2, in float64;
//   * the per-stage relative gap (d2 - d1) / d2 between the best and the
//     second-best distance is reported (0 when d2 == 0), so that a comparison
//     can tell near-ties from clear decisions;
//   * decode codes outside [0, K) contribute nothing and are counted.
//
// Optional Linear layers around the quantizer (omnivoice.cpp ARCHITECTURE.md,
// "Audio tokenizer" data flow and tensor table): fc (D_in -> D) maps the frame
// to the quantizer's input before the residual loop, fc2 (D -> D_out) maps the
// decoded sum afterwards; both are weight [out][in] plus bias, in float64.
//
// The normalised metric (metric 1) is the quantizer of moss-tts.cpp AGENTS.md,
// gotcha 9: both the projected encoding and every codeword are L2-normalised,
// v / max(||v||_2, 1e-12), before the argmin; decode stays gather + sum, so
// the residual update and the decode use the stored codeword itself (the
// "no extra scaling" of that gotcha is read this way).
//
// All arithmetic is float64 (inputs are float32 and widen exactly).  Frames
// are independent; threads split the frames into contiguous chunks and each
// frame's arithmetic order is fixed, so the result does not depend on the
// thread count.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

struct Weights {
  int D, d, K, Q;
  const float *w_in, *b_in, *codebook, *w_out, *b_out;
};

template <class F>
void parallel_frames(int64_t N, int threads, F &&body) {
  if (threads <= 0) threads = (int)std::max(1u, std::thread::hardware_concurrency());
  if (N < 64 || threads == 1) {
    body(int64_t(0), N);
    return;
  }
  int64_t t = std::min<int64_t>(threads, N);
  std::vector<std::thread> pool;
  pool.reserve((size_t)t);
  for (int64_t i = 0; i < t; ++i) {
    int64_t lo = N * i / t, hi = N * (i + 1) / t;
    pool.emplace_back([&body, lo, hi] { body(lo, hi); });
  }
  for (auto &th : pool) th.join();
}

// One frame of the residual loop.  residual holds x on entry (float64) and
// the final residual on exit.
constexpr double kNormEps = 1e-12;

// v / max(||v||_2, 1e-12), in place.
void l2_normalise(std::vector<double> &v) {
  double ss = 0.0;
  for (double t : v) ss += t * t;
  const double n = std::max(std::sqrt(ss), kNormEps);
  for (double &t : v) t /= n;
}

void encode_frame(const Weights &W, int n_q, int metric, std::vector<double> &residual, std::vector<double> &e,
                  std::vector<double> &c_n, int32_t *codes, double *gap, double *best_dist) {
  const int D = W.D, d = W.d, K = W.K;
  for (int k = 0; k < n_q; ++k) {
    // e_k = project_in[k](residual)
    const float *Win = W.w_in + (size_t)k * d * D;
    for (int j = 0; j < d; ++j) {
      double s = 0.0;
      const float *row = Win + (size_t)j * D;
      for (int i = 0; i < D; ++i) s += (double)row[i] * residual[i];
      if (W.b_in) s += (double)W.b_in[(size_t)k * d + j];
      e[j] = s;
    }
    // codes_k = argmin_i || e_k - embed[i] ||^2, lowest index on ties
    // (metric 1: both sides L2-normalised first)
    if (metric == 1) l2_normalise(e);
    const float *embed = W.codebook + (size_t)k * K * d;
    int best = -1;
    double d1 = std::numeric_limits<double>::infinity();
    double d2 = std::numeric_limits<double>::infinity();
    for (int i = 0; i < K; ++i) {
      const float *c = embed + (size_t)i * d;
      for (int j = 0; j < d; ++j) c_n[j] = (double)c[j];
      if (metric == 1) l2_normalise(c_n);
      double dist = 0.0;
      for (int j = 0; j < d; ++j) {
        double t = e[j] - c_n[j];
        dist += t * t;
      }
      if (dist < d1) {
        d2 = d1;
        d1 = dist;
        best = i;
      } else if (dist < d2) {
        d2 = dist;
      }
    }
    codes[k] = best;
    if (gap) gap[k] = (d2 > 0.0) ? (d2 - d1) / d2 : 0.0;
    if (best_dist) best_dist[k] = d1;
    // quantized = project_out[k](embed[codes_k]); residual -= quantized
    const float *Wout = W.w_out + (size_t)k * D * d;
    const float *c = embed + (size_t)best * d;
    for (int i = 0; i < D; ++i) {
      double s = 0.0;
      const float *row = Wout + (size_t)i * d;
      for (int j = 0; j < d; ++j) s += (double)row[j] * (double)c[j];
      if (W.b_out) s += (double)W.b_out[(size_t)k * D + i];
      residual[i] -= s;
    }
  }
}

}  // namespace

extern "C" {

// Encode N frames [N][D_in] with the first n_q stages; with fc_w, the frame is
// first mapped by fc (fc_w [D][D_in], fc_b [D] nullable), otherwise D_in == D.
//   metric    0: squared L2; 1: squared L2 between L2-normalised vectors
//   codes     [N][n_q] int32   (required)
//   gap       [N][n_q] float64 relative gap (d2-d1)/d2 per stage (nullable)
//   best_dist [N][n_q] float64 best squared distance per stage (nullable)
//   residual  [N][D]   float64 final residual (nullable)
// Returns 0 on success, -1 on a bad argument.
int rvq_oracle_encode_ex(int D_in, int D, int d, int K, int Q, const float *w_in, const float *b_in,
                         const float *codebook, const float *w_out, const float *b_out, const float *fc_w,
                         const float *fc_b, const float *x, int64_t N, int n_q, int32_t *codes, double *gap,
                         double *best_dist, double *residual, int metric, int threads) {
  if (D <= 0 || d <= 0 || K <= 0 || Q <= 0 || N < 0 || n_q < 1 || n_q > Q) return -1;
  if (metric != 0 && metric != 1) return -1;
  if (D_in <= 0 || (!fc_w && D_in != D)) return -1;
  if (!w_in || !codebook || !w_out || (!x && N > 0) || (!codes && N > 0)) return -1;
  Weights W{D, d, K, Q, w_in, b_in, codebook, w_out, b_out};
  parallel_frames(N, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> r((size_t)D), e((size_t)d), c_n((size_t)d);
    for (int64_t n = lo; n < hi; ++n) {
      const float *xn = x + (size_t)n * D_in;
      if (fc_w) {
        // residual = fc(x) = fc_w . x + fc_b
        for (int i = 0; i < D; ++i) {
          double s = 0.0;
          const float *row = fc_w + (size_t)i * D_in;
          for (int j = 0; j < D_in; ++j) s += (double)row[j] * (double)xn[j];
          if (fc_b) s += (double)fc_b[i];
          r[i] = s;
        }
      } else {
        for (int i = 0; i < D; ++i) r[i] = (double)xn[i];
      }
      encode_frame(W, n_q, metric, r, e, c_n, codes + (size_t)n * n_q, gap ? gap + (size_t)n * n_q : nullptr,
                   best_dist ? best_dist + (size_t)n * n_q : nullptr);
      if (residual)
        for (int i = 0; i < D; ++i) residual[(size_t)n * D + i] = r[i];
    }
  });
  return 0;
}

// Without fc.
int rvq_oracle_encode_metric(int D, int d, int K, int Q, const float *w_in, const float *b_in,
                             const float *codebook, const float *w_out, const float *b_out,
                             const float *x, int64_t N, int n_q, int32_t *codes, double *gap,
                             double *best_dist, double *residual, int metric, int threads) {
  return rvq_oracle_encode_ex(D, D, d, K, Q, w_in, b_in, codebook, w_out, b_out, nullptr, nullptr, x, N, n_q,
                              codes, gap, best_dist, residual, metric, threads);
}

// Squared-L2 encode (metric 0), without fc.
int rvq_oracle_encode(int D, int d, int K, int Q, const float *w_in, const float *b_in,
                      const float *codebook, const float *w_out, const float *b_out,
                      const float *x, int64_t N, int n_q, int32_t *codes, double *gap,
                      double *best_dist, double *residual, int threads) {
  return rvq_oracle_encode_metric(D, d, K, Q, w_in, b_in, codebook, w_out, b_out, x, N, n_q, codes, gap,
                                  best_dist, residual, 0, threads);
}

// Decode N frames of codes [N][n_q] into y [N][D_out] float64:
//   s[n] = sum_{k < n_q} ( w_out[k] . codebook[k][codes[n][k]] + b_out[k] ),
//   y[n] = fc2_w . s[n] + fc2_b  (fc2_w [D_out][D], fc2_b nullable)  or  s[n] (D_out == D).
// A code outside [0, K) contributes nothing and is counted in *n_bad.
int rvq_oracle_decode_ex(int D, int D_out, int d, int K, int Q, const float *codebook, const float *w_out,
                         const float *b_out, const float *fc2_w, const float *fc2_b, const int32_t *codes,
                         int64_t N, int n_q, double *y, int64_t *n_bad, int threads) {
  if (D <= 0 || d <= 0 || K <= 0 || Q <= 0 || N < 0 || n_q < 1 || n_q > Q) return -1;
  if (D_out <= 0 || (!fc2_w && D_out != D)) return -1;
  if (!codebook || !w_out || (!codes && N > 0) || (!y && N > 0)) return -1;
  std::vector<int64_t> bad_per_frame((size_t)std::max<int64_t>(N, 1), 0);
  parallel_frames(N, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> sum((size_t)D);
    for (int64_t n = lo; n < hi; ++n) {
      double *acc = fc2_w ? sum.data() : y + (size_t)n * D;
      for (int i = 0; i < D; ++i) acc[i] = 0.0;
      for (int k = 0; k < n_q; ++k) {
        int32_t code = codes[(size_t)n * n_q + k];
        if (code < 0 || code >= K) {
          bad_per_frame[(size_t)n] += 1;
          continue;
        }
        const float *e = codebook + ((size_t)k * K + code) * d;
        const float *Wout = w_out + (size_t)k * D * d;
        for (int i = 0; i < D; ++i) {
          double s = 0.0;
          const float *row = Wout + (size_t)i * d;
          for (int j = 0; j < d; ++j) s += (double)row[j] * (double)e[j];
          if (b_out) s += (double)b_out[(size_t)k * D + i];
          acc[i] += s;
        }
      }
      if (fc2_w) {
        // y = fc2(s) = fc2_w . s + fc2_b
        double *out = y + (size_t)n * D_out;
        for (int i = 0; i < D_out; ++i) {
          double t = 0.0;
          const float *row = fc2_w + (size_t)i * D;
          for (int j = 0; j < D; ++j) t += (double)row[j] * acc[j];
          if (fc2_b) t += (double)fc2_b[i];
          out[i] = t;
        }
      }
    }
  });
  if (n_bad) {
    int64_t total = 0;
    for (int64_t n = 0; n < N; ++n) total += bad_per_frame[(size_t)n];
    *n_bad = total;
  }
  return 0;
}

// Without fc2.
int rvq_oracle_decode(int D, int d, int K, int Q, const float *codebook, const float *w_out,
                      const float *b_out, const int32_t *codes, int64_t N, int n_q, double *y,
                      int64_t *n_bad, int threads) {
  return rvq_oracle_decode_ex(D, D, d, K, Q, codebook, w_out, b_out, nullptr, nullptr, codes, N, n_q, y, n_bad,
                              threads);
}

const char *rvq_oracle_version(void) { return "rvq-oracle f64 3"; }

}  // extern "C"
