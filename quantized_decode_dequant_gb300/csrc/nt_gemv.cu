// nt_gemv.cu -- launch-shape selection for the fused dequantize-GEMV and the
// nt_gemv_q entry point.
#include "nt_gemv_pipe.cuh"

namespace nt {

int64_t gemv_logical_rows(const GemvArgs& a) {
  int64_t n = 0;
  for (int i = 0; i < a.nseg; i++) n += a.seg[i].rows;
  return n;
}

// Shape of the shared-memory pipeline for a GEMV (false: it does not take it):
// whole 1024-column tiles, one 16-warp CTA per SM, x staged once per CTA, the
// ring as deep as fits beside it (rounded down to the instantiated depths).
// 4-bit formats with at least 8192 rows take four rows per warp, so each x read
// serves four rows: measured on GB300, those GEMVs are bound by decode
// instructions per byte, and sharing x cuts them.
bool pipe_shape(int fmt, int64_t nrows, int64_t cols, int epi, int& R, int& S) {
  if (cols % 1024) return false;
  const size_t xb = pipe_x_bytes(cols, epi);
  const size_t ring = xb < size_t(kPipeMaxSmem) ? size_t(kPipeMaxSmem) - xb : 0;
  const size_t row_tile = size_t(kPipeWarps) * pipe_row_bytes(fmt);
  const bool four_bit = fmt == NT_Q4_0 || fmt == NT_Q4_K || fmt == NT_Q5_K;
  R = 2;
  S = int(ring / (2 * row_tile));
  if (four_bit && nrows >= 8192 && ring / (4 * row_tile) >= 3) {
    R = 4;
    S = int(ring / (4 * row_tile));
  }
  return S >= 3;
}

cudaError_t launch_gemv(const GemvArgs& a_in, int epi, cudaStream_t s, bool pdl, int* grid_used) {
  GemvArgs a = a_in;
  const int64_t cols = a.seg[0].cols;
  if (cols <= 0 || cols % 32 || cols > 32768 || a.nseg < 1 || a.nseg > 3) return cudaErrorInvalidValue;
  for (int i = 1; i < a.nseg; i++)
    if (a.seg[i].type != a.seg[0].type || a.seg[i].cols != cols) return cudaErrorInvalidValue;
  if (a.max_grid <= 0 || a.max_grid > kMaxGemvGrid) a.max_grid = kMaxGemvGrid;
  const int fmt = a.seg[0].type;
  const int64_t nrows = gemv_logical_rows(a);
  a.col0 = 0;
  a.ncols = cols;
  int R = 0, S = 0;
  if (pipe_shape(fmt, nrows, cols, epi, R, S)) {
    switch (fmt) {
      case NT_Q8_0: return launch_gemv_pipe_q8_0(a, epi, R, S, s, pdl, grid_used);
      case NT_Q4_0: return launch_gemv_pipe_q4_0(a, epi, R, S, s, pdl, grid_used);
      case NT_Q4_K: return launch_gemv_pipe_q4_k(a, epi, R, S, s, pdl, grid_used);
      case NT_Q6_K: return launch_gemv_pipe_q6_k(a, epi, R, S, s, pdl, grid_used);
      case NT_Q5_K: return launch_gemv_pipe_q5_k(a, epi, R, S, s, pdl, grid_used);
    }
    return cudaErrorInvalidValue;
  }
  // other widths: the register-path kernel (fp32 decode of the same formats)
  const int Rr = nrows >= 8192 ? 4 : 2;
  switch (fmt) {
    case NT_Q8_0: return launch_gemv_q8_0(a, epi, Rr, s, pdl, grid_used);
    case NT_Q4_0: return launch_gemv_q4_0(a, epi, Rr, s, pdl, grid_used);
    case NT_Q4_K: return launch_gemv_q4_k(a, epi, Rr, s, pdl, grid_used);
    case NT_Q6_K: return launch_gemv_q6_k(a, epi, Rr, s, pdl, grid_used);
    case NT_Q5_K: return launch_gemv_q5_k(a, epi, Rr, s, pdl, grid_used);
  }
  return cudaErrorInvalidValue;
}

// The pipeline GEMV over the column window [col0, col0 + ncols) of a (ncols a
// multiple of 1024, at most 32768): rows of W restricted to the window times
// x[col0, col0 + ncols), through epi.
static cudaError_t launch_gemv_window(const GemvArgs& a_in, int epi, int64_t col0, int64_t ncols, cudaStream_t s,
                                      bool pdl) {
  GemvArgs a = a_in;
  if (ncols <= 0 || ncols % 1024 || ncols > 32768 || col0 < 0 || col0 + ncols > a.seg[0].cols || a.nseg != 1)
    return cudaErrorInvalidValue;
  if (a.max_grid <= 0 || a.max_grid > kMaxGemvGrid) a.max_grid = kMaxGemvGrid;
  a.col0 = col0;
  a.ncols = ncols;
  int R = 0, S = 0;
  const int64_t nrows = gemv_logical_rows(a);
  if (!pipe_shape(a.seg[0].type, nrows, ncols, epi, R, S)) return cudaErrorInvalidValue;
  switch (a.seg[0].type) {
    case NT_Q8_0: return launch_gemv_pipe_q8_0(a, epi, R, S, s, pdl, nullptr);
    case NT_Q4_0: return launch_gemv_pipe_q4_0(a, epi, R, S, s, pdl, nullptr);
    case NT_Q4_K: return launch_gemv_pipe_q4_k(a, epi, R, S, s, pdl, nullptr);
    case NT_Q6_K: return launch_gemv_pipe_q6_k(a, epi, R, S, s, pdl, nullptr);
    case NT_Q5_K: return launch_gemv_pipe_q5_k(a, epi, R, S, s, pdl, nullptr);
  }
  return cudaErrorInvalidValue;
}

// Tokens [0, k) through the GEMV a, each with the arithmetic of its own
// single-token launch (launch_gemv, or the two-format kernel for a pair),
// several tokens per launch where their staged x fit beside a ring of depth 3:
// the weights are then read once per launch instead of once per token.  R: the
// rows per warp of the single-token launch (0: as launch_gemv picks).
cudaError_t launch_gemv_batch(const GemvArgs& a_in, int epi, const BatchTok* toks, int k, int R_single,
                              cudaStream_t s, bool pdl, int* launches) {
  GemvArgs a = a_in;
  const int64_t cols = a.seg[0].cols, nrows = gemv_logical_rows(a);
  const int fmt = a.seg[0].type;
  if (a.max_grid <= 0 || a.max_grid > kMaxGemvGrid) a.max_grid = kMaxGemvGrid;
  a.col0 = 0;
  a.ncols = cols;
  int R = 0, S = 0;
  const bool pipe = pipe_shape(fmt, nrows, cols, epi, R, S);
  if (R_single) R = R_single;
  const size_t xb = pipe_x_bytes(cols, epi), stage3 = size_t(kPipeWarps) * 3 * R * pipe_row_bytes(fmt);
  int kb = 0;   // tokens per launch
  if (pipe && epi != EPI_LOGITS)
    while (kb < kBatchMax && size_t(kb + 1) * xb + stage3 <= size_t(kPipeMaxSmem)) kb++;
  if (launches) *launches = kb < 2 ? k : (k + kb - 1) / kb;
  // (Two-format pairs, R_single != 0, never take the per-token path: their x is
  // at most 56 KB, and two staged x with a depth-3 ring of four Q4_K rows or one
  // Q6_K row per warp fit.)
  if (kb < 2) {   // one token per launch: the single-token kernel itself
    for (int i = 0; i < k; i++) {
      a.x = toks[i].x;
      a.epi.y = toks[i].y;
      a.epi.pos = toks[i].pos;
      cudaError_t e = launch_gemv(a, epi, s, pdl, nullptr);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  for (int i0 = 0; i0 < k; i0 += kb) {
    GemvBatch b;
    b.n = k - i0 < kb ? k - i0 : kb;
    for (int j = 0; j < b.n; j++) b.tok[j] = toks[i0 + j];
    const size_t ring = size_t(kPipeMaxSmem) - size_t(b.n) * xb;
    const int Sb = int(ring / (size_t(kPipeWarps) * R * pipe_row_bytes(fmt)));
    cudaError_t e;
    switch (fmt) {
      case NT_Q8_0: e = launch_gemv_pipe_q8_0_batch(a, epi, R, Sb, b, s, pdl); break;
      case NT_Q4_0: e = launch_gemv_pipe_q4_0_batch(a, epi, R, Sb, b, s, pdl); break;
      case NT_Q4_K: e = launch_gemv_pipe_q4_k_batch(a, epi, R, Sb, b, s, pdl); break;
      case NT_Q6_K: e = launch_gemv_pipe_q6_k_batch(a, epi, R, Sb, b, s, pdl); break;
      case NT_Q5_K: e = launch_gemv_pipe_q5_k_batch(a, epi, R, Sb, b, s, pdl); break;
      default: e = cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Whether launch_gemv_pair takes the two-format kernel for a1 and a2.
static bool pair_kernel(const GemvArgs& a1, const GemvArgs& a2, int epi) {
  const int64_t cols = a1.seg[0].cols;
  bool pair = epi == EPI_QKV && a1.seg[0].type == NT_Q4_K && a2.seg[0].type == NT_Q6_K &&
              a2.seg[0].cols == cols && cols % 1024 == 0 && pipe_x_bytes(cols, EPI_QKV) <= 56 * 1024;
  for (int i = 1; i < a1.nseg; i++) pair = pair && a1.seg[i].type == NT_Q4_K && a1.seg[i].cols == cols;
  return pair && a2.nseg == 1 && !a1.interleave && !a2.interleave;
}

cudaError_t launch_gemv_pair_batch(const GemvArgs& a1, const GemvArgs& a2, int epi, const BatchTok* toks1,
                                   const BatchTok* toks2, int k, cudaStream_t s, bool pdl, int* launches) {
  // the two-format kernel's rows per warp: four for the Q4_K rows, one for the Q6_K rows
  const bool pair = pair_kernel(a1, a2, epi);
  int n1 = 0, n2 = 0;
  cudaError_t e = launch_gemv_batch(a1, epi, toks1, k, pair ? 4 : 0, s, pdl, &n1);
  if (e == cudaSuccess) e = launch_gemv_batch(a2, epi, toks2, k, pair ? 1 : 0, s, pdl, &n2);
  if (launches) *launches = n1 > n2 ? n1 : n2;
  return e;
}

cudaError_t launch_gemv_pair(const GemvArgs& a1_in, const GemvArgs& a2_in, int epi, cudaStream_t s, bool pdl,
                             int* launches) {
  const int64_t cols = a1_in.seg[0].cols;
  if (pair_kernel(a1_in, a2_in, epi)) {
    GemvArgs a1 = a1_in, a2 = a2_in;
    a1.col0 = a2.col0 = 0;
    a1.ncols = a2.ncols = cols;
    if (launches) *launches = 1;
    return launch_gemv_pipe2_q4k_q6k<EPI_QKV>(a1, a2, s, pdl);
  }
  if (launches) *launches = 2;
  cudaError_t e = launch_gemv(a1_in, epi, s, pdl, nullptr);
  if (e == cudaSuccess) e = launch_gemv(a2_in, epi, s, pdl, nullptr);
  return e;
}

}  // namespace nt

using namespace nt;

extern "C" nt_status nt_gemv_q_batch(const nt_qtensor* t, const float* const* dev_x, float* const* dev_y, int32_t k,
                                     int32_t* launches, void* stream) {
  if (!t || !dev_x || !dev_y) return fail(NT_E_INVAL, "nt_gemv_q_batch: NULL argument");
  if (k < 1 || k > 8) return fail(NT_E_INVAL, "nt_gemv_q_batch: k outside [1, 8]");
  if (t->on_host) return fail(NT_E_STATE, "nt_gemv_q_batch: tensor lives in host memory (streamed layer)");
  if (t->m.cols > 32768) return fail(NT_E_UNSUPPORTED, "nt_gemv_q_batch: more than 32768 columns");
  BatchTok toks[8];
  for (int i = 0; i < k; i++) {
    if (!dev_x[i] || !dev_y[i]) return fail(NT_E_INVAL, "nt_gemv_q_batch: NULL vector");
    if ((reinterpret_cast<uintptr_t>(dev_x[i]) | reinterpret_cast<uintptr_t>(dev_y[i])) & 15)
      return fail(NT_E_INVAL, "nt_gemv_q_batch: every x and y must be 16-byte aligned");
    toks[i] = {dev_x[i], dev_y[i], nullptr};
  }
  for (int i = 0; i < k; i++)   // no output may overlap an input or another output
    for (int j = 0; j < k; j++) {
      const char* yb = reinterpret_cast<const char*>(dev_y[i]);
      const char* xb = reinterpret_cast<const char*>(dev_x[j]);
      const char* y2 = reinterpret_cast<const char*>(dev_y[j]);
      if (xb < yb + t->m.rows * 4 && yb < xb + t->m.cols * 4) return fail(NT_E_INVAL, "nt_gemv_q_batch: an x and a y overlap");
      if (i != j && y2 < yb + t->m.rows * 4 && yb < y2 + t->m.rows * 4)
        return fail(NT_E_INVAL, "nt_gemv_q_batch: two y overlap");
    }
  GemvArgs a;
  a.seg[0] = t->m;
  a.nseg = 1;
  int n = 0;
  cudaError_t e = launch_gemv_batch(a, EPI_STORE, toks, k, 0, static_cast<cudaStream_t>(stream), true, &n);
  if (e != cudaSuccess) return cuda_fail(e, "nt_gemv_q_batch");
  if (launches) *launches = n;
  return NT_OK;
}

extern "C" nt_status nt_gemv_q(const nt_qtensor* t, const float* dev_x, float* dev_y, void* stream) {
  if (!t || !dev_x || !dev_y) return fail(NT_E_INVAL, "nt_gemv_q: NULL argument");
  if (t->on_host) return fail(NT_E_STATE, "nt_gemv_q: tensor lives in host memory (streamed layer)");
  if ((reinterpret_cast<uintptr_t>(dev_x) | reinterpret_cast<uintptr_t>(dev_y)) & 15)
    return fail(NT_E_INVAL, "nt_gemv_q: x and y must be 16-byte aligned");
  if (t->m.cols > 32768 && t->m.cols % 1024)
    return fail(NT_E_UNSUPPORTED, "nt_gemv_q: more than 32768 columns, not a multiple of 1024");
  const char* xb = reinterpret_cast<const char*>(dev_x);
  const char* yb = reinterpret_cast<const char*>(dev_y);
  if (xb < yb + t->m.rows * 4 && yb < xb + t->m.cols * 4) return fail(NT_E_INVAL, "nt_gemv_q: x and y overlap");
  GemvArgs a;
  a.seg[0] = t->m;
  a.nseg = 1;
  a.x = dev_x;
  a.epi.y = dev_y;
  if (t->m.cols > 32768) {   // column windows of at most 32768, their products added in window order
    for (int64_t c0 = 0; c0 < t->m.cols; c0 += 32768) {
      const int64_t n = t->m.cols - c0 < 32768 ? t->m.cols - c0 : 32768;
      cudaError_t e = launch_gemv_window(a, c0 == 0 ? EPI_STORE : EPI_ADD, c0, n, static_cast<cudaStream_t>(stream),
                                         true);
      if (e != cudaSuccess) return cuda_fail(e, "nt_gemv_q");
    }
    return NT_OK;
  }
  // programmatic dependent launch: the kernel reads only the (never rewritten)
  // weight codes before waiting for the previous kernel in the stream to finish
  cudaError_t e = launch_gemv(a, EPI_STORE, static_cast<cudaStream_t>(stream), true, nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "nt_gemv_q");
  return NT_OK;
}
