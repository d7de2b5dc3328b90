// nt_gemv.cu -- launch-shape selection for the fused dequantize-GEMV and the
// nt_gemv_q entry point.
#include "nt_gemv_pipe.cuh"

namespace nt {

int64_t gemv_logical_rows(const GemvArgs& a) {
  int64_t n = 0;
  for (int i = 0; i < a.nseg; i++) n += a.seg[i].rows;
  return n;
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
  // The shared-memory pipeline takes whole 1024-column tiles: one 16-warp CTA
  // per SM, x staged once per CTA, the ring as deep as fits beside it (rounded
  // down to the instantiated depths).  4-bit formats with at least 8192 rows take
  // four rows per warp, so each x read serves four rows: measured on GB300, those
  // GEMVs are bound by decode instructions per byte, and sharing x cuts them.
  if (cols % 1024 == 0) {
    const size_t xb = pipe_x_bytes(cols, epi);
    const size_t ring = xb < size_t(kPipeMaxSmem) ? size_t(kPipeMaxSmem) - xb : 0;
    const size_t row_tile = size_t(kPipeWarps) * pipe_row_bytes(fmt);
    const bool four_bit = fmt == NT_Q4_0 || fmt == NT_Q4_K || fmt == NT_Q5_K;
    int R = 2, S = int(ring / (2 * row_tile));
    if (four_bit && nrows >= 8192 && ring / (4 * row_tile) >= 3) {
      R = 4;
      S = int(ring / (4 * row_tile));
    }
    if (S >= 3) {
      switch (fmt) {
        case NT_Q8_0: return launch_gemv_pipe_q8_0(a, epi, R, S, s, pdl, grid_used);
        case NT_Q4_0: return launch_gemv_pipe_q4_0(a, epi, R, S, s, pdl, grid_used);
        case NT_Q4_K: return launch_gemv_pipe_q4_k(a, epi, R, S, s, pdl, grid_used);
        case NT_Q6_K: return launch_gemv_pipe_q6_k(a, epi, R, S, s, pdl, grid_used);
        case NT_Q5_K: return launch_gemv_pipe_q5_k(a, epi, R, S, s, pdl, grid_used);
      }
      return cudaErrorInvalidValue;
    }
  }
  // other widths: the register-path kernel (fp32 decode of the same formats)
  const int R = nrows >= 8192 ? 4 : 2;
  switch (fmt) {
    case NT_Q8_0: return launch_gemv_q8_0(a, epi, R, s, pdl, grid_used);
    case NT_Q4_0: return launch_gemv_q4_0(a, epi, R, s, pdl, grid_used);
    case NT_Q4_K: return launch_gemv_q4_k(a, epi, R, s, pdl, grid_used);
    case NT_Q6_K: return launch_gemv_q6_k(a, epi, R, s, pdl, grid_used);
    case NT_Q5_K: return launch_gemv_q5_k(a, epi, R, s, pdl, grid_used);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemv_pair(const GemvArgs& a1_in, const GemvArgs& a2_in, int epi, cudaStream_t s, bool pdl,
                             int* launches) {
  const int64_t cols = a1_in.seg[0].cols;
  bool pair = epi == EPI_QKV && a1_in.seg[0].type == NT_Q4_K && a2_in.seg[0].type == NT_Q6_K &&
              a2_in.seg[0].cols == cols && cols % 1024 == 0 && pipe_x_bytes(cols, EPI_QKV) <= 56 * 1024;
  for (int i = 1; i < a1_in.nseg; i++) pair = pair && a1_in.seg[i].type == NT_Q4_K && a1_in.seg[i].cols == cols;
  pair = pair && a2_in.nseg == 1 && !a1_in.interleave && !a2_in.interleave;
  if (pair) {
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

extern "C" nt_status nt_gemv_q(const nt_qtensor* t, const float* dev_x, float* dev_y, void* stream) {
  if (!t || !dev_x || !dev_y) return fail(NT_E_INVAL, "nt_gemv_q: NULL argument");
  if (t->on_host) return fail(NT_E_STATE, "nt_gemv_q: tensor lives in host memory (streamed layer)");
  if ((reinterpret_cast<uintptr_t>(dev_x) | reinterpret_cast<uintptr_t>(dev_y)) & 15)
    return fail(NT_E_INVAL, "nt_gemv_q: x and y must be 16-byte aligned");
  if (t->m.cols > 32768) return fail(NT_E_UNSUPPORTED, "nt_gemv_q: more than 32768 columns");
  const char* xb = reinterpret_cast<const char*>(dev_x);
  const char* yb = reinterpret_cast<const char*>(dev_y);
  if (xb < yb + t->m.rows * 4 && yb < xb + t->m.cols * 4) return fail(NT_E_INVAL, "nt_gemv_q: x and y overlap");
  GemvArgs a;
  a.seg[0] = t->m;
  a.nseg = 1;
  a.x = dev_x;
  a.epi.y = dev_y;
  // programmatic dependent launch: the kernel reads only the (never rewritten)
  // weight codes before waiting for the previous kernel in the stream to finish
  cudaError_t e = launch_gemv(a, EPI_STORE, static_cast<cudaStream_t>(stream), true, nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "nt_gemv_q");
  return NT_OK;
}
