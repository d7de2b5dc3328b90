// nt_gemv.cu -- launch-shape selection for the fused dequantize-GEMV and the
// nt_gemv_q entry point.
#include "nt_gemv.cuh"

namespace nt {

int64_t gemv_logical_rows(const GemvArgs& a) {
  int64_t n = 0;
  for (int i = 0; i < a.nseg; i++) n += a.seg[i].rows;
  return n;
}

cudaError_t launch_gemv(const GemvArgs& a, int epi, cudaStream_t s, bool pdl, int* grid_used) {
  const int64_t cols = a.seg[0].cols;
  if (cols <= 0 || cols % 32 || a.nseg < 1 || a.nseg > 3) return cudaErrorInvalidValue;
  for (int i = 1; i < a.nseg; i++)
    if (a.seg[i].type != a.seg[0].type || a.seg[i].cols != cols) return cudaErrorInvalidValue;
  const int U = gemv_units_per_thread(cols);
  const int tr = gemv_tr(cols, U);
  if (tr > gemv_max_threads(U)) return cudaErrorInvalidValue;
  int groups = gemv_max_threads(U) / tr;
  if (groups < 1) groups = 1;
  const int threads = tr * groups;
  switch (a.seg[0].type) {
    case NT_Q8_0: return launch_gemv_q8_0(a, epi, threads, tr, U, s, pdl, grid_used);
    case NT_Q4_0: return launch_gemv_q4_0(a, epi, threads, tr, U, s, pdl, grid_used);
    case NT_Q4_K: return launch_gemv_q4_k(a, epi, threads, tr, U, s, pdl, grid_used);
    case NT_Q6_K: return launch_gemv_q6_k(a, epi, threads, tr, U, s, pdl, grid_used);
  }
  return cudaErrorInvalidValue;
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
  cudaError_t e = launch_gemv(a, EPI_STORE, static_cast<cudaStream_t>(stream), false, nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "nt_gemv_q");
  return NT_OK;
}
