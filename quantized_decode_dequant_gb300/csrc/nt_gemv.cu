// nt_gemv.cu -- launch-shape selection for the fused dequantize-GEMV and the
// nt_gemv_q entry point.
#include <cstdlib>

#include "nt_gemv_pipe.cuh"

namespace nt {

int64_t gemv_logical_rows(const GemvArgs& a) {
  int64_t n = 0;
  for (int i = 0; i < a.nseg; i++) n += a.seg[i].rows;
  return n;
}

// CTAs per SM the 8-warp layout is sized for (its x staging and ring split the
// SM's shared memory evenly); NT_GEMV_CTAS_PER_SM (1..4) overrides.
static int pipe_ctas_per_sm() {
  static const int v = [] {
    const char* e = getenv("NT_GEMV_CTAS_PER_SM");
    const int n = e ? atoi(e) : 2;
    return n >= 1 && n <= 4 ? n : 2;
  }();
  return v;
}

// Warps per CTA for 4-bit formats with four rows per warp: 16 (one CTA per SM,
// measured slightly faster on GB300) unless NT_GEMV_R4_WARPS=8.
static int pipe_r4_warps() {
  static const int v = [] {
    const char* e = getenv("NT_GEMV_R4_WARPS");
    return e && atoi(e) == 8 ? 8 : 16;
  }();
  return v;
}

// Layout of the pipeline: 0 automatic, 8 (8-warp CTAs) or 16 (one 16-warp CTA
// per SM), from NT_GEMV_WARPS.
static int pipe_layout() {
  static const int v = [] {
    const char* e = getenv("NT_GEMV_WARPS");
    const int n = e ? atoi(e) : 0;
    return n == 8 || n == 16 ? n : 0;
  }();
  return v;
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
  int R = nrows >= 8192 ? 4 : 2;   // four rows per warp for tall 4-bit matrices (measured from 8192 rows)
  const int64_t align = 1024;   // whole 32-unit tiles for the pipeline
  static const bool force_register_path = getenv("NT_GEMV_REGISTER_PATH") != nullptr;
  if (cols % align == 0 && !force_register_path) {
    int parts = 1;
    if (epi == EPI_STORE || epi == EPI_ADD)
      while (pipe_x_bytes(cols / parts, epi) > 140 * 1024 && (cols / parts) % (2 * align) == 0) parts *= 2;
    const int64_t w = cols / parts;
    const size_t xb = pipe_x_bytes(w, epi);
    const size_t target = size_t(kPipeSmPerSm) / size_t(pipe_ctas_per_sm()) - 2048;
    // four rows per warp share each x read, but only if the ring still holds at least
    // four stages (three tiles in flight)
    if (R == 4 && xb < target && (target - xb) / (size_t(8) * 4 * pipe_row_bytes(fmt)) < 4) R = 2;
    const size_t ring_stage = size_t(8) * R * pipe_row_bytes(fmt);
    // ring depth: what fits beside x at the chosen CTAs per SM, else in a whole SM
    size_t budget = xb < target ? target - xb : 0;
    int S = int(budget / ring_stage);
    if (S < 2) {
      budget = xb < size_t(kPipeMaxSmem) ? size_t(kPipeMaxSmem) - xb : 0;
      S = int(budget / ring_stage);
    }
    // rounded down to the instantiated depths (see launch_gemv_pipe_fmt)
    if (R == 4) S = S >= 4 ? 4 : S;
    else S = S >= 8 ? 8 : (S >= 6 ? 6 : S);
    // the 16-warp layout stages x once per SM and gives the ring the rest of it
    const size_t ring16 = xb < size_t(kPipeMaxSmem) ? size_t(kPipeMaxSmem) - xb : 0;
    int S16 = int(ring16 / (size_t(16) * 2 * pipe_row_bytes(fmt)));
    S16 = S16 >= 8 ? 8 : (S16 >= 6 ? 6 : (S16 >= 4 ? 4 : S16));
    int S16r4 = int(ring16 / (size_t(16) * 4 * pipe_row_bytes(fmt)));
    S16r4 = S16r4 >= 4 ? 4 : S16r4;
    const bool four_bit_tall = R == 4 && (fmt == NT_Q4_0 || fmt == NT_Q4_K || fmt == NT_Q5_K);
    int NW = 8;
    if (pipe_layout() == 16 && S16 >= 3) {
      NW = 16;
      R = 2;
      S = S16;
    } else if (pipe_layout() == 0 && four_bit_tall && pipe_r4_warps() == 16 && S16r4 >= 3) {
      NW = 16;
      S = S16r4;
    } else if (pipe_layout() == 0 && S16 >= 3 && !four_bit_tall) {
      // measured on GB300: one 16-warp CTA per SM (x staged once, the deeper ring) is
      // faster than two 8-warp CTAs for every shape; 4-bit formats with enough rows
      // keep four rows per warp (each x read shared over four rows)
      NW = 16;
      R = 2;
      S = S16;
    }
    if (S >= 2) {
      for (int p = 0; p < parts; p++) {
        a.col0 = p * w;
        a.ncols = w;
        const int e_p = p == 0 ? epi : EPI_ADD;
        cudaError_t e;
        switch (fmt) {
          case NT_Q8_0: e = launch_gemv_pipe_q8_0(a, e_p, R, S, NW, s, pdl, grid_used); break;
          case NT_Q4_0: e = launch_gemv_pipe_q4_0(a, e_p, R, S, NW, s, pdl, grid_used); break;
          case NT_Q4_K: e = launch_gemv_pipe_q4_k(a, e_p, R, S, NW, s, pdl, grid_used); break;
          case NT_Q6_K: e = launch_gemv_pipe_q6_k(a, e_p, R, S, NW, s, pdl, grid_used); break;
          case NT_Q5_K: e = launch_gemv_pipe_q5_k(a, e_p, R, S, NW, s, pdl, grid_used); break;
          default: e = cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
      }
      return cudaSuccess;
    }
  }
  a.col0 = 0;
  a.ncols = cols;
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
  static const bool force_register_path = getenv("NT_GEMV_REGISTER_PATH") != nullptr;
  const int64_t cols = a1_in.seg[0].cols;
  bool pair = !force_register_path && epi == EPI_QKV && a1_in.seg[0].type == NT_Q4_K && a2_in.seg[0].type == NT_Q6_K &&
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
