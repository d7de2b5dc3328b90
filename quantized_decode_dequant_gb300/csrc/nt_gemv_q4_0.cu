// nt_gemv_q4_0.cu -- instantiation of the fused dequantize-GEMV for Q4_0 weights.
#include "nt_gemv.cuh"

namespace nt {
cudaError_t launch_gemv_q4_0(const GemvArgs& a, int epi, int threads, int tr, int U, cudaStream_t s, bool pdl,
                             int* grid_used) {
  return launch_gemv_fmt<NT_Q4_0>(a, epi, threads, tr, U, s, pdl, grid_used);
}
}  // namespace nt
