// nt_gemv_q4_k.cu -- instantiation of the fused dequantize-GEMV for Q4_K weights.
#include "nt_gemv.cuh"

namespace nt {
cudaError_t launch_gemv_q4_k(const GemvArgs& a, int epi, int threads, int tr, int U, cudaStream_t s, bool pdl,
                             int* grid_used) {
  return launch_gemv_fmt<NT_Q4_K>(a, epi, threads, tr, U, s, pdl, grid_used);
}
}  // namespace nt
