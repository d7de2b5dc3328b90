// nt_gemv_q6_k.cu -- instantiation of the fused dequantize-GEMV for Q6_K weights.
#include "nt_gemv.cuh"

namespace nt {
cudaError_t launch_gemv_q6_k(const GemvArgs& a, int epi, int threads, int tr, int U, cudaStream_t s, bool pdl,
                             int* grid_used) {
  return launch_gemv_fmt<NT_Q6_K>(a, epi, threads, tr, U, s, pdl, grid_used);
}
}  // namespace nt
