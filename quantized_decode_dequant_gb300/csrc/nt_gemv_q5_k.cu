// nt_gemv_q5_k.cu -- instantiations of the fused dequantize-GEMV for Q5_K weights.
#include "nt_gemv_pipe.cuh"

namespace nt {
cudaError_t launch_gemv_q5_k(const GemvArgs& a, int epi, int R, cudaStream_t s, bool pdl, int* grid_used) {
  return launch_gemv_fmt<NT_Q5_K>(a, epi, R, s, pdl, grid_used);
}
cudaError_t launch_gemv_pipe_q5_k(const GemvArgs& a, int epi, int R, int S, cudaStream_t s, bool pdl,
                                  int* grid_used) {
  return launch_gemv_pipe_fmt<NT_Q5_K>(a, epi, R, S, s, pdl, grid_used);
}
cudaError_t launch_gemv_pipe_q5_k_batch(const GemvArgs& a, int epi, int R, int S, const GemvBatch& b,
                                        cudaStream_t s, bool pdl) {
  return launch_gemv_batch_fmt<NT_Q5_K>(a, epi, R, S, b, s, pdl);
}
}  // namespace nt
