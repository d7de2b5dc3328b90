// nt_step_q4_k_m.cu -- the step kernel for the Q4_K_M mix (Q4_K with attn_v,
// ffn_down and the output head in Q6_K), 128-dim heads, eight query heads per
// kv head (Llama-3.1-70B shape).
#include "nt_step.cuh"

namespace nt {

cudaError_t launch_step_q4_k_m_g8(const StepArgs& a, size_t smem, cudaStream_t s) {
  return launch_step_t<NT_Q4_K, NT_Q6_K, NT_Q4_K, NT_Q4_K, NT_Q6_K, NT_Q6_K, 128, 8>(a, smem, s);
}
cudaError_t step_fits_q4_k_m_g8(size_t smem, bool* ok) {
  return step_fits_t<NT_Q4_K, NT_Q6_K, NT_Q4_K, NT_Q4_K, NT_Q6_K, NT_Q6_K, 128, 8>(smem, ok);
}

}  // namespace nt
