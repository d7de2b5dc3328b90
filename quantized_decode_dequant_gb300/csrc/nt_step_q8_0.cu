// nt_step_q8_0.cu -- the step kernel for Q8_0 weights throughout, 128-dim heads,
// four query heads per kv head (Llama-3.1-8B shape).
#include "nt_step.cuh"

namespace nt {

cudaError_t launch_step_q8_0_g4(const StepArgs& a, size_t smem, cudaStream_t s) {
  return launch_step_t<NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, 128, 4>(a, smem, s);
}
cudaError_t step_fits_q8_0_g4(size_t smem, bool* ok) {
  return step_fits_t<NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, 128, 4>(smem, ok);
}

}  // namespace nt
