// nt_step.cu -- plan matching and shared-memory sizing of the step kernel.
#include "nt_step.cuh"

namespace nt {

size_t step_smem(const StepPlan& p, int64_t max_cols, int64_t qkv_cols, int attn_chunk, size_t* ring_off) {
  // staged x of the widest GEMV input, or of the Q/K/V input with its three slices
  size_t xb = pipe_x_bytes(max_cols, EPI_ADD);
  if (pipe_x_bytes(qkv_cols, EPI_QKV) > xb) xb = pipe_x_bytes(qkv_cols, EPI_QKV);
  const size_t lo = (xb + 127) & ~size_t(127);
  *ring_off = lo;
  const size_t gemv = lo + kStepRingBytes;
  const size_t attn = attn_item_smem(p.hd, p.G, attn_chunk);
  return gemv > attn ? gemv : attn;
}

static bool is_plan(const StepPlan& p, int qk, int v, int o, int gu, int d, int out, int hd, int G) {
  return p.f_qk == qk && p.f_v == v && p.f_o == o && p.f_gu == gu && p.f_d == d && p.f_out == out && p.hd == hd &&
         p.G == G;
}

cudaError_t launch_step(const StepPlan& p, const StepArgs& a, size_t smem, cudaStream_t s) {
  if (is_plan(p, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, 128, 4))
    return launch_step_q8_0_g4(a, smem, s);
  if (is_plan(p, NT_Q4_K, NT_Q6_K, NT_Q4_K, NT_Q4_K, NT_Q6_K, NT_Q6_K, 128, 8))
    return launch_step_q4_k_m_g8(a, smem, s);
  return cudaErrorNotSupported;
}

cudaError_t step_fits(const StepPlan& p, size_t smem, bool* ok) {
  *ok = false;
  if (is_plan(p, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, NT_Q8_0, 128, 4)) return step_fits_q8_0_g4(smem, ok);
  if (is_plan(p, NT_Q4_K, NT_Q6_K, NT_Q4_K, NT_Q4_K, NT_Q6_K, NT_Q6_K, 128, 8)) return step_fits_q4_k_m_g8(smem, ok);
  return cudaErrorNotSupported;
}

}  // namespace nt
