// nt_gemv_pipe.cuh -- the fused dequantize-GEMV with weights staged through a
// per-warp shared-memory ring by asynchronous copies.
//
// Same work split and decode arithmetic as nt_gemv.cuh (warps own groups of R
// rows, lanes own 32-column units, x staged once per CTA), but the codes and
// scales of each (row group, 32-unit column tile) are copied global -> shared
// with cp.async (16-byte LDGSTS, L2-only) S-1 tiles ahead of the one being
// decoded.  Bytes in flight per warp are (S-1) * R * (row tile bytes) with no
// register cost, which is what a bandwidth-bound GEMV needs to cover DRAM
// latency; the only waits are cp.async.wait_group on the warp's own copies
// plus __syncwarp for the scale bytes other lanes copied.
//
// Row tile layout in shared memory (one row, 32 units):
//   Q8_0  32 x 32 B codes | 32 x f16 d                                  1088 B
//   Q4_0  32 x 16 B codes | 32 x f16 d                                   576 B
//   Q4_K  32 x 16 B codes | 4 x 16 B superblock headers                  576 B
//   Q6_K  32 x 16 B low codes | 32 x 8 B high-bit words | 32 x 2 B sc | 4 x f16 d (16 B slot)   848 B
// Requires the window width (and start) to be a multiple of 256 columns (512
// for Q6_K) so every scale piece is a whole number of aligned 16-byte (4-byte
// for Q6_K d) copies.
#pragma once

#include "nt_gemv.cuh"

namespace nt {

constexpr int kPipeWarps = 8;                 // 256 threads per CTA
constexpr int kPipeMaxSmem = 221 * 1024;      // dynamic shared memory a CTA may ask for

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// wait_group takes an immediate; the ring depth is at most 8 (so n <= 6)
__device__ __forceinline__ void cp_wait_dyn(int n) {
  switch (n) {
    case 0: cp_wait<0>(); break;
    case 1: cp_wait<1>(); break;
    case 2: cp_wait<2>(); break;
    case 3: cp_wait<3>(); break;
    case 4: cp_wait<4>(); break;
    case 5: cp_wait<5>(); break;
    default: cp_wait<6>(); break;
  }
}

template <int FMT> struct Pipe;

template <> struct Pipe<NT_Q8_0> {
  static constexpr int RB = 32 * 32 + 64;
  static constexpr bool kXSum = false;
  // e_row: flat element index of the row's first column in the window; u0: first unit of the tile
  __device__ static void issue(const QMat& m, int64_t e_row, int u0, int nu, uint32_t dst, int lane) {
    if (lane < nu) {
      const uint8_t* src = m.q + e_row + int64_t(u0 + lane) * 32;
      cp16(dst + lane * 32, src);
      cp16(dst + lane * 32 + 16, src + 16);
    }
    if (lane < nu / 8)
      cp16(dst + 1024 + lane * 16, reinterpret_cast<const uint8_t*>(m.d + (e_row >> 5) + u0) + lane * 16);
  }
  __device__ static float dot(const uint8_t* blk, int lane, const float4* xs, float) {
    const uint4 c0 = *reinterpret_cast<const uint4*>(blk + lane * 32);
    const uint4 c1 = *reinterpret_cast<const uint4*>(blk + lane * 32 + 16);
    const uint32_t d = *reinterpret_cast<const uint16_t*>(blk + 1024 + lane * 2);
    return h2f_bits(d) * (q8_dot16(c0, xs) + q8_dot16(c1, xs + 4));
  }
  __device__ static int xpos(int c) { return c; }
  __device__ static float xscale(int) { return 1.0f; }
};

template <> struct Pipe<NT_Q4_0> {
  static constexpr int RB = 32 * 16 + 64;
  static constexpr bool kXSum = false;
  __device__ static void issue(const QMat& m, int64_t e_row, int u0, int nu, uint32_t dst, int lane) {
    if (lane < nu) cp16(dst + lane * 16, m.q + ((e_row + int64_t(u0 + lane) * 32) >> 1));
    if (lane < nu / 8)
      cp16(dst + 512 + lane * 16, reinterpret_cast<const uint8_t*>(m.d + (e_row >> 5) + u0) + lane * 16);
  }
  __device__ static float dot(const uint8_t* blk, int lane, const float4* xs, float) {
    Fmt<NT_Q4_0>::Pay p;
    p.c = *reinterpret_cast<const uint4*>(blk + lane * 16);
    p.d = *reinterpret_cast<const uint16_t*>(blk + 512 + lane * 2);
    return Fmt<NT_Q4_0>::dot(p, xs, 0.f);
  }
  __device__ static int xpos(int c) { return c; }
  __device__ static float xscale(int c) { return nib_xscale(c); }
};

template <> struct Pipe<NT_Q4_K> {
  static constexpr int RB = 32 * 16 + 64;
  static constexpr bool kXSum = true;
  __device__ static void issue(const QMat& m, int64_t e_row, int u0, int nu, uint32_t dst, int lane) {
    if (lane < nu) cp16(dst + lane * 16, m.q + ((e_row + int64_t(u0 + lane) * 32) >> 1));
    if (lane < nu / 8) cp16(dst + 512 + lane * 16, m.meta + ((e_row >> 8) + u0 / 8 + lane) * 16);
  }
  __device__ static float dot(const uint8_t* blk, int lane, const float4* xs, float xsum) {
    Fmt<NT_Q4_K>::Pay p;
    p.c = *reinterpret_cast<const uint4*>(blk + lane * 16);
    p.meta = *reinterpret_cast<const uint4*>(blk + 512 + (lane >> 3) * 16);
    p.j = lane & 7;
    return Fmt<NT_Q4_K>::dot(p, xs, xsum);
  }
  __device__ static int xpos(int c) { return c; }
  __device__ static float xscale(int c) { return nib_xscale(c); }
};

template <> struct Pipe<NT_Q6_K> {
  static constexpr int RB = 32 * 16 + 256 + 64 + 16;
  static constexpr bool kXSum = false;
  __device__ static void issue(const QMat& m, int64_t e_row, int u0, int nu, uint32_t dst, int lane) {
    const int64_t e0 = e_row + int64_t(u0) * 32;   // first element of the tile
    if (lane < nu) cp16(dst + lane * 16, m.q + ((e0 + int64_t(lane) * 32) >> 1));
    if (lane < nu / 2) cp16(dst + 512 + lane * 16, m.qh + (e0 >> 2) + lane * 16);
    if (lane < nu / 8) cp16(dst + 768 + lane * 16, m.meta + (e0 >> 4) + lane * 16);
    if (lane < nu / 16) cp4(dst + 832 + lane * 4, reinterpret_cast<const uint8_t*>(m.d + (e0 >> 8)) + lane * 4);
  }
  __device__ static float dot(const uint8_t* blk, int lane, const float4* xs, float) {
    Fmt<NT_Q6_K>::Pay p;
    p.c = *reinterpret_cast<const uint4*>(blk + lane * 16);
    p.h = *reinterpret_cast<const uint2*>(blk + 512 + lane * 8);
    p.sc = *reinterpret_cast<const uint16_t*>(blk + 768 + lane * 2);
    p.d = *reinterpret_cast<const uint16_t*>(blk + 832 + (lane >> 3) * 2);
    return Fmt<NT_Q6_K>::dot(p, xs, 0.f);
  }
  __device__ static int xpos(int c) { return Fmt<NT_Q6_K>::xpos(c); }
  __device__ static float xscale(int) { return 1.0f; }
};

// Rows of one group as seen by the copy issuer.
template <int R>
struct GroupRows {
  int seg[R];
  int64_t e[R];
  bool live[R];
};

template <int R>
__device__ __forceinline__ void rows_setup(const GemvArgs& a, int64_t grp, int64_t nrows, GroupRows<R>& g) {
#pragma unroll
  for (int r = 0; r < R; r++) {
    const int64_t row = grp * R + r;
    g.live[r] = row < nrows;
    int s = 0;
    int64_t lr = 0;
    if (g.live[r]) map_row(a, row, s, lr);
    g.seg[r] = s;
    g.e[r] = lr * a.seg[0].cols + a.col0;
  }
}

template <int FMT, int R, int EPI>
__global__ void __launch_bounds__(kPipeWarps * 32) k_gemv_pipe(const __grid_constant__ GemvArgs a,
                                                              const int64_t nrows, const int S) {
  using P = Pipe<FMT>;
  constexpr int US = 32 + kXPad;                  // x floats per unit in shared memory
  constexpr int nw = kPipeWarps;
  extern __shared__ float4 smem4[];
  const int64_t cols = a.ncols;                   // window width
  const int units = int(cols / 32);
  float* xsh = reinterpret_cast<float*>(smem4);
  float* xsum = xsh + units * US;
  uint8_t* ring = reinterpret_cast<uint8_t*>(xsum + ((units + 3) & ~3));
  __shared__ float s_red[kPipeWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ngroups = (nrows + R - 1) / R;
  const int64_t stride = int64_t(gridDim.x) * nw;
  const int kiters = (units + 31) / 32;
  uint8_t* wring = ring + size_t(warp) * S * R * P::RB;
  const uint32_t wring_s = smem_addr(wring);

  // tile t of this warp = (its k-th row group, column tile it), t = k * kiters + it
  const int64_t g0 = int64_t(blockIdx.x) * nw + warp;
  const int64_t my_groups = g0 < ngroups ? (ngroups - 1 - g0) / stride + 1 : 0;
  const int64_t ntiles = my_groups * kiters;

  // copy issuer state (runs S-1 tiles ahead)
  int64_t t_issue = 0;
  GroupRows<R> ig;
  auto issue_tile = [&](int64_t t) {
    if (t < ntiles) {
      const int64_t k = t / kiters;
      const int it = int(t - k * kiters);
      if (it == 0) rows_setup<R>(a, g0 + k * stride, nrows, ig);
      const int u0 = it * 32;
      const int nu = min(32, units - u0);
      const uint32_t dst = wring_s + uint32_t((t % S) * R * P::RB);
#pragma unroll
      for (int r = 0; r < R; r++)
        if (ig.live[r]) P::issue(a.seg[ig.seg[r]], ig.e[r], u0, nu, dst + r * P::RB, lane);
    }
    cp_commit();   // one group per tile, empty past the end, so the wait_group counts stay aligned
  };

  // prologue: the first S-1 tiles before waiting for the producer of x
  for (; t_issue < S - 1; t_issue++) issue_tile(t_issue);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- stage x ---------------------------------------------------------------
  {
    const float* xg = a.x + a.col0;
    float ss = 0.f;
    for (int c = tid; c < cols; c += blockDim.x) {
      const float v = xg[c];
      ss += v * v;
      xsh[(c >> 5) * US + P::xpos(c & 31)] = v;
    }
    float scale = 1.0f;
    if (a.norm) {
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_red[warp] = ss;
      __syncthreads();
      float t = 0.f;
      for (int w = 0; w < nw; w++) t += s_red[w];
      scale = rsqrtf(t / float(cols) + a.eps);
    }
    __syncthreads();
    if (a.norm || P::kXSum || FMT != NT_Q8_0) {
      for (int u = warp; u < units; u += nw) {
        const int p = u * US + P::xpos(lane);
        float v = xsh[p] * scale;
        xsh[p] = v * P::xscale(lane);
        if (P::kXSum) {
#pragma unroll
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) xsum[u] = v;
        }
      }
      __syncthreads();
    }
  }

  float best = -INFINITY, second = -INFINITY;
  int best_i = 0x7fffffff;
  float acc[R];
#pragma unroll
  for (int r = 0; r < R; r++) acc[r] = 0.f;

  for (int64_t t = 0; t < ntiles; t++) {
    cp_wait_dyn(S - 2);   // this lane's copies of tile t have landed
    __syncwarp();         // ... and every lane's (scales are copied by a few lanes); slot t-1 is free
    issue_tile(t_issue++);
    const int64_t k = t / kiters;
    const int it = int(t - k * kiters);
    const int64_t grp = g0 + k * stride;
    const int u = it * 32 + lane;
    if (u < units) {
      const uint8_t* blk = wring + (t % S) * R * P::RB;
      const float4* xs = reinterpret_cast<const float4*>(xsh + u * US);
      const float xu = P::kXSum ? xsum[u] : 0.f;
#pragma unroll
      for (int r = 0; r < R; r++)
        if (grp * R + r < nrows) acc[r] += P::dot(blk + r * P::RB, lane, xs, xu);
    }
    if (it != kiters - 1) continue;
    const float kk = warp_reduce_rows<R>(acc, lane);
#pragma unroll
    for (int r = 0; r < R; r++) acc[r] = 0.f;
    epilogue<R, EPI>(a, grp, nrows, lane, kk, best, best_i, second);
  }
  cp_wait<0>();

  asm volatile("griddepcontrol.launch_dependents;");
  if (EPI == EPI_LOGITS) cta_top2<kPipeWarps>(a, best, best_i, second);
}

inline size_t pipe_x_bytes(int64_t cols) {
  const int64_t units = cols / 32;
  return size_t(units) * (32 + kXPad) * 4 + size_t((units + 3) & ~3) * 4;
}
inline int pipe_row_bytes(int fmt) {
  switch (fmt) {
    case NT_Q8_0: return Pipe<NT_Q8_0>::RB;
    case NT_Q4_0: return Pipe<NT_Q4_0>::RB;
    case NT_Q4_K: return Pipe<NT_Q4_K>::RB;
    default: return Pipe<NT_Q6_K>::RB;
  }
}

template <int FMT, int R, int EPI>
cudaError_t launch_gemv_pipe_t(const GemvArgs& a, int S, cudaStream_t s, bool pdl, int* grid_used) {
  const int64_t nrows = gemv_logical_rows(a);
  const size_t smem = pipe_x_bytes(a.ncols) + size_t(kPipeWarps) * S * R * Pipe<FMT>::RB;
  if (smem > size_t(kPipeMaxSmem)) return cudaErrorInvalidValue;
  auto kern = k_gemv_pipe<FMT, R, EPI>;
  static int s_sms = 0;
  static size_t s_occ_smem = ~size_t(0);
  static int s_occ = 0;
  if (!s_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&s_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPipeMaxSmem);
    if (e != cudaSuccess) return e;
  }
  if (s_occ_smem != smem) {
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kPipeWarps * 32, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    s_occ = occ;
    s_occ_smem = smem;
  }
  const int64_t grid = one_wave_grid(s_sms, s_occ, (nrows + R - 1) / R, kPipeWarps, a.max_grid);
  if (grid_used) *grid_used = int(grid);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(kPipeWarps * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, nrows, S);
}

template <int FMT>
cudaError_t launch_gemv_pipe_fmt(const GemvArgs& a, int epi, int R, int S, cudaStream_t s, bool pdl,
                                 int* grid_used) {
#define NT_EPI_CASES(RR)                                                                       \
  switch (epi) {                                                                               \
    case EPI_STORE: return launch_gemv_pipe_t<FMT, RR, EPI_STORE>(a, S, s, pdl, grid_used);    \
    case EPI_ADD: return launch_gemv_pipe_t<FMT, RR, EPI_ADD>(a, S, s, pdl, grid_used);        \
    case EPI_QKV: return launch_gemv_pipe_t<FMT, RR, EPI_QKV>(a, S, s, pdl, grid_used);        \
    case EPI_SWIGLU: return launch_gemv_pipe_t<FMT, RR, EPI_SWIGLU>(a, S, s, pdl, grid_used);  \
    case EPI_LOGITS: return launch_gemv_pipe_t<FMT, RR, EPI_LOGITS>(a, S, s, pdl, grid_used);  \
  }
  if (R == 4) {
    NT_EPI_CASES(4)
  } else {
    NT_EPI_CASES(2)
  }
#undef NT_EPI_CASES
  return cudaErrorInvalidValue;
}

#define NT_DECLARE_GEMV_PIPE(NAME) \
  cudaError_t NAME(const GemvArgs& a, int epi, int R, int S, cudaStream_t s, bool pdl, int* grid_used);
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q8_0)
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q4_0)
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q4_k)
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q6_k)
#undef NT_DECLARE_GEMV_PIPE

}  // namespace nt
