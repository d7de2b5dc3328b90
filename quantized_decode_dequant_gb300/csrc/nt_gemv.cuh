// nt_gemv.cuh -- fused dequantize-GEMV, y = W x at batch 1 (hada "Architektur und
// Codestruktur": "cuda/: GEMV-... Kernel"; the step's cost is these weight reads).
//
// Work split.  A thread owns U "units" of 32 consecutive columns and keeps the
// matching 32*U activations in registers for the whole launch, so x is read
// from shared memory once per CTA and every weight byte is fetched exactly once
// with 128-bit non-allocating loads.  Tr threads cover one row (the split over
// K inside a row group); G = blockDim/Tr groups per CTA work on different rows.
// Each group handles R = 4 rows per iteration: a thread issues the loads of all
// four rows before any arithmetic, dequantizes in registers and accumulates in
// fp32; a transposed warp reduction then leaves one sum per row per warp and
// the group's warps are summed through shared memory.  Row groups are dealt
// round-robin over all (CTA, group) slots of a one-wave grid.
//
// Dequantization arithmetic (exact per element, scale applied per unit):
//  - 8-bit codes: the byte (sign bit flipped) is placed under the exponent of
//    2^23 with one byte permute, and 2^23 + 128 subtracted: the code q exactly.
//  - 4-bit codes: nibble i of a 16-bit half is masked in place (value q*16^i)
//    under the exponent of 2^23 and 2^23 (+ offset*16^i) subtracted; the
//    activation it multiplies was pre-scaled by 16^-i when x was loaded.
//  - Q4_K: sum_c (d sc q_c - dmin m) x_c = d sc sum q_c x_c - dmin m sum x_c,
//    with sum x_c per unit computed once per CTA.
#pragma once

#include "nt_internal.cuh"

namespace nt {

constexpr int kMaxThreads = 512;
// rows per group iteration: 4 when a thread owns one 32-column unit, 2 when it owns two
template <int U> struct RowsPer { static constexpr int value = U == 1 ? 4 : 2; };
template <int U> struct ThreadsMax { static constexpr int value = U == 1 ? 512 : 448; };

__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float h2f_bits(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)b)); }

// (q - off) * 16^i exactly, from the nibble already masked in place at bits [4i, 4i+4)
template <int I, int OFF>
__device__ __forceinline__ float nib_val(uint32_t masked) {
  return __int_as_float(int(masked | 0x4B000000u)) - (8388608.0f + float(OFF) * float(1 << (4 * I)));
}

// ------------------------------------------------------------ formats --

// Per-(row, unit) register payload and its dot product with the unit's
// activations xs[32] (pre-scaled as the format requires) and their sum.
template <int FMT> struct Unit;

template <> struct Unit<NT_Q8_0> {
  uint4 a, b;
  uint32_t d;
  static constexpr bool kScaledX = false;
  __device__ __forceinline__ void load(const QMat& m, int64_t lr, int unit) {
    const uint8_t* q = m.q + lr * m.cols + int64_t(unit) * 32;
    a = ldg_stream16(q);
    b = ldg_stream16(q + 16);
    d = ldg_u16(m.d + lr * (m.cols / 32) + unit);
  }
  __device__ __forceinline__ float dot(const float* xs, float /*xsum*/) const {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const uint32_t u = w[k] ^ 0x80808080u;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float q = __int_as_float(int(__byte_perm(u, 0x4B000000u, 0x7440u | i))) - 8388736.0f;
        if (i & 1) s1 = fmaf(q, xs[4 * k + i], s1);
        else s0 = fmaf(q, xs[4 * k + i], s0);
      }
    }
    return h2f_bits(d) * (s0 + s1);
  }
};

// 8 nibbles of one word against x[0..7] (scaled by 16^-(i%4)); offset subtracted per code
template <int OFF>
__device__ __forceinline__ void nib8(uint32_t w, const float* x, float& s0, float& s1) {
  const uint32_t h = w >> 16;
  s0 = fmaf(nib_val<0, OFF>(w & 0xFu), x[0], s0);
  s1 = fmaf(nib_val<1, OFF>(w & 0xF0u), x[1], s1);
  s0 = fmaf(nib_val<2, OFF>(w & 0xF00u), x[2], s0);
  s1 = fmaf(nib_val<3, OFF>(w & 0xF000u), x[3], s1);
  s0 = fmaf(nib_val<0, OFF>(h & 0xFu), x[4], s0);
  s1 = fmaf(nib_val<1, OFF>(h & 0xF0u), x[5], s1);
  s0 = fmaf(nib_val<2, OFF>(h & 0xF00u), x[6], s0);
  s1 = fmaf(nib_val<3, OFF>(h & 0xF000u), x[7], s1);
}

template <> struct Unit<NT_Q4_0> {
  uint4 a;
  uint32_t d;
  static constexpr bool kScaledX = true;
  __device__ __forceinline__ void load(const QMat& m, int64_t lr, int unit) {
    a = ldg_stream16(m.q + (lr * m.cols + int64_t(unit) * 32) / 2);
    d = ldg_u16(m.d + lr * (m.cols / 32) + unit);
  }
  __device__ __forceinline__ float dot(const float* xs, float /*xsum*/) const {
    float s0 = 0.f, s1 = 0.f;
    nib8<8>(a.x, xs, s0, s1);
    nib8<8>(a.y, xs + 8, s0, s1);
    nib8<8>(a.z, xs + 16, s0, s1);
    nib8<8>(a.w, xs + 24, s0, s1);
    return h2f_bits(d) * (s0 + s1);
  }
};

template <> struct Unit<NT_Q4_K> {
  uint4 a, meta;
  int j;
  static constexpr bool kScaledX = true;
  __device__ __forceinline__ void load(const QMat& m, int64_t lr, int unit) {
    a = ldg_stream16(m.q + (lr * m.cols + int64_t(unit) * 32) / 2);
    meta = __ldg(reinterpret_cast<const uint4*>(m.meta + (lr * (m.cols / 256) + unit / 8) * 16));
    j = unit & 7;
  }
  __device__ __forceinline__ float dot(const float* xs, float xsum) const {
    float s0 = 0.f, s1 = 0.f;
    nib8<0>(a.x, xs, s0, s1);
    nib8<0>(a.y, xs + 8, s0, s1);
    nib8<0>(a.z, xs + 16, s0, s1);
    nib8<0>(a.w, xs + 24, s0, s1);
    // 6-bit fields: sc_j at bit 6j, m_j at bit 6(8+j) of the 96-bit stream (meta.y, meta.z, meta.w)
    const uint64_t lo = uint64_t(meta.y) | (uint64_t(meta.z) << 32);
    const uint32_t sc = uint32_t(lo >> (6 * j)) & 63u;
    const int mb = 48 + 6 * j;
    const uint32_t mm = mb >= 64 ? (meta.w >> (mb - 64)) & 63u
                                 : uint32_t((lo >> mb) | (uint64_t(meta.w) << (64 - mb))) & 63u;
    const float a_ = h2f_bits(meta.x & 0xFFFFu) * float(sc);
    const float b_ = h2f_bits(meta.x >> 16) * float(mm);
    return a_ * (s0 + s1) - b_ * xsum;
  }
};

template <> struct Unit<NT_Q6_K> {
  uint4 a;
  uint2 h;
  uint32_t sc, d;
  static constexpr bool kScaledX = true;
  __device__ __forceinline__ void load(const QMat& m, int64_t lr, int unit) {
    const int64_t e = lr * m.cols + int64_t(unit) * 32;
    a = ldg_stream16(m.q + e / 2);
    h = ldg_stream8(m.qh + e / 4);
    sc = ldg_u16(m.meta + e / 16);
    d = ldg_u16(m.d + e / 256);
  }
  // word w (elements 8k..8k+7) with the high bits h16 (element 8k+i at bits 2i)
  __device__ __forceinline__ static void six8(uint32_t w, uint32_t h16, const float* x, float& s0, float& s1) {
    const uint32_t wh = w >> 16, hh = h16 >> 8;
    s0 = fmaf(nib_val<0, 32>((w & 0xFu) | ((h16 << 4) & 0x30u)), x[0], s0);
    s1 = fmaf(nib_val<1, 32>((w & 0xF0u) | ((h16 << 6) & 0x300u)), x[1], s1);
    s0 = fmaf(nib_val<2, 32>((w & 0xF00u) | ((h16 << 8) & 0x3000u)), x[2], s0);
    s1 = fmaf(nib_val<3, 32>((w & 0xF000u) | ((h16 << 10) & 0x30000u)), x[3], s1);
    s0 = fmaf(nib_val<0, 32>((wh & 0xFu) | ((hh << 4) & 0x30u)), x[4], s0);
    s1 = fmaf(nib_val<1, 32>((wh & 0xF0u) | ((hh << 6) & 0x300u)), x[5], s1);
    s0 = fmaf(nib_val<2, 32>((wh & 0xF00u) | ((hh << 8) & 0x3000u)), x[6], s0);
    s1 = fmaf(nib_val<3, 32>((wh & 0xF000u) | ((hh << 10) & 0x30000u)), x[7], s1);
  }
  __device__ __forceinline__ float dot(const float* xs, float /*xsum*/) const {
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    six8(a.x, h.x & 0xFFFFu, xs, a0, a1);
    six8(a.y, h.x >> 16, xs + 8, a0, a1);
    six8(a.z, h.y & 0xFFFFu, xs + 16, b0, b1);
    six8(a.w, h.y >> 16, xs + 24, b0, b1);
    const float dd = h2f_bits(d);
    const float sc0 = float(int8_t(sc & 0xFF)), sc1 = float(int8_t(sc >> 8));
    return dd * (sc0 * (a0 + a1) + sc1 * (b0 + b1));
  }
};

// --------------------------------------------------------------- kernel --

struct RowRef {
  int seg;
  int64_t lr;
};

__device__ __forceinline__ RowRef map_row(const GemvArgs& a, int64_t row) {
  RowRef r;
  if (a.interleave) {
    r.seg = int(row & 1);
    r.lr = row >> 1;
    return r;
  }
  r.seg = 0;
  r.lr = row;
  if (a.nseg > 1 && r.lr >= a.seg[0].rows) {
    r.lr -= a.seg[0].rows;
    r.seg = 1;
    if (a.nseg > 2 && r.lr >= a.seg[1].rows) {
      r.lr -= a.seg[1].rows;
      r.seg = 2;
    }
  }
  return r;
}

__device__ __forceinline__ const QMat& seg_ref(const GemvArgs& a, int s) {
  return s == 0 ? a.seg[0] : (s == 1 ? a.seg[1] : a.seg[2]);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// keep (best value, its index, second value); ties go to the lower index
__device__ __forceinline__ void top2_push(float v, int i, float& b, int& bi, float& s) {
  if (v > b || (v == b && i < bi)) {
    s = fmaxf(s, b);
    b = v;
    bi = i;
  } else {
    s = fmaxf(s, v);
  }
}

template <int FMT, int U, int EPI>
__global__ void __launch_bounds__(ThreadsMax<U>::value, 1)
    k_gemv(const __grid_constant__ GemvArgs a, const int64_t nrows, const int tr) {
  constexpr int kRows = RowsPer<U>::value;
  extern __shared__ float4 smem4[];
  float* xsh = reinterpret_cast<float*>(smem4);                      // [cols]
  const int64_t cols = a.seg[0].cols;
  float* red = xsh + cols;                                           // [2][warps][kRows]
  __shared__ float s_norm[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int groups = blockDim.x / tr;
  const int g = tid / tr;                 // row group of this thread
  const int gt = tid - g * tr;            // thread within the group
  const int wpg = tr >> 5;                // warps per group
  const int units = int(cols / 32);

  // weights never depend on the previous kernel: only x (and the epilogue's
  // outputs) do, so wait for the producer grid here, before touching them
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- stage x (and the RMSNorm scale) ------------------------------------
  {
    const float4* x4 = reinterpret_cast<const float4*>(a.x);
    float ss = 0.f;
    for (int i = tid; i < cols / 4; i += blockDim.x) {
      float4 v = x4[i];
      smem4[i] = v;
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    if (a.norm) {
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_norm[warp] = ss;
    }
    __syncthreads();
  }
  float scale = 1.0f;
  if (a.norm) {
    float t = 0.f;
    for (int w = 0; w < nwarps; w++) t += s_norm[w];
    scale = rsqrtf(t / float(cols) + a.eps);
  }

  float xs[U][32];
  float xsum[U];
  bool uact[U];
#pragma unroll
  for (int u = 0; u < U; u++) {
    const int unit = gt * U + u;
    uact[u] = unit < units;
    xsum[u] = 0.f;
#pragma unroll
    for (int c = 0; c < 32; c++) {
      float v = uact[u] ? xsh[unit * 32 + c] * scale : 0.f;
      xsum[u] += v;
      if (Unit<FMT>::kScaledX) {
        const int i = c & 3;   // nibble position within its 16-bit half
        v *= (i == 0 ? 1.f : (i == 1 ? 0.0625f : (i == 2 ? 0.00390625f : 0.000244140625f)));
      }
      xs[u][c] = v;
    }
  }

  // ---- rows ----------------------------------------------------------------
  const int64_t ngroups_rows = (nrows + kRows - 1) / kRows;
  const int64_t slots = int64_t(gridDim.x) * groups;
  const int64_t iters = (ngroups_rows + slots - 1) / slots;
  const int64_t slot = int64_t(blockIdx.x) * groups + g;

  float best = -INFINITY, second = -INFINITY;
  int best_i = 0x7fffffff;

  for (int64_t it = 0; it < iters; it++) {
    const int64_t rg = slot + it * slots;
    const int64_t r0 = rg * kRows;
    Unit<FMT> ld[kRows][U];
    bool ract[kRows];
#pragma unroll
    for (int rr = 0; rr < kRows; rr++) {
      const int64_t row = r0 + rr;
      ract[rr] = rg < ngroups_rows && row < nrows;
      if (ract[rr]) {
        const RowRef ref = map_row(a, row);
        const QMat& m = seg_ref(a, ref.seg);
#pragma unroll
        for (int u = 0; u < U; u++)
          if (uact[u]) ld[rr][u].load(m, ref.lr, gt * U + u);
      }
    }
    float acc[kRows];
#pragma unroll
    for (int rr = 0; rr < kRows; rr++) {
      acc[rr] = 0.f;
#pragma unroll
      for (int u = 0; u < U; u++)
        if (ract[rr] && uact[u]) acc[rr] += ld[rr][u].dot(xs[u], xsum[u]);
    }
    // transposed warp reduction: after it lane l holds the warp sum of row l / (32 / kRows)
    {
      float k;
      if (kRows == 4) {
        const bool up = lane & 16;
        float k0 = up ? acc[2 % kRows] : acc[0], k1 = up ? acc[3 % kRows] : acc[1 % kRows];
        const float s0 = up ? acc[0] : acc[2 % kRows], s1 = up ? acc[1 % kRows] : acc[3 % kRows];
        k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
        k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
        const bool up2 = lane & 8;
        k = up2 ? k1 : k0;
        const float s = up2 ? k0 : k1;
        k += __shfl_xor_sync(0xffffffffu, s, 8);
      } else {
        const bool up = lane & 16;
        k = up ? acc[1 % kRows] : acc[0];
        const float s = up ? acc[0] : acc[1 % kRows];
        k += __shfl_xor_sync(0xffffffffu, s, 16);
        k += __shfl_xor_sync(0xffffffffu, k, 8);
      }
      k += __shfl_xor_sync(0xffffffffu, k, 4);
      k += __shfl_xor_sync(0xffffffffu, k, 2);
      k += __shfl_xor_sync(0xffffffffu, k, 1);
      constexpr int lanes_per_row = 32 / kRows;
      if ((lane & (lanes_per_row - 1)) == 0) red[((it & 1) * nwarps + warp) * kRows + lane / lanes_per_row] = k;
    }
    __syncthreads();
    // epilogue: thread t < groups*kRows finishes row (t % kRows) of group t / kRows
    if (tid < 64) {   // whole warps: groups * kRows <= 64 epilogue threads
      const int eg = tid / kRows, rr = tid % kRows;
      const int64_t rge = int64_t(blockIdx.x) * groups + eg + it * slots;
      const int64_t row = rge * kRows + rr;
      const bool mine = tid < groups * kRows;
      float v = 0.f;
      if (mine)
        for (int w = 0; w < wpg; w++) v += red[((it & 1) * nwarps + eg * wpg + w) * kRows + rr];
      const bool live = mine && rge < ngroups_rows && row < nrows;
      if (EPI == EPI_STORE) {
        if (live) a.epi.y[row] = v;
      } else if (EPI == EPI_ADD) {
        if (live) a.epi.y[row] += v;
      } else if (EPI == EPI_LOGITS) {
        if (live) {
          a.epi.y[row] = v;
          top2_push(v, int(row), best, best_i, second);
        }
      } else {
        // pair epilogues: rows (2i, 2i+1) sit in the same group, adjacent lanes
        const float other = __shfl_xor_sync(0xffffffffu, v, 1);
        if (live && (rr & 1) == 0) {
          const float v0 = v, v1 = other;
          if (EPI == EPI_SWIGLU) {
            a.epi.y[row >> 1] = silu(v0) * v1;
          } else {  // EPI_QKV
            const int L = a.epi.row_base + int(row);
            const int hd = a.epi.head_dim;
            const int p = *a.epi.pos;
            if (L < a.epi.q_rows + a.epi.k_rows) {
              const int d = L % hd;
              const float2 cs = a.epi.rope[int64_t(p) * (hd / 2) + d / 2];
              const float r0v = v0 * cs.x - v1 * cs.y;
              const float r1v = v0 * cs.y + v1 * cs.x;
              if (L < a.epi.q_rows) {
                a.epi.y[L] = r0v;
                a.epi.y[L + 1] = r1v;
              } else {
                const int kr = L - a.epi.q_rows;
                __half* dst = a.epi.k_cache + (int64_t(kr / hd) * a.epi.max_ctx + p) * hd + d;
                dst[0] = __float2half_rn(r0v);
                dst[1] = __float2half_rn(r1v);
              }
            } else {
              const int vr = L - a.epi.q_rows - a.epi.k_rows;
              const int d = vr % hd;
              __half* dst = a.epi.v_cache + (int64_t(vr / hd) * a.epi.max_ctx + p) * hd + d;
              dst[0] = __float2half_rn(v0);
              dst[1] = __float2half_rn(v1);
            }
          }
        }
      }
    }
  }

  asm volatile("griddepcontrol.launch_dependents;");

  if (EPI == EPI_LOGITS) {
    // CTA-wide top-2 over the epilogue threads (at most 32 * kRows... all < 64)
    __shared__ float s_b[64], s_s[64];
    __shared__ int s_i[64];
    __syncthreads();
    if (tid < groups * kRows) {
      s_b[tid] = best;
      s_s[tid] = second;
      s_i[tid] = best_i;
    }
    __syncthreads();
    if (tid == 0) {
      float b = -INFINITY, s = -INFINITY;
      int bi = 0x7fffffff;
      for (int t = 0; t < groups * kRows; t++) {
        if (s_i[t] == 0x7fffffff) continue;
        top2_push(s_b[t], s_i[t], b, bi, s);
        s = fmaxf(s, s_s[t]);
      }
      a.epi.top2[blockIdx.x] = make_float4(b, __int_as_float(bi), s, 0.f);
    }
  }
}

// Threads per row group for a given column count: ceil(units / U) rounded up to a warp.
inline int gemv_tr(int64_t cols, int U) {
  const int64_t units = cols / 32;
  int64_t t = (units + U - 1) / U;
  t = (t + 31) / 32 * 32;
  return int(t);
}

inline int gemv_units_per_thread(int64_t cols) { return cols / 32 > kMaxThreads ? 2 : 1; }
inline int gemv_max_threads(int U) { return U == 1 ? ThreadsMax<1>::value : ThreadsMax<2>::value; }
inline int gemv_rows_per_iter(int U) { return U == 1 ? RowsPer<1>::value : RowsPer<2>::value; }

inline size_t gemv_smem(int64_t cols, int threads, int U) {
  return size_t(cols) * 4 + size_t(2 * (threads / 32) * gemv_rows_per_iter(U)) * 4;
}

template <int FMT, int U, int EPI>
cudaError_t launch_gemv_t(const GemvArgs& a, int threads, int tr, cudaStream_t s, bool pdl, int* grid_used) {
  const int64_t nrows = gemv_logical_rows(a);
  const size_t smem = gemv_smem(a.seg[0].cols, threads, U);
  constexpr int kRows = RowsPer<U>::value;
  auto kern = k_gemv<FMT, U, EPI>;
  static int s_sms = 0;
  static int s_occ_threads = 0, s_occ = 0;
  static size_t s_occ_smem = 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  if (!s_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&s_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  if (s_occ_threads != threads || s_occ_smem != smem) {
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
    if (e != cudaSuccess) return e;
    s_occ = occ < 1 ? 1 : occ;
    s_occ_threads = threads;
    s_occ_smem = smem;
  }
  const int groups = threads / tr;
  const int64_t row_groups = (nrows + kRows - 1) / kRows;
  int64_t grid = int64_t(s_sms) * s_occ;
  const int64_t need = (row_groups + groups - 1) / groups;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  if (grid_used) *grid_used = int(grid);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, nrows, tr);
}

template <int FMT>
cudaError_t launch_gemv_fmt(const GemvArgs& a, int epi, int threads, int tr, int U, cudaStream_t s, bool pdl,
                            int* grid_used) {
#define NT_EPI_CASES(UU)                                                                              \
  switch (epi) {                                                                                      \
    case EPI_STORE: return launch_gemv_t<FMT, UU, EPI_STORE>(a, threads, tr, s, pdl, grid_used);      \
    case EPI_ADD: return launch_gemv_t<FMT, UU, EPI_ADD>(a, threads, tr, s, pdl, grid_used);          \
    case EPI_QKV: return launch_gemv_t<FMT, UU, EPI_QKV>(a, threads, tr, s, pdl, grid_used);          \
    case EPI_SWIGLU: return launch_gemv_t<FMT, UU, EPI_SWIGLU>(a, threads, tr, s, pdl, grid_used);    \
    case EPI_LOGITS: return launch_gemv_t<FMT, UU, EPI_LOGITS>(a, threads, tr, s, pdl, grid_used);    \
  }
  if (U == 1) {
    NT_EPI_CASES(1)
  } else {
    NT_EPI_CASES(2)
  }
#undef NT_EPI_CASES
  return cudaErrorInvalidValue;
}

#define NT_DECLARE_GEMV(NAME) \
  cudaError_t NAME(const GemvArgs& a, int epi, int threads, int tr, int U, cudaStream_t s, bool pdl, int* grid_used);
NT_DECLARE_GEMV(launch_gemv_q8_0)
NT_DECLARE_GEMV(launch_gemv_q4_0)
NT_DECLARE_GEMV(launch_gemv_q4_k)
NT_DECLARE_GEMV(launch_gemv_q6_k)
#undef NT_DECLARE_GEMV

}  // namespace nt
