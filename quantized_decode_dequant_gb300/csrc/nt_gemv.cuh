// nt_gemv.cuh -- fused dequantize-GEMV, y = W x at batch 1 (hada "Architektur und
// Codestruktur": "cuda/: GEMV-... Kernel"; the decode step's cost is these weight reads).
//
// This header holds the per-format decode arithmetic and the register-path
// kernel, used for column counts the shared-memory pipeline (nt_gemv_pipe.cuh)
// does not take.  Work split: a CTA stages x once in shared memory
// (RMS-normalised when asked, pre-scaled or permuted for the format's decode,
// padded so 16-byte reads of consecutive lanes hit distinct banks) and then
// every warp works alone: it owns groups of R consecutive rows, its lanes split
// the columns into "units" (16 columns for Q8_0, 32 for the 4/6-bit formats;
// lane l takes units l, l+32, ...), and each unit's codes are fetched with one
// 128-bit non-allocating load per row.  The loads of the next unit (or of the
// next row group's first unit) are issued before the current unit is decoded.
// No barrier is taken in the loop; a transposed warp reduction ends each row
// group and the epilogue runs on the lanes that hold the row sums.  Row groups
// are dealt round-robin over all warps of a one-wave grid.  Weights do not
// depend on the previous kernel, so the first loads are issued before
// griddepcontrol.wait (programmatic dependent launch).
//
// Decode arithmetic (exact per element; the scales are applied once per unit,
// fp32 accumulation, packed f32x2 FMA):
//  - Q8_0: byte b (sign bit flipped) is placed under the exponent of 2^23 by a
//    byte permute; subtracting 2^23 + 128 gives the code q exactly.
//  - Q4_0 / Q4_K: nibble i of a 16-bit half is masked in place (value q*16^i)
//    under the exponent of 2^23; subtracting 2^23 (+ 8*16^i for Q4_0) gives
//    (q - off)*16^i exactly and x was pre-scaled by 16^-i when staged.
//    Q4_K: sum_c (d sc q_c - dmin m) x_c = d sc sum q_c x_c - dmin m sum x_c,
//    with sum x_c per unit staged once per CTA.
//  - Q6_K: the low nibbles of the even (odd) elements of a code word are
//    masked (shifted) into bytes, the two high bits OR-ed in from the device's
//    high-bit word, each byte placed under 2^23 and 2^23 + 32 subtracted;
//    x is staged in the matching even/odd order.
#pragma once

#include "nt_internal.cuh"

namespace nt {

constexpr int kThreads = 512;   // 16 warps per CTA
constexpr int kXPad = 4;        // floats of padding after each unit's x in shared memory

__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg8(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg2(const void* p) {
  unsigned short v;
  asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float h2f_bits(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)b)); }
__device__ __forceinline__ float bits_f(uint32_t b) { return __uint_as_float(b); }

constexpr uint32_t kMagicBits = 0x4B000000u;   // 2^23
constexpr float kMagic = 8388608.0f;

// ------------------------------------------------------------ formats --

template <int FMT> struct Fmt;

// 16 int8 codes of one 16-byte vector against x[0..15]
__device__ __forceinline__ float q8_dot16(uint4 c, const float4* xs) {
  const float2 off = make_float2(-(kMagic + 128.0f), -(kMagic + 128.0f));
  float2 acc = make_float2(0.f, 0.f);
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const uint32_t u = w[k] ^ 0x80808080u;
    const float4 x = xs[k];
    const float2 q01 = __fadd2_rn(make_float2(bits_f(__byte_perm(u, kMagicBits, 0x7440u)),
                                              bits_f(__byte_perm(u, kMagicBits, 0x7441u))), off);
    const float2 q23 = __fadd2_rn(make_float2(bits_f(__byte_perm(u, kMagicBits, 0x7442u)),
                                              bits_f(__byte_perm(u, kMagicBits, 0x7443u))), off);
    acc = __ffma2_rn(q01, make_float2(x.x, x.y), acc);
    acc = __ffma2_rn(q23, make_float2(x.z, x.w), acc);
  }
  return acc.x + acc.y;
}

template <> struct Fmt<NT_Q8_0> {
  static constexpr int kCols = 16;
  static constexpr bool kXSum = false;
  struct Pay {
    uint4 c;
    uint32_t d;
  };
  __device__ static void load(Pay& p, const QMat& m, int64_t e) {   // e: flat index of the unit's first element
    p.c = ldg16(m.q + e);
    p.d = ldg2(m.d + (e >> 5));
  }
  // x staged in natural order
  __device__ static int xpos(int c) { return c; }
  __device__ static float xscale(int) { return 1.0f; }
  __device__ static float dot(const Pay& p, const float4* xs, float) { return h2f_bits(p.d) * q8_dot16(p.c, xs); }
};

// 8 nibbles of one word against x[0..7] (pre-scaled by 16^-(i%4)); OFF subtracted per code
template <int OFF>
__device__ __forceinline__ float2 nib8(uint32_t w, float4 xa, float4 xb, float2 acc) {
  const float2 o01 = make_float2(-(kMagic + float(OFF)), -(kMagic + float(OFF) * 16.0f));
  const float2 o23 = make_float2(-(kMagic + float(OFF) * 256.0f), -(kMagic + float(OFF) * 4096.0f));
  const uint32_t h = w >> 16;
  const float2 a = __fadd2_rn(make_float2(bits_f((w & 0xFu) | kMagicBits), bits_f((w & 0xF0u) | kMagicBits)), o01);
  const float2 b = __fadd2_rn(make_float2(bits_f((w & 0xF00u) | kMagicBits), bits_f((w & 0xF000u) | kMagicBits)), o23);
  const float2 c = __fadd2_rn(make_float2(bits_f((h & 0xFu) | kMagicBits), bits_f((h & 0xF0u) | kMagicBits)), o01);
  const float2 d = __fadd2_rn(make_float2(bits_f((h & 0xF00u) | kMagicBits), bits_f((h & 0xF000u) | kMagicBits)), o23);
  acc = __ffma2_rn(a, make_float2(xa.x, xa.y), acc);
  acc = __ffma2_rn(b, make_float2(xa.z, xa.w), acc);
  acc = __ffma2_rn(c, make_float2(xb.x, xb.y), acc);
  acc = __ffma2_rn(d, make_float2(xb.z, xb.w), acc);
  return acc;
}

__device__ __forceinline__ float nib_xscale(int c) {
  const int i = c & 3;
  return i == 0 ? 1.f : (i == 1 ? 0.0625f : (i == 2 ? 0.00390625f : 0.000244140625f));
}

template <> struct Fmt<NT_Q4_0> {
  static constexpr int kCols = 32;
  static constexpr bool kXSum = false;
  struct Pay {
    uint4 c;
    uint32_t d;
  };
  __device__ static void load(Pay& p, const QMat& m, int64_t e) {
    p.c = ldg16(m.q + (e >> 1));
    p.d = ldg2(m.d + (e >> 5));
  }
  __device__ static int xpos(int c) { return c; }
  __device__ static float xscale(int c) { return nib_xscale(c); }
  __device__ static float dot(const Pay& p, const float4* xs, float) {
    float2 acc = make_float2(0.f, 0.f);
    acc = nib8<8>(p.c.x, xs[0], xs[1], acc);
    acc = nib8<8>(p.c.y, xs[2], xs[3], acc);
    acc = nib8<8>(p.c.z, xs[4], xs[5], acc);
    acc = nib8<8>(p.c.w, xs[6], xs[7], acc);
    return h2f_bits(p.d) * (acc.x + acc.y);
  }
};

template <> struct Fmt<NT_Q4_K> {
  static constexpr int kCols = 32;
  static constexpr bool kXSum = true;
  struct Pay {
    uint4 c, meta;
    int j;
  };
  __device__ static void load(Pay& p, const QMat& m, int64_t e) {
    p.c = ldg16(m.q + (e >> 1));
    p.meta = __ldg(reinterpret_cast<const uint4*>(m.meta + (e >> 8) * 16));
    p.j = int(e >> 5) & 7;
  }
  __device__ static int xpos(int c) { return c; }
  __device__ static float xscale(int c) { return nib_xscale(c); }
  __device__ static float dot(const Pay& p, const float4* xs, float xsum) {
    float2 acc = make_float2(0.f, 0.f);
    acc = nib8<0>(p.c.x, xs[0], xs[1], acc);
    acc = nib8<0>(p.c.y, xs[2], xs[3], acc);
    acc = nib8<0>(p.c.z, xs[4], xs[5], acc);
    acc = nib8<0>(p.c.w, xs[6], xs[7], acc);
    uint32_t sc, mm;
    kquant_scale_min(p.meta, p.j, sc, mm);
    const float a = h2f_bits(p.meta.x & 0xFFFFu) * float(sc);
    const float b = h2f_bits(p.meta.x >> 16) * float(mm);
    return a * (acc.x + acc.y) - b * xsum;
  }
};

// Q5_K: code bytes built as for Q6_K (x staged [0,2,4,6,1,3,5,7] per 8 columns):
// low nibble | fifth bit from the unit's word H at bit 4; Q4_K's scale and min.
template <> struct Fmt<NT_Q5_K> {
  static constexpr int kCols = 32;
  static constexpr bool kXSum = true;
  struct Pay {
    uint4 c, meta;
    uint32_t h;
    int j;
  };
  __device__ static void load(Pay& p, const QMat& m, int64_t e) {
    p.c = ldg16(m.q + (e >> 1));
    p.h = __ldg(reinterpret_cast<const unsigned int*>(m.qh + (e >> 3)));
    p.meta = __ldg(reinterpret_cast<const uint4*>(m.meta + (e >> 8) * 16));
    p.j = int(e >> 5) & 7;
  }
  __device__ static int xpos(int c) { return (c & ~7) | ((c & 1) ? 4 + ((c & 7) >> 1) : ((c & 7) >> 1)); }
  __device__ static float xscale(int) { return 1.0f; }
  __device__ static float2 bytes4(uint32_t q, float4 x, float2 acc) {
    const float2 off = make_float2(-kMagic, -kMagic);
    const float2 a = __fadd2_rn(make_float2(bits_f(__byte_perm(q, kMagicBits, 0x7440u)),
                                            bits_f(__byte_perm(q, kMagicBits, 0x7441u))), off);
    const float2 b = __fadd2_rn(make_float2(bits_f(__byte_perm(q, kMagicBits, 0x7442u)),
                                            bits_f(__byte_perm(q, kMagicBits, 0x7443u))), off);
    acc = __ffma2_rn(a, make_float2(x.x, x.y), acc);
    return __ffma2_rn(b, make_float2(x.z, x.w), acc);
  }
  __device__ static float dot(const Pay& p, const float4* xs, float xsum) {
    const uint32_t L = 0x0F0F0F0Fu, M = 0x10101010u, H = p.h;
    float2 acc = make_float2(0.f, 0.f);
    acc = bytes4((p.c.x & L) | ((H << 4) & M), xs[0], acc);
    acc = bytes4(((p.c.x >> 4) & L) | ((H << 3) & M), xs[1], acc);
    acc = bytes4((p.c.y & L) | ((H << 2) & M), xs[2], acc);
    acc = bytes4(((p.c.y >> 4) & L) | ((H << 1) & M), xs[3], acc);
    acc = bytes4((p.c.z & L) | (H & M), xs[4], acc);
    acc = bytes4(((p.c.z >> 4) & L) | ((H >> 1) & M), xs[5], acc);
    acc = bytes4((p.c.w & L) | ((H >> 2) & M), xs[6], acc);
    acc = bytes4(((p.c.w >> 4) & L) | ((H >> 3) & M), xs[7], acc);
    uint32_t sc, mm;
    kquant_scale_min(p.meta, p.j, sc, mm);
    const float a = h2f_bits(p.meta.x & 0xFFFFu) * float(sc);
    const float b = h2f_bits(p.meta.x >> 16) * float(mm);
    return a * (acc.x + acc.y) - b * xsum;
  }
};

template <> struct Fmt<NT_Q6_K> {
  static constexpr int kCols = 32;
  static constexpr bool kXSum = false;
  struct Pay {
    uint4 c;
    uint2 h;
    uint32_t sc, d;
  };
  __device__ static void load(Pay& p, const QMat& m, int64_t e) {
    p.c = ldg16(m.q + (e >> 1));
    p.h = ldg8(m.qh + (e >> 2));
    p.sc = ldg2(m.meta + (e >> 4));
    p.d = ldg2(m.d + (e >> 8));
  }
  // within each group of 8 columns x is staged as [0,2,4,6,1,3,5,7]
  __device__ static int xpos(int c) { return (c & ~7) | ((c & 1) ? 4 + ((c & 7) >> 1) : ((c & 7) >> 1)); }
  __device__ static float xscale(int) { return 1.0f; }
  // four 6-bit codes (one per byte) minus 32, against x[0..3]
  __device__ static float2 bytes4(uint32_t q, float4 x, float2 acc) {
    const float2 off = make_float2(-(kMagic + 32.0f), -(kMagic + 32.0f));
    const float2 a = __fadd2_rn(make_float2(bits_f(__byte_perm(q, kMagicBits, 0x7440u)),
                                            bits_f(__byte_perm(q, kMagicBits, 0x7441u))), off);
    const float2 b = __fadd2_rn(make_float2(bits_f(__byte_perm(q, kMagicBits, 0x7442u)),
                                            bits_f(__byte_perm(q, kMagicBits, 0x7443u))), off);
    acc = __ffma2_rn(a, make_float2(x.x, x.y), acc);
    return __ffma2_rn(b, make_float2(x.z, x.w), acc);
  }
  __device__ static float dot(const Pay& p, const float4* xs, float) {
    // device high-bit word G (one per 16 elements): byte j holds, for code words
    // W (elements 0..7) and W' (elements 8..15), hi(W,2j) at bits 4-5,
    // hi(W',2j) at bits 6-7, hi(W,2j+1) at bits 0-1, hi(W',2j+1) at bits 2-3
    const uint32_t M = 0x30303030u, L = 0x0F0F0F0Fu;
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
    const uint32_t g0 = p.h.x, g1 = p.h.y;
    a0 = bytes4((p.c.x & L) | (g0 & M), xs[0], a0);
    a0 = bytes4(((p.c.x >> 4) & L) | ((g0 << 4) & M), xs[1], a0);
    a0 = bytes4((p.c.y & L) | ((g0 >> 2) & M), xs[2], a0);
    a0 = bytes4(((p.c.y >> 4) & L) | ((g0 << 2) & M), xs[3], a0);
    a1 = bytes4((p.c.z & L) | (g1 & M), xs[4], a1);
    a1 = bytes4(((p.c.z >> 4) & L) | ((g1 << 4) & M), xs[5], a1);
    a1 = bytes4((p.c.w & L) | ((g1 >> 2) & M), xs[6], a1);
    a1 = bytes4(((p.c.w >> 4) & L) | ((g1 << 2) & M), xs[7], a1);
    const float sc0 = float(int8_t(p.sc & 0xFF)), sc1 = float(int8_t(p.sc >> 8));
    return h2f_bits(p.d) * (sc0 * (a0.x + a0.y) + sc1 * (a1.x + a1.y));
  }
};

// --------------------------------------------------------------- helpers --

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
__device__ __forceinline__ void top2_merge(float b2, int i2, float s2, float& b, int& bi, float& s) {
  if (i2 == 0x7fffffff) return;
  top2_push(b2, i2, b, bi, s);
  s = fmaxf(s, s2);
}

// logical row -> (segment, row inside the segment)
__device__ __forceinline__ void map_row(const GemvArgs& a, int64_t row, int& seg, int64_t& lr) {
  if (a.interleave) {
    seg = int(row & 1);
    lr = row >> 1;
    return;
  }
  seg = 0;
  lr = row;
  if (a.nseg > 1 && lr >= a.seg[0].rows) {
    lr -= a.seg[0].rows;
    seg = 1;
    if (a.nseg > 2 && lr >= a.seg[1].rows) {
      lr -= a.seg[1].rows;
      seg = 2;
    }
  }
}

// Transposed warp reduction of R per-lane partial sums: afterwards lane l holds
// the warp total of row l / (32 / R).
template <int R>
__device__ __forceinline__ float warp_reduce_rows(const float (&acc)[R], int lane) {
  float k;
  const bool up = lane & 16;
  if (R == 4) {
    float k0 = up ? acc[2 % R] : acc[0], k1 = up ? acc[3 % R] : acc[1 % R];
    const float s0 = up ? acc[0] : acc[2 % R], s1 = up ? acc[1 % R] : acc[3 % R];
    k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    const bool up2 = lane & 8;
    k = up2 ? k1 : k0;
    k += __shfl_xor_sync(0xffffffffu, up2 ? k0 : k1, 8);
  } else {
    k = up ? acc[1 % R] : acc[0];
    k += __shfl_xor_sync(0xffffffffu, up ? acc[0] : acc[1 % R], 16);
    k += __shfl_xor_sync(0xffffffffu, k, 8);
  }
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

// Epilogue of one finished row group: k is this lane's reduced row sum (valid
// on lanes l % (32/R) == 0), rows grp*R + l/(32/R).  All lanes must call it.
// y and pos: the output and the position counter (a.epi.y and a.epi.pos, or one
// token's of a multi-token launch).
template <int R, int EPI>
__device__ __forceinline__ void epilogue_to(const GemvArgs& a, float* y, const int32_t* pos, int64_t grp,
                                            int64_t nrows, int lane, float k, float& best, int& best_i,
                                            float& second) {
  constexpr int LPR = 32 / R;
  const int rr = lane / LPR;
  const int64_t row = grp * R + rr;
  const bool holder = (lane % LPR) == 0 && row < nrows;
  // pair epilogues need rows 2i and 2i+1: the odd row's sum moves onto the even holder
  const float other = __shfl_down_sync(0xffffffffu, k, LPR);
  if (!holder) return;
  if constexpr (R == 1 && EPI == EPI_QKV) {
    // one row per group, used only for V rows (the two-format Q/K/V launch's
    // second range): no RoPE pair, the f16 store of the row at the current position
    const int L = a.epi.row_base + int(row);
    const int vr = L - a.epi.q_rows - a.epi.k_rows;
    if (vr < 0) return;
    const int hd = a.epi.head_dim, p = __ldcg(pos);
    a.epi.v_cache[(int64_t(vr / hd) * a.epi.max_ctx + p) * hd + vr % hd] = __float2half_rn(k);
    return;
  }
  if (EPI == EPI_STORE) {
    y[row] = k;
  } else if (EPI == EPI_ADD) {
    y[row] = __fadd_rn(__ldcg(y + row), k);
  } else if (EPI == EPI_LOGITS) {
    y[row] = k;
    top2_push(k, int(row), best, best_i, second);
  } else if ((rr & 1) == 0) {
    const float v0 = k, v1 = other;
    if (EPI == EPI_SWIGLU) {
      y[row >> 1] = __fmul_rn(silu(v0), v1);
    } else {  // EPI_QKV: RoPE on q and k pairs, f16 store of k and v at the current position
      const int L = a.epi.row_base + int(row);
      const int hd = a.epi.head_dim;
      const int p = __ldcg(pos);
      if (L < a.epi.q_rows + a.epi.k_rows) {
        const int d = L % hd;
        const float2 cs = a.epi.rope[int64_t(p) * (hd / 2) + d / 2];
        const float r0 = __fmaf_rn(v0, cs.x, -__fmul_rn(v1, cs.y));
        const float r1 = __fmaf_rn(v0, cs.y, __fmul_rn(v1, cs.x));
        if (L < a.epi.q_rows) {
          y[L] = r0;
          y[L + 1] = r1;
        } else {
          const int kr = L - a.epi.q_rows;
          __half* dst = a.epi.k_cache + (int64_t(kr / hd) * a.epi.max_ctx + p) * hd + d;
          dst[0] = __float2half_rn(r0);
          dst[1] = __float2half_rn(r1);
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

template <int R, int EPI>
__device__ __forceinline__ void epilogue(const GemvArgs& a, int64_t grp, int64_t nrows, int lane, float k,
                                         float& best, int& best_i, float& second) {
  epilogue_to<R, EPI>(a, a.epi.y, a.epi.pos, grp, nrows, lane, k, best, best_i, second);
}

// CTA-wide top-2 of the rows this CTA finished, written to top2[blockIdx.x].
template <int NW>
__device__ __forceinline__ void cta_top2(const GemvArgs& a, int cta, float best, int best_i, float second) {
  __shared__ float s_b[NW], s_s[NW];
  __shared__ int s_i[NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, second, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, best_i, o);
    top2_merge(b2, i2, s2, best, best_i, second);
  }
  if (lane == 0) {
    s_b[warp] = best;
    s_s[warp] = second;
    s_i[warp] = best_i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = -INFINITY, s = -INFINITY;
    int bi = 0x7fffffff;
    for (int w = 0; w < NW; w++) top2_merge(s_b[w], s_i[w], s_s[w], b, bi, s);
    a.epi.top2[cta] = make_float4(b, __int_as_float(bi), s, 0.f);
  }
}

// ------------------------------------------------------ register-path kernel --

template <int FMT, int R>
struct Group {
  typename Fmt<FMT>::Pay pay[R];
  int seg[R];
  int64_t e[R];     // flat element index of the row start (row-in-segment * cols)
  bool live[R];
};

template <int FMT, int R>
__device__ __forceinline__ void group_setup(const GemvArgs& a, int64_t grp, int64_t nrows, int64_t cols,
                                            Group<FMT, R>& g) {
#pragma unroll
  for (int r = 0; r < R; r++) {
    const int64_t row = grp * R + r;
    g.live[r] = row < nrows;
    int s = 0;
    int64_t lr = 0;
    if (g.live[r]) map_row(a, row, s, lr);
    g.seg[r] = s;
    g.e[r] = lr * cols;
  }
}

template <int FMT, int R>
__device__ __forceinline__ void group_load(const GemvArgs& a, Group<FMT, R>& g, int unit) {
#pragma unroll
  for (int r = 0; r < R; r++)
    if (g.live[r]) Fmt<FMT>::load(g.pay[r], a.seg[g.seg[r]], g.e[r] + int64_t(unit) * Fmt<FMT>::kCols);
}

template <int FMT, int R, int EPI>
__global__ void __launch_bounds__(kThreads) k_gemv(const __grid_constant__ GemvArgs a, const int64_t nrows) {
  using F = Fmt<FMT>;
  constexpr int C = F::kCols, US = C + kXPad;    // unit columns, unit stride in shared memory
  extern __shared__ float4 smem4[];
  float* xsh = reinterpret_cast<float*>(smem4);
  const int64_t cols = a.seg[0].cols;
  const int units = int(cols / C);
  float* xsum = xsh + units * US;                // per 32-column unit (Q4_K)
  __shared__ float s_red[kThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int64_t ngroups = (nrows + R - 1) / R;
  const int64_t stride = int64_t(gridDim.x) * nw;
  const int kiters = (units + 31) / 32;
  int64_t grp = int64_t(blockIdx.x) * nw + warp;

  // first loads before waiting for the producer of x
  Group<FMT, R> cur;
  if (grp < ngroups) {
    group_setup<FMT, R>(a, grp, nrows, cols, cur);
    if (lane < units) group_load<FMT, R>(a, cur, lane);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- stage x ---------------------------------------------------------------
  {
    float ss = 0.f;
    for (int c = tid; c < cols; c += blockDim.x) {
      const float v = a.x[c];
      ss += v * v;
      xsh[(c / C) * US + F::xpos(c % C)] = v;
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
    if (a.norm || F::kXSum || FMT != NT_Q8_0) {
      // scale (norm, nibble position) in place; per-unit sums of the normalised x
      for (int u = warp; u < units; u += nw) {
        float v = 0.f;
        if (lane < C) {
          const int p = u * US + F::xpos(lane);
          v = xsh[p] * scale;
          xsh[p] = v * F::xscale(lane);
        }
        if (F::kXSum) {
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

  for (; grp < ngroups; grp += stride) {
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; r++) acc[r] = 0.f;
    for (int it = 0; it < kiters; it++) {
      const int u = it * 32 + lane;
      // prefetch: next unit of this group, or the first unit of the next group
      Group<FMT, R> nxt;
      bool have_next = false;
      if (it + 1 < kiters) {
        nxt = cur;
        if (u + 32 < units) group_load<FMT, R>(a, nxt, u + 32);
        have_next = true;
      } else if (grp + stride < ngroups) {
        group_setup<FMT, R>(a, grp + stride, nrows, cols, nxt);
        if (lane < units) group_load<FMT, R>(a, nxt, lane);
        have_next = true;
      }
      if (u < units) {
        const float4* xs = reinterpret_cast<const float4*>(xsh + u * US);
        const float xu = F::kXSum ? xsum[u] : 0.f;
#pragma unroll
        for (int r = 0; r < R; r++)
          if (cur.live[r]) acc[r] += F::dot(cur.pay[r], xs, xu);
      }
      if (have_next) cur = nxt;
    }
    const float k = warp_reduce_rows<R>(acc, lane);
    epilogue<R, EPI>(a, grp, nrows, lane, k, best, best_i, second);
  }

  asm volatile("griddepcontrol.launch_dependents;");
  if (EPI == EPI_LOGITS) cta_top2<kThreads / 32>(a, blockIdx.x, best, best_i, second);
}

inline size_t gemv_smem(int fmt, int64_t cols) {
  const int C = fmt == NT_Q8_0 ? 16 : 32;
  return size_t(cols / C) * (C + kXPad) * 4 + size_t(cols / 32) * 4;
}

// One-wave grid: SMs x resident CTAs, capped by the work and by a.max_grid.
inline int64_t one_wave_grid(int sms, int occ, int64_t groups, int warps_per_cta, int max_grid) {
  int64_t grid = int64_t(sms) * occ;
  const int64_t need = (groups + warps_per_cta - 1) / warps_per_cta;
  if (grid > need) grid = need;
  if (grid > max_grid) grid = max_grid;
  if (grid < 1) grid = 1;
  return grid;
}

template <int FMT, int R, int EPI>
cudaError_t launch_gemv_t(const GemvArgs& a, cudaStream_t s, bool pdl, int* grid_used) {
  const int64_t nrows = gemv_logical_rows(a);
  const size_t smem = gemv_smem(FMT, a.seg[0].cols);
  auto kern = k_gemv<FMT, R, EPI>;
  static const KernelSetup setup = kernel_setup(kern, 200 * 1024);
  if (setup.err != cudaSuccess) return setup.err;
  const int s_sms = setup.sms;
  thread_local size_t s_occ_smem = ~size_t(0);   // occupancy of the last shared-memory size (per thread)
  thread_local int s_occ = 0;
  if (s_occ_smem != smem) {
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    s_occ = occ;
    s_occ_smem = smem;
  }
  const int64_t grid = one_wave_grid(s_sms, s_occ, (nrows + R - 1) / R, kThreads / 32, a.max_grid);
  if (grid_used) *grid_used = int(grid);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(kThreads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, nrows);
}

template <int FMT>
cudaError_t launch_gemv_fmt(const GemvArgs& a, int epi, int R, cudaStream_t s, bool pdl, int* grid_used) {
#define NT_EPI_CASES(RR)                                                                   \
  switch (epi) {                                                                           \
    case EPI_STORE: return launch_gemv_t<FMT, RR, EPI_STORE>(a, s, pdl, grid_used);        \
    case EPI_ADD: return launch_gemv_t<FMT, RR, EPI_ADD>(a, s, pdl, grid_used);            \
    case EPI_QKV: return launch_gemv_t<FMT, RR, EPI_QKV>(a, s, pdl, grid_used);            \
    case EPI_SWIGLU: return launch_gemv_t<FMT, RR, EPI_SWIGLU>(a, s, pdl, grid_used);      \
    case EPI_LOGITS: return launch_gemv_t<FMT, RR, EPI_LOGITS>(a, s, pdl, grid_used);      \
  }
  if (R == 4) {
    NT_EPI_CASES(4)
  } else {
    NT_EPI_CASES(2)
  }
#undef NT_EPI_CASES
  return cudaErrorInvalidValue;
}

#define NT_DECLARE_GEMV(NAME) \
  cudaError_t NAME(const GemvArgs& a, int epi, int R, cudaStream_t s, bool pdl, int* grid_used);
NT_DECLARE_GEMV(launch_gemv_q8_0)
NT_DECLARE_GEMV(launch_gemv_q4_0)
NT_DECLARE_GEMV(launch_gemv_q4_k)
NT_DECLARE_GEMV(launch_gemv_q5_k)
NT_DECLARE_GEMV(launch_gemv_q6_k)
#undef NT_DECLARE_GEMV

}  // namespace nt
