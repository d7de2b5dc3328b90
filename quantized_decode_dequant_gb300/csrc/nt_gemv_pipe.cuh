// nt_gemv_pipe.cuh -- the fused dequantize-GEMV with weights staged through a
// per-warp shared-memory ring by asynchronous copies, decoded with integer dot
// products.
//
// Work split (as nt_gemv.cuh): warps own groups of R rows, lanes own 32-column
// units, x is staged once per CTA.  The codes and scales of each (row group,
// 32-unit column tile) are copied global -> shared with cp.async (16-byte
// LDGSTS, L2-only) S-1 tiles ahead of the tile being decoded, so every warp
// keeps (S-1) * R row tiles in flight without spending registers on them; the
// only waits are cp.async.wait_group on the warp's own copies plus __syncwarp
// for the scale bytes other lanes copied.
//
// Arithmetic.  Each 32-column block of x is carried as 16-bit fixed point: an
// fp32 scale sx = max|x|/32512 and integers t_c = round(x_c/sx) split as
// t = 256 h + l, h = floor(t / 256) a signed byte and l = t mod 256 an unsigned
// one (the two bytes of t).  The codes are exact small integers, so
// sum_c q_c t_c = 256 sum q h + sum q l is computed exactly with DP4A (four
// byte products per instruction) and only the per-block combination with the
// fp16 scales is floating point, accumulated in fp32 (the block's x scale sx
// joins in the accumulating FMA).  The offsets of the formats use the staged
// block sums T = sum t:
//   Q8_0  d sx S,                       S = 256 Sh + Sl
//   Q4_0  d sx (S - 8 T)
//   Q4_K  sx (d sc S - dmin m T)
//   Q6_K  d sx (sc_0 (S_0 - 32 T_0) + sc_1 (S_1 - 32 T_1))  (two 16-element halves)
// The only approximation beyond fp32 is x's rounding to 16 bits per block
// (|error| <= sx/2, i.e. 2^-16 of the block's largest |x|).  Nibble codes are
// spread to bytes by masking even and odd nibbles (x staged in the matching
// [0,2,4,6 | 1,3,5,7] order per 8 columns); Q6_K codes get their two high
// bits OR-ed in from the device's high-bit words.
//
// Row tile layout in shared memory (one row, 32 units):
//   Q8_0  32 x 32 B codes | 32 x f16 d                                  1088 B
//   Q4_0  32 x 16 B codes | 32 x f16 d                                   576 B
//   Q4_K  32 x 16 B codes | 4 x 16 B superblock headers                  576 B
//   Q6_K  32 x 16 B low codes | 32 x 8 B high-bit words | 32 x 2 B sc | 4 x f16 d (16 B slot)   848 B
// Requires the window width and start to be multiples of 1024 columns, so every
// tile is whole and every scale piece an aligned 16-byte (4-byte for Q6_K d) copy.
#pragma once

#include "nt_gemv.cuh"

namespace nt {

constexpr int kPipeWarps = 16;                // 512 threads per CTA, one CTA per SM
constexpr int kPipeMaxSmem = 221 * 1024;      // dynamic shared memory a CTA may ask for
constexpr int kPipeSmPerSm = 228 * 1024;      // shared memory of an SM (each resident CTA also reserves 1 KB)
// Staged x per 32 columns, in int8 slices of fixed point t = round(x/sx):
// two slices (t = 256 h + l, |t| <= 32512): h[32] | l[32] | sx, T0, T1, sum of squares;
// three slices (t = 4096 h + 16 m + l, |t| <= 520192, l in 0..15): h[32] | m[32] | l[32] | the same.
// The Q/K/V GEMV takes three: its error reaches the logits through the softmax
// over the whole context and dominates theirs with two; every other GEMV takes two.
constexpr int kXUnit = 80;
template <int XS>
__host__ __device__ constexpr int x_unit() { return XS == 3 ? 112 : 80; }
__host__ __device__ constexpr int x_slices(int epi) { return epi == EPI_QKV ? 3 : 2; }
// Before the producer of x is done only the first kPipeEarly tiles of a warp's
// ring are copied: the x loads of the staging that follows would otherwise queue
// behind a whole ring of weight copies; the rest is issued once x is staged.
// (Measured on GB300: one tile made the 70B step 0.2% faster than two, a whole
// ring 1% slower, and none 1.4% slower, 3.2% for the 8B step.  A bulk L2
// prefetch of each warp's next eight tiles of codes, issued with that tile, made
// the 70B step 2.3% slower.)
constexpr int kPipeEarly = 1;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// the same, issued only when on != 0 (a predicated copy: no branch)
__device__ __forceinline__ void cp16_if(uint32_t on, uint32_t dst, const void* src) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %2, 0;\n @p cp.async.cg.shared.global [%0], [%1], 16;\n}\n" ::"r"(dst),
      "l"(src), "r"(on)
      : "memory");
}
__device__ __forceinline__ void cp4_if(uint32_t on, uint32_t dst, const void* src) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %2, 0;\n @p cp.async.ca.shared.global [%0], [%1], 4;\n}\n" ::"r"(dst),
      "l"(src), "r"(on)
      : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// One staged x block in registers.
struct XBlock {
  int h[8], m[8], l[8];   // byte slices, four per word, in the format's element order (m: three slices only;
                          // l: unsigned with two slices)
  float sx;         // block scale
  int t0, t1;       // sums of t over elements 0..15 and 16..31
};

template <int XS>
__device__ __forceinline__ void load_xblock(const uint8_t* p, XBlock& x) {
  auto words = [](const uint8_t* q, int (&w)[8]) {
    const uint4 a = *reinterpret_cast<const uint4*>(q), b = *reinterpret_cast<const uint4*>(q + 16);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  };
  words(p, x.h);
  if (XS == 3) words(p + 32, x.m);
  words(p + 32 * (XS - 1), x.l);
  const uint4 m = *reinterpret_cast<const uint4*>(p + 32 * XS);
  x.sx = __uint_as_float(m.x);
  x.t0 = int(m.y);
  x.t1 = int(m.z);
}

// Exact integer dot of codes and t over at most 32 elements, in int32 for both
// slice counts: the largest sum is 32 x 127 x 520192 = 2,114,060,288 (8-bit codes,
// three slices), and with |h| <= 127 the partial 4096 (codes . h) and the added
// 16 (codes . m) + (codes . l) stay below 2^31 - 1 as well.  (A 64-bit sum would
// convert to float on the FP64 pipe, which is narrow on this GPU.)
template <int XS>
using xacc_t = int;
__device__ __forceinline__ float xacc_f(int v) { return __int2float_rn(v); }

// sum over words [W0, W1) of (codes . t): 256 (codes . h) + (codes . l), or
// 4096 (codes . h) + 16 (codes . m) + (codes . l)
// DP4A of signed code bytes with unsigned x bytes (the low slice of a two-slice x)
__device__ __forceinline__ int dp4a_su(int a, int b, int c) {
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ int dp4a_us(int a, int b, int c) {   // unsigned a bytes, signed b bytes
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(int a, int b, int c) {   // unsigned a and b bytes
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <int W0, int W1, int XS>
__device__ __forceinline__ xacc_t<XS> idot(const int (&c)[8], const XBlock& x) {
  int ah0 = 0, ah1 = 0, am0 = 0, am1 = 0, al0 = 0, al1 = 0;
#pragma unroll
  for (int k = W0; k < W1; k += 2) {
    ah0 = __dp4a(c[k], x.h[k], ah0);
    if (XS == 3) am0 = __dp4a(c[k], x.m[k], am0);
    al0 = XS == 3 ? __dp4a(c[k], x.l[k], al0) : dp4a_su(c[k], x.l[k], al0);
    ah1 = __dp4a(c[k + 1], x.h[k + 1], ah1);
    if (XS == 3) am1 = __dp4a(c[k + 1], x.m[k + 1], am1);
    al1 = XS == 3 ? __dp4a(c[k + 1], x.l[k + 1], al1) : dp4a_su(c[k + 1], x.l[k + 1], al1);
  }
  if constexpr (XS == 3) return (ah0 + ah1) * 4096 + ((am0 + am1) * 16 + (al0 + al1));
  else return (ah0 + ah1) * 256 + (al0 + al1);
}

// (codes . t) over one lane's 32 nibble codes straight from the four code words
// w: the low nibbles (elements 8k+0,2,4,6 of word k) are masked to bytes; the
// high nibbles (8k+1,3,5,7) stay in place as 16 x code (mask 0xF0), go through
// DP4A as unsigned bytes, and their sums are divided by 16 exactly at the end.
// The same integer as idot over nibble_bytes(w), one shift fewer per word.
template <int XS>
__device__ __forceinline__ xacc_t<XS> idot_nib(const uint4 w, const XBlock& x) {
  const uint32_t L = 0x0F0F0F0Fu, H = 0xF0F0F0F0u;
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  int hl = 0, ml = 0, ll = 0, hh = 0, mh = 0, lh = 0;   // slice x (low | high nibbles)
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const int lo = int(ws[k] & L), hi = int(ws[k] & H);
    hl = __dp4a(lo, x.h[2 * k], hl);
    hh = dp4a_us(hi, x.h[2 * k + 1], hh);
    if (XS == 3) {
      ml = __dp4a(lo, x.m[2 * k], ml);
      mh = dp4a_us(hi, x.m[2 * k + 1], mh);
      ll = __dp4a(lo, x.l[2 * k], ll);
      lh = dp4a_us(hi, x.l[2 * k + 1], lh);
    } else {
      ll = dp4a_su(lo, x.l[2 * k], ll);
      lh = dp4a_uu(hi, x.l[2 * k + 1], lh);
    }
  }
  // hh, mh, lh are 16 x the high nibbles' sums, exact multiples of 16
  if constexpr (XS == 3) return (hl * 4096 + hh * 256) + ((ml * 16 + mh) + (ll + (lh >> 4)));
  else return (hl * 256 + hh * 16) + (ll + (lh >> 4));
}

// even and odd nibbles of each code word as bytes: words 2k (elements 8k+0,2,4,6) and 2k+1 (8k+1,3,5,7)
__device__ __forceinline__ void nibble_bytes(const uint4 w, int (&c)[8]) {
  const uint32_t L = 0x0F0F0F0Fu;
  c[0] = int(w.x & L); c[1] = int((w.x >> 4) & L);
  c[2] = int(w.y & L); c[3] = int((w.y >> 4) & L);
  c[4] = int(w.z & L); c[5] = int((w.z >> 4) & L);
  c[6] = int(w.w & L); c[7] = int((w.w >> 4) & L);
}

template <int FMT> struct Pipe;

template <> struct Pipe<NT_Q8_0> {
  static constexpr int CB = 32, RB = 32 * 32 + 64;
  static constexpr bool NIB = false;                 // x bytes in natural order
  __device__ static int xbyte(int c) { return c; }
  // copy plan per row: code bytes per tile, then scale pieces (source, smem offset, bytes per tile, size)
  static constexpr int CODE_STRIDE = 1024, NPA = 4, NPB = 0;
  __device__ static const uint8_t* code_base(const QMat& m, int64_t e_row) { return m.q + e_row; }
  __device__ static void piece(const QMat& m, int64_t e_row, int i, const uint8_t*& src, int& off, int& stride,
                               int& size) {
    src = reinterpret_cast<const uint8_t*>(m.d + (e_row >> 5)) + i * 16;
    off = 1024 + i * 16;
    stride = 64;
    size = 16;
  }
  struct Frag {
    uint4 c0, c1;
    uint32_t d;
  };
  // Lanes 4..7 of every eight read the second 16 bytes of their 32 first: the
  // eight lanes of one phase of a 16-byte shared load then hit eight distinct
  // 16-byte bank slots (at a 32-byte lane stride lanes j and j + 4 would share one).
  __device__ static void load(const uint8_t* blk, int lane, Frag& f) {
    const int sw = (lane >> 2) & 1;
    const uint4 u0 = *reinterpret_cast<const uint4*>(blk + lane * 32 + 16 * sw);
    const uint4 u1 = *reinterpret_cast<const uint4*>(blk + lane * 32 + 16 * (sw ^ 1));
    f.c0 = sw ? u1 : u0;
    f.c1 = sw ? u0 : u1;
    f.d = *reinterpret_cast<const uint16_t*>(blk + 1024 + lane * 2);
  }
  template <int XS>
  __device__ static float compute(const Frag& f, int lane, const XBlock& x) {
    const int c[8] = {int(f.c0.x), int(f.c0.y), int(f.c0.z), int(f.c0.w),
                      int(f.c1.x), int(f.c1.y), int(f.c1.z), int(f.c1.w)};
    return __fmul_rn(h2f_bits(f.d), xacc_f(idot<0, 8, XS>(c, x)));
  }
};

__device__ __forceinline__ int nibble_xbyte(int c) { return (c & ~7) + ((c & 1) << 2) + ((c & 7) >> 1); }

template <> struct Pipe<NT_Q4_0> {
  static constexpr int CB = 16, RB = 32 * 16 + 64;
  static constexpr bool NIB = true;
  __device__ static int xbyte(int c) { return nibble_xbyte(c); }
  static constexpr int CODE_STRIDE = 512, NPA = 4, NPB = 0;
  __device__ static const uint8_t* code_base(const QMat& m, int64_t e_row) { return m.q + (e_row >> 1); }
  __device__ static void piece(const QMat& m, int64_t e_row, int i, const uint8_t*& src, int& off, int& stride,
                               int& size) {
    src = reinterpret_cast<const uint8_t*>(m.d + (e_row >> 5)) + i * 16;
    off = 512 + i * 16;
    stride = 64;
    size = 16;
  }
  struct Frag {
    uint4 w;
    uint32_t d;
  };
  __device__ static void load(const uint8_t* blk, int lane, Frag& f) {
    f.w = *reinterpret_cast<const uint4*>(blk + lane * 16);
    f.d = *reinterpret_cast<const uint16_t*>(blk + 512 + lane * 2);
  }
  template <int XS>
  __device__ static float compute(const Frag& f, int lane, const XBlock& x) {
    return __fmul_rn(h2f_bits(f.d), xacc_f(idot_nib<XS>(f.w, x) - xacc_t<XS>(8) * (x.t0 + x.t1)));
  }
};

// One K-quant sub-block (Q4_K / Q5_K): sx * (d sc_j * sum q x - dmin m_j * sum x),
// unit `lane` of the tile is sub-block j = lane % 8 of super-block lane / 8.
template <int XS>
__device__ __forceinline__ float kquant_unit_s(const uint4 meta, int lane, xacc_t<XS> dot, const XBlock& x) {
  uint32_t sc, mm;
  kquant_scale_min(meta, lane & 7, sc, mm);
  const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(&meta.x));   // (d, dmin)
  const float a = __fmul_rn(dm.x, float(sc));
  const float b = __fmul_rn(dm.y, float(mm));
  return __fmaf_rn(a, xacc_f(dot), -__fmul_rn(b, __int2float_rn(x.t0 + x.t1)));
}
template <int XS>
__device__ __forceinline__ float kquant_unit(const uint4 meta, int lane, const int (&c)[8], const XBlock& x) {
  return kquant_unit_s<XS>(meta, lane, idot<0, 8, XS>(c, x), x);
}

template <> struct Pipe<NT_Q4_K> {
  static constexpr int CB = 16, RB = 32 * 16 + 64;
  static constexpr bool NIB = true;
  __device__ static int xbyte(int c) { return nibble_xbyte(c); }
  static constexpr int CODE_STRIDE = 512, NPA = 4, NPB = 0;
  __device__ static const uint8_t* code_base(const QMat& m, int64_t e_row) { return m.q + (e_row >> 1); }
  __device__ static void piece(const QMat& m, int64_t e_row, int i, const uint8_t*& src, int& off, int& stride,
                               int& size) {
    src = m.meta + (e_row >> 8) * 16 + i * 16;
    off = 512 + i * 16;
    stride = 64;
    size = 16;
  }
  struct Frag {
    uint4 w, meta;
  };
  __device__ static void load(const uint8_t* blk, int lane, Frag& f) {
    f.w = *reinterpret_cast<const uint4*>(blk + lane * 16);
    f.meta = *reinterpret_cast<const uint4*>(blk + 512 + (lane >> 3) * 16);
  }
  template <int XS>
  __device__ static float compute(const Frag& f, int lane, const XBlock& x) {
    return kquant_unit_s<XS>(f.meta, lane, idot_nib<XS>(f.w, x), x);
  }
};

// Q5_K: the Q4_K unit with a fifth code bit per element from the unit's word H
// (byte i of H, bit v: code word v's byte i), OR-ed in at bit 4 of each byte.
template <> struct Pipe<NT_Q5_K> {
  static constexpr int CB = 16, RB = 32 * 16 + 128 + 64;
  static constexpr bool NIB = true;
  __device__ static int xbyte(int c) { return nibble_xbyte(c); }
  // 8 pieces of fifth-bit words (128 bytes per row and tile), 4 of super-block meta
  static constexpr int CODE_STRIDE = 512, NPA = 12, NPB = 0;
  __device__ static const uint8_t* code_base(const QMat& m, int64_t e_row) { return m.q + (e_row >> 1); }
  __device__ static void piece(const QMat& m, int64_t e_row, int i, const uint8_t*& src, int& off, int& stride,
                               int& size) {
    if (i < 8) {
      src = m.qh + (e_row >> 3) + i * 16;
      off = 512 + i * 16;
      stride = 128;
    } else {
      src = m.meta + (e_row >> 8) * 16 + (i - 8) * 16;
      off = 640 + (i - 8) * 16;
      stride = 64;
    }
    size = 16;
  }
  struct Frag {
    uint4 w, meta;
    uint32_t h;
  };
  __device__ static void load(const uint8_t* blk, int lane, Frag& f) {
    f.w = *reinterpret_cast<const uint4*>(blk + lane * 16);
    f.h = *reinterpret_cast<const uint32_t*>(blk + 512 + lane * 4);
    f.meta = *reinterpret_cast<const uint4*>(blk + 640 + (lane >> 3) * 16);
  }
  template <int XS>
  __device__ static float compute(const Frag& f, int lane, const XBlock& x) {
    int c[8];
    nibble_bytes(f.w, c);
    const uint32_t H = f.h, M = 0x10101010u;
    c[0] |= int((H << 4) & M);
    c[1] |= int((H << 3) & M);
    c[2] |= int((H << 2) & M);
    c[3] |= int((H << 1) & M);
    c[4] |= int(H & M);
    c[5] |= int((H >> 1) & M);
    c[6] |= int((H >> 2) & M);
    c[7] |= int((H >> 3) & M);
    return kquant_unit<XS>(f.meta, lane, c, x);
  }
};

template <> struct Pipe<NT_Q6_K> {
  static constexpr int CB = 16, RB = 32 * 16 + 256 + 64 + 16;
  static constexpr bool NIB = true;
  __device__ static int xbyte(int c) { return nibble_xbyte(c); }
  // 16 pieces of high-bit words and 4 of sub-block scales (16 bytes), 2 four-byte pieces of d
  static constexpr int CODE_STRIDE = 512, NPA = 20, NPB = 2;
  __device__ static const uint8_t* code_base(const QMat& m, int64_t e_row) { return m.q + (e_row >> 1); }
  __device__ static void piece(const QMat& m, int64_t e_row, int i, const uint8_t*& src, int& off, int& stride,
                               int& size) {
    if (i < 16) {
      src = m.qh + (e_row >> 2) + i * 16;
      off = 512 + i * 16;
      stride = 256;
      size = 16;
    } else if (i < 20) {
      src = m.meta + (e_row >> 4) + (i - 16) * 16;
      off = 768 + (i - 16) * 16;
      stride = 64;
      size = 16;
    } else {
      src = reinterpret_cast<const uint8_t*>(m.d + (e_row >> 8)) + (i - 20) * 4;
      off = 832 + (i - 20) * 4;
      stride = 8;
      size = 4;
    }
  }
  struct Frag {
    uint4 w;
    uint2 g;
    uint32_t sc2, db;
  };
  __device__ static void load(const uint8_t* blk, int lane, Frag& f) {
    f.w = *reinterpret_cast<const uint4*>(blk + lane * 16);
    f.g = *reinterpret_cast<const uint2*>(blk + 512 + lane * 8);
    f.sc2 = *reinterpret_cast<const uint16_t*>(blk + 768 + lane * 2);
    f.db = *reinterpret_cast<const uint16_t*>(blk + 832 + (lane >> 3) * 2);
  }
  template <int XS>
  __device__ static float compute(const Frag& f, int lane, const XBlock& x) {
    const uint4 w = f.w;
    const uint2 g = f.g;
    const uint32_t sc2 = f.sc2;
    const float d = h2f_bits(f.db);
    // device high-bit word G (one per 16 elements): byte j holds, for code words
    // W (elements 0..7) and W' (elements 8..15), hi(W,2j) at bits 4-5,
    // hi(W',2j) at bits 6-7, hi(W,2j+1) at bits 0-1, hi(W',2j+1) at bits 2-3
    const uint32_t M = 0x30303030u, L = 0x0F0F0F0Fu;
    const int c[8] = {int((w.x & L) | (g.x & M)),        int(((w.x >> 4) & L) | ((g.x << 4) & M)),
                      int((w.y & L) | ((g.x >> 2) & M)), int(((w.y >> 4) & L) | ((g.x << 2) & M)),
                      int((w.z & L) | (g.y & M)),        int(((w.z >> 4) & L) | ((g.y << 4) & M)),
                      int((w.w & L) | ((g.y >> 2) & M)), int(((w.w >> 4) & L) | ((g.y << 2) & M))};
    const xacc_t<XS> s0 = idot<0, 4, XS>(c, x) - xacc_t<XS>(32) * x.t0;
    const xacc_t<XS> s1 = idot<4, 8, XS>(c, x) - xacc_t<XS>(32) * x.t1;
    const float sc0 = float(int8_t(sc2 & 0xFF)), sc1 = float(int8_t(sc2 >> 8));
    return __fmul_rn(d, __fmaf_rn(sc0, xacc_f(s0), __fmul_rn(sc1, xacc_f(s1))));
  }
};

__device__ __forceinline__ void cp16z(uint32_t dst, const void* src, uint32_t n) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

// Tiles of one warp: its row groups g0, g0 + stride, ... (g0 = warp * ncta + cta,
// stride = ncta * NW, so consecutive groups land on different CTAs and every SM
// gets an equal share), each in kiters column tiles.  (Measured on GB300:
// cutting the groups into contiguous per-CTA shares split evenly over the warps
// at tile granularity, pieces of a group added in shared memory, was slower at
// every shape, even where whole groups leave a last round to a tenth of the warps.)
struct WarpTiles {
  int64_t g0, stride;
  int ntiles;
};
__device__ __forceinline__ WarpTiles warp_tiles(int64_t nrows, int R, int kiters, int warp, int nw, int cta,
                                                int ncta) {
  WarpTiles w;
  const int64_t ngroups = (nrows + R - 1) / R;
  w.g0 = int64_t(warp) * ncta + cta;
  w.stride = int64_t(ncta) * nw;
  w.ntiles = w.g0 < ngroups ? int((ngroups - 1 - w.g0) / w.stride + 1) * kiters : 0;
  return w;
}

// Copy cursor of one warp over its tiles.  Every lane issues the same copies
// for every tile, so there are no divergent branches: 16 (or twice 16) code bytes
// of each of the R rows (a row past the matrix copies zero bytes, src-size 0,
// from a valid address, so its products are zero) and its share of the rows'
// scale pieces (16-byte pieces, and 4-byte ones for Q6_K's d; a lane slot
// without a piece of its own is a predicated-off copy).  Sources advance by a fixed stride
// per tile; the per-lane plan is rebuilt at each new row group.  One cursor per
// warp serves the whole launch: the copies issued before the dependency wait,
// those issued during the x staging and those of the tile loop.
template <int FMT, int R, int S>
struct PipeCursor {
  using P = Pipe<FMT>;
  static constexpr int NA = (R * P::NPA + 31) / 32;
  static constexpr int NB = P::NPB ? (R * P::NPB + 31) / 32 : 1;
  const uint8_t* code[R];
  uint32_t csz[R];
  const uint8_t* asrc[NA];
  uint32_t aoff[NA], aon[NA];
  int astr[NA];
  const uint8_t* bsrc[NB];
  uint32_t boff[NB], bon[NB];
  int bstr[NB];
  int64_t grp, stride;
  int left, it, kiters;
  bool fresh;
  uint32_t dst, ring0, ring_end;

  __device__ __forceinline__ void init(const WarpTiles& w, int kiters_, uint32_t wring_s) {
    grp = w.g0;
    stride = w.stride;
    left = w.ntiles;
    it = 0;
    kiters = kiters_;
    fresh = true;
    ring0 = dst = wring_s;
    ring_end = wring_s + uint32_t(S * R * P::RB);
  }

  __device__ __forceinline__ void setup(const GemvArgs& a, int64_t nrows, int lane) {
    const int nlive = int(nrows - grp * R < R ? nrows - grp * R : R);
    int seg[R];
    int64_t e[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
      int sg = 0;
      int64_t lr = 0;
      map_row(a, grp * R + (r < nlive ? r : 0), sg, lr);
      seg[r] = sg;
      e[r] = lr * a.seg[0].cols + a.col0;
      code[r] = P::code_base(a.seg[sg], e[r]) + lane * 16;
      csz[r] = r < nlive ? 16u : 0u;
    }
    // piece slot k of this lane: piece p = lane + 32k of the group's R rows; a slot
    // past the live pieces copies nothing (its plan points at a piece of row 0)
#pragma unroll
    for (int k = 0; k < NA; k++) {
      const int p = lane + 32 * k;
      int r = p / P::NPA, i = p - r * P::NPA;
      aon[k] = p < R * P::NPA && r < nlive;
      if (!aon[k]) {
        r = 0;
        i = p % P::NPA;
      }
      int sg = seg[0];
      int64_t er = e[0];
#pragma unroll
      for (int rr = 1; rr < R; rr++)
        if (r == rr) {
          sg = seg[rr];
          er = e[rr];
        }
      const uint8_t* src;
      int off, str, size;
      P::piece(a.seg[sg], er, i, src, off, str, size);
      asrc[k] = src;
      aoff[k] = uint32_t(off + r * P::RB);
      astr[k] = str;
    }
    if (P::NPB) {
      constexpr int npb = P::NPB ? P::NPB : 1;
#pragma unroll
      for (int k = 0; k < NB; k++) {
        const int p = lane + 32 * k;
        int r = p / npb, i = p - r * npb;
        bon[k] = p < R * P::NPB && r < nlive;
        if (!bon[k]) {
          r = 0;
          i = p % npb;
        }
        int sg = seg[0];
        int64_t er = e[0];
#pragma unroll
        for (int rr = 1; rr < R; rr++)
          if (r == rr) {
            sg = seg[rr];
            er = e[rr];
          }
        const uint8_t* src;
        int off, str, size;
        P::piece(a.seg[sg], er, P::NPA + i, src, off, str, size);
        bsrc[k] = src;
        boff[k] = uint32_t(off + r * P::RB);
        bstr[k] = str;
      }
    }
  }

  template <bool ISSUE>
  __device__ __forceinline__ void step(const GemvArgs& a, int64_t nrows, int lane) {
    if (left > 0) {
      if (fresh) {
        setup(a, nrows, lane);
        fresh = false;
      }
      if (ISSUE) {
#pragma unroll
        for (int r = 0; r < R; r++) {
          // lane l copies bytes [16 l, 16 l + 16) of the row's codes (and, with 32
          // code bytes per unit, [512 + 16 l, ...)): each copy instruction of the
          // warp reads 512 contiguous bytes, whole 32-byte sectors
          const uint32_t d = dst + uint32_t(r * P::RB + lane * 16);
          cp16z(d, code[r], csz[r]);
          if (P::CB == 32) cp16z(d + 512, code[r] + 512, csz[r]);
        }
#pragma unroll
        for (int k = 0; k < NA; k++) cp16_if(aon[k], dst + aoff[k], asrc[k]);
        if (P::NPB) {
#pragma unroll
          for (int k = 0; k < NB; k++) cp4_if(bon[k], dst + boff[k], bsrc[k]);
        }
      }
#pragma unroll
      for (int r = 0; r < R; r++) code[r] += P::CODE_STRIDE;
#pragma unroll
      for (int k = 0; k < NA; k++) asrc[k] += astr[k];
      if (P::NPB) {
#pragma unroll
        for (int k = 0; k < NB; k++) bsrc[k] += bstr[k];
      }
      dst += uint32_t(R * P::RB);
      if (dst == ring_end) dst = ring0;
      --left;
      if (++it == kiters) {
        it = 0;
        grp += stride;
        fresh = true;
      }
    }
    if (ISSUE) cp_commit();   // one group per tile, empty past the end, so the wait_group counts stay aligned
  }
};

template <int FMT, int R, int S>
__host__ __device__ constexpr size_t pipe_ring_bytes(int nw) {
  return size_t(nw) * S * R * Pipe<FMT>::RB;
}

// Ring bytes of one warp: SLICE when given (a fixed per-warp slice shared by
// GEMVs of several formats), else exactly S tiles of R rows.
template <int FMT, int R, int S, int SLICE>
__host__ __device__ constexpr size_t pipe_slice() {
  return SLICE ? size_t(SLICE) : size_t(S) * R * Pipe<FMT>::RB;
}

// Issues the copies of the cursor's next n tiles (one commit group each).
template <class Cur>
__device__ __forceinline__ void pipe_issue(Cur& cur, const GemvArgs& a, int64_t nrows, int n) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int t = 0; t < n; t++) cur.template step<true>(a, nrows, lane);
}

// Converts one lane's eight elements of a 32-column block: columns
// [256 p, 256 p + 256) of the window are eight blocks, four lanes per block,
// eight consecutive elements per lane.  Per block: sx = max|x|/T (T = 32512 or
// 520192), t = round(x/sx) split into the slices, the sums T0, T1 of t over
// elements 0..15 and 16..31, and with norm the sum of squares (each lane's
// eight in element order, then the four lanes as (l0 + l1) + (l2 + l3)).
// |t| <= T needs no clamp: |x| <= max|x|, and x (T / max|x|) with its two
// roundings exceeds T by less than T 2^-22 < 1/2 (a NaN x, which the maximum
// skips, converts to 0).  Two slices are the two bytes of t, gathered with byte
// permutes; three slices are rounded as 4096 h + 16 m + l.
template <int FMT, int XS>
__device__ __forceinline__ void stage_convert(float4 f0, float4 f1, int p, uint8_t* xq, bool norm) {
  using P = Pipe<FMT>;
  const int lane = threadIdx.x & 31, q = lane & 3;          // q: eighth of the block
  const int blk = p * 8 + (lane >> 2);
  const float v[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; j++) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  float sq = 0.f;
  if (norm) {
    sq = __fmul_rn(v[0], v[0]);
#pragma unroll
    for (int j = 1; j < 8; j++) sq = __fmaf_rn(v[j], v[j], sq);
    sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, 1));   // (l0 + l1), (l2 + l3)
    sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, 2));   // then their sum
  }
  constexpr int kT = XS == 3 ? 520192 : 32512;   // 127 * 4096, 127 * 256
  const float inv = amax > 0.f ? float(kT) / amax : 0.f;
  uint8_t* dst = xq + size_t(blk) * x_unit<XS>();
  int ts = 0;
  if constexpr (XS == 2) {
    int t[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      t[j] = __float2int_rn(__fmul_rn(v[j], inv));
      ts += t[j];
    }
    // the lane's eight bytes in the format's order: elements e0..e3, then e4..e7
    constexpr int e1 = P::NIB ? 2 : 1, e2 = P::NIB ? 4 : 2, e3 = P::NIB ? 6 : 3;
    constexpr int e4 = P::NIB ? 1 : 4, e5 = P::NIB ? 3 : 5, e6 = P::NIB ? 5 : 6;
    auto bytes4 = [](int a, int b, int c, int d, unsigned sel) {   // byte sel of a, b, c, d
      return __byte_perm(__byte_perm(a, b, sel), __byte_perm(c, d, sel), 0x5410);
    };
    const uint32_t h0 = bytes4(t[0], t[e1], t[e2], t[e3], 0x0051), h1 = bytes4(t[e4], t[e5], t[e6], t[7], 0x0051);
    const uint32_t l0 = bytes4(t[0], t[e1], t[e2], t[e3], 0x0040), l1 = bytes4(t[e4], t[e5], t[e6], t[7], 0x0040);
    *reinterpret_cast<uint2*>(dst + q * 8) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(dst + 32 + q * 8) = make_uint2(l0, l1);
  } else {
    uint32_t hw[2] = {0, 0}, mw[2] = {0, 0}, lw[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 8; j++) {
      int t = __float2int_rn(__fmul_rn(v[j], inv));
      t = max(-kT, min(kT, t));
      ts += t;
      const int h = (t + 2048) >> 12;   // |h| <= 127
      const int r = t - 4096 * h;       // -2048 .. 2047
      const int m = r >> 4;             // -128 .. 127
      const int l = r & 15;             // 0 .. 15
      const int b = P::xbyte(j);        // position inside this lane's eight bytes (the format's order)
      hw[b >> 2] |= uint32_t(uint8_t(int8_t(h))) << (8 * (b & 3));
      mw[b >> 2] |= uint32_t(uint8_t(int8_t(m))) << (8 * (b & 3));
      lw[b >> 2] |= uint32_t(uint8_t(int8_t(l))) << (8 * (b & 3));
    }
    *reinterpret_cast<uint2*>(dst + q * 8) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(dst + 32 + q * 8) = make_uint2(mw[0], mw[1]);
    *reinterpret_cast<uint2*>(dst + 64 + q * 8) = make_uint2(lw[0], lw[1]);
  }
  const int t01 = ts + __shfl_xor_sync(0xffffffffu, ts, 1);   // lanes q = 0,1: elements 0..15; q = 2,3: 16..31
  const int t_hi = __shfl_xor_sync(0xffffffffu, t01, 2);
  if (q == 0)
    *reinterpret_cast<uint4*>(dst + 32 * XS) =
        make_uint4(__float_as_uint(amax / float(kT)), uint32_t(t01), uint32_t(t_hi), __float_as_uint(sq));
}

// RMSNorm factor rsqrt(mean(x^2) + eps) from the staged per-block squares,
// summed by one warp's lanes in a fixed order (1 without norm).
template <int XS>
__device__ __forceinline__ float x_scale_n(int norm, int64_t ncols, float eps, const uint8_t* xq) {
  if (!norm) return 1.0f;
  const int lane = threadIdx.x & 31;
  const int units = int(ncols / 32);
  constexpr int U = x_unit<XS>(), SQ = 32 * XS + 12;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  for (int b = lane; b < units; b += 128) {
    s0 = __fadd_rn(s0, *reinterpret_cast<const float*>(xq + size_t(b) * U + SQ));
    if (b + 32 < units) s1 = __fadd_rn(s1, *reinterpret_cast<const float*>(xq + size_t(b + 32) * U + SQ));
    if (b + 64 < units) s2 = __fadd_rn(s2, *reinterpret_cast<const float*>(xq + size_t(b + 64) * U + SQ));
    if (b + 96 < units) s3 = __fadd_rn(s3, *reinterpret_cast<const float*>(xq + size_t(b + 96) * U + SQ));
  }
  float t = __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
#pragma unroll
  for (int o = 16; o; o >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
  return rsqrtf(t / float(ncols) + eps);
}
template <int XS>
__device__ __forceinline__ float x_scale(const GemvArgs& a, const uint8_t* xq) {
  return x_scale_n<XS>(a.norm, a.ncols, a.eps, xq);
}

// Whole window staged up front by the CTA's NW warps (256-column pass p by warp
// p % NW); each warp loads up to four of its passes before converting any, so
// the staging costs one memory latency per 16384 columns.  between() runs
// after the first loads are issued and before they are used (the caller issues
// weight copies there, behind the x loads).  (Measured on GB300: loading up to
// eight passes at once, one latency for any window, made the 70B step 1%
// slower; CTA pairs launched as clusters of two, each converting half the
// passes into both CTAs' shared memory, made it 1.4% slower and the 8B step 7%.)
struct NoOp {
  __device__ __forceinline__ void operator()() const {}
};
// The same for the window x[0, ncols) into xq, without the closing barrier;
// norm: keep the per-block sums of squares of an RMSNorm.
template <int FMT, int NW, int XS, class F>
__device__ __forceinline__ void stage_x_from(const float* x, int64_t ncols, uint8_t* xq, bool norm, F between) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, np = int(ncols / 256);
  constexpr int kPasses = 4;
  bool first = true;
  for (int p0 = warp; p0 < np || first; p0 += kPasses * NW) {
    float4 f[kPasses][2];
#pragma unroll
    for (int i = 0; i < kPasses; i++) {
      const int p = p0 + i * NW;
      if (p < np) {
        const float4* src = reinterpret_cast<const float4*>(x + size_t(p) * 256 + lane * 8);
        f[i][0] = __ldcg(src);
        f[i][1] = __ldcg(src + 1);
      }
    }
    if (first) {
      between();
      first = false;
    }
#pragma unroll
    for (int i = 0; i < kPasses; i++)
      if (p0 + i * NW < np) stage_convert<FMT, XS>(f[i][0], f[i][1], p0 + i * NW, xq, norm);
  }
}

template <int FMT, int NW, int XS, class F = NoOp>
__device__ __forceinline__ void stage_x(const GemvArgs& a, uint8_t* xq, F between = F()) {
  stage_x_from<FMT, NW, XS>(a.x + a.col0, a.ncols, xq, a.norm != 0, between);
  __syncthreads();
}


// Running top-2 of the rows a warp finished (EPI_LOGITS).
struct Top2 {
  float best = -INFINITY, second = -INFINITY;
  int best_i = 0x7fffffff;
};

// The GEMV of the calling warp's groups w: the tile loop and the row-group
// epilogues.  cur is the warp's copy cursor with its first S-1 tiles issued
// (ring slices at wring); x is staged in xq and `scale` is the RMS factor.
// Operands are read one tile ahead: the next tile's codes, scales and x block
// come from shared memory while the cursor issues copies, before they are used.
template <int FMT, int R, int S, int EPI, int NW>
__device__ __forceinline__ void pipe_loop_w(const GemvArgs& a, int64_t nrows, const WarpTiles& w, uint8_t* xq,
                                            const uint8_t* wring, float scale, PipeCursor<FMT, R, S>& cur,
                                            Top2& t2) {
  static_assert(S >= 3, "the loop keeps one tile's operands ahead");
  using P = Pipe<FMT>;
  constexpr int XS = x_slices(EPI), XU = x_unit<XS>();
  const int lane = threadIdx.x & 31;
  const int kiters = int(a.ncols / 1024);
  if (w.ntiles == 0) return;
  float acc[R];
#pragma unroll
  for (int r = 0; r < R; r++) acc[r] = 0.f;
  int64_t c_grp = w.g0;
  int c_it = 0;
  const uint8_t* rd = wring;                               // slot of the tile being decoded
  const uint8_t* const rd_end = wring + S * R * P::RB;
  const uint8_t* xp = xq + size_t(lane) * XU;             // this lane's x block of the tile
  typename P::Frag fr[R];
  XBlock xb;
  cp_wait<S - 2>();   // tile 0 has landed
  __syncwarp();
#pragma unroll
  for (int r = 0; r < R; r++) P::load(rd + r * P::RB, lane, fr[r]);
  load_xblock<XS>(xp, xb);
#pragma unroll 1
  for (int t = 0; t < w.ntiles; t++) {
#pragma unroll
    for (int r = 0; r < R; r++) acc[r] = __fmaf_rn(xb.sx, P::template compute<XS>(fr[r], lane, xb), acc[r]);   // dead rows read zeros
    rd += R * P::RB;
    if (rd == rd_end) rd = wring;
    xp += 32 * XU;
    if (++c_it == kiters) {
      // ---- row group done: transposed warp reduction, epilogue --------------
      c_it = 0;
      xp = xq + size_t(lane) * XU;
      float kk = warp_reduce_rows<R>(acc, lane);
#pragma unroll
      for (int r = 0; r < R; r++) acc[r] = 0.f;
      kk = __fmul_rn(kk, scale);
      epilogue<R, EPI>(a, c_grp, nrows, lane, kk, t2.best, t2.best_i, t2.second);
      c_grp += w.stride;
    }
    cp_wait<S - 3>();   // tile t + 1 has landed
    __syncwarp();       // ... every lane's copies; the slot of tile t - 1 is free
#pragma unroll
    for (int r = 0; r < R; r++) P::load(rd + r * P::RB, lane, fr[r]);
    load_xblock<XS>(xp, xb);
    cur.template step<true>(a, nrows, lane);   // tile t + S - 1
  }
  cp_wait<0>();
  __syncwarp();
}

template <int FMT, int R, int S, int EPI, int NW>
__global__ void __launch_bounds__(NW * 32, 16 / NW) k_gemv_pipe(const __grid_constant__ GemvArgs a,
                                                                const int64_t nrows) {
  constexpr int E = S - 1 < kPipeEarly ? S - 1 : kPipeEarly;
  extern __shared__ float4 smem4[];
  uint8_t* xq = reinterpret_cast<uint8_t*>(smem4);
  constexpr int XS = x_slices(EPI);
  uint8_t* ring = xq + size_t(a.ncols / 32) * x_unit<XS>();
  const int warp = threadIdx.x >> 5, kiters = int(a.ncols / 1024);
  const WarpTiles w = warp_tiles(nrows, R, kiters, warp, NW, blockIdx.x, gridDim.x);
  uint8_t* wring = ring + size_t(warp) * pipe_slice<FMT, R, S, 0>();
  PipeCursor<FMT, R, S> cur;
  cur.init(w, kiters, smem_addr(wring));
  pipe_issue(cur, a, nrows, E);   // weights only: before the producer of x has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  stage_x<FMT, NW, XS>(a, xq, [&] { pipe_issue(cur, a, nrows, S - 1 - E); });
  const float scale = x_scale<XS>(a, xq);
  // the next kernel may start its own weight prefetch on SMs this grid frees;
  // it waits for this grid to finish before it reads anything this grid writes
  asm volatile("griddepcontrol.launch_dependents;");
  Top2 t2;
  pipe_loop_w<FMT, R, S, EPI, NW>(a, nrows, w, xq, wring, scale, cur, t2);
  if (EPI == EPI_LOGITS) cta_top2<NW>(a, blockIdx.x, t2.best, t2.best_i, t2.second);
}

// Two GEMVs over the same x in one launch: rows [0, n1) of a1 in format F1 and
// rows [0, n2) of a2 in F2 (both 4-bit-nibble formats, so one staged x serves
// both).  The group indices of the two (R1 rows per a1 group, R2 per a2 group)
// run on as one range over the warps, a1's first; each warp works through its
// a1 groups, then its a2 groups, with each format's own ring depth in one
// per-warp slice.  Used for a Q4_K Q/K GEMV (four rows per warp, each x read
// shared by four rows) with a Q6_K V GEMV (one row per warp: at 70B widths the
// 2304 Q/K groups leave 128 of the 2432 warps free, and one-row V groups spread
// the V rows' second round over 896 warps instead of two-row groups over 384,
// so fewer warps run on alone at the end; 70B step 0.6% faster than two-row V
// groups).  (Measured on GB300: cutting the V groups into column parts spread
// over the warps of a CTA, added in shared memory, balanced the launch and made
// the GEMVs 2.5% faster, yet the 70B decode step 0.4% slower.)
template <int F1, int F2, int R1, int R2, int S1, int S2, int EPI, int NW>
__global__ void __launch_bounds__(NW * 32, 16 / NW) k_gemv_pipe2(const __grid_constant__ GemvArgs a1,
                                                       const __grid_constant__ GemvArgs a2, const int64_t n1,
                                                       const int64_t n2) {
  static_assert(F1 != NT_Q8_0 && F2 != NT_Q8_0, "one staged x: nibble formats only");
  constexpr int SLICE = int(pipe_slice<F1, R1, S1, 0>() > pipe_slice<F2, R2, S2, 0>() ? pipe_slice<F1, R1, S1, 0>()
                                                                                       : pipe_slice<F2, R2, S2, 0>());
  extern __shared__ float4 smem4[];
  uint8_t* xq = reinterpret_cast<uint8_t*>(smem4);
  constexpr int XS = x_slices(EPI);
  uint8_t* ring = xq + size_t(a1.ncols / 32) * x_unit<XS>();
  const int warp = threadIdx.x >> 5, kiters = int(a1.ncols / 1024);
  const int64_t G1 = (n1 + R1 - 1) / R1, G = G1 + (n2 + R2 - 1) / R2;
  WarpTiles w1, w2;
  w1.g0 = int64_t(warp) * gridDim.x + blockIdx.x;
  w1.stride = int64_t(gridDim.x) * NW;
  const int64_t c1 = w1.g0 < G1 ? (G1 - 1 - w1.g0) / w1.stride + 1 : 0;
  w1.ntiles = int(c1) * kiters;
  const int64_t g2 = w1.g0 + c1 * w1.stride;            // first combined index past a1
  w2.g0 = g2 - G1;
  w2.stride = w1.stride;
  w2.ntiles = g2 < G ? int((G - 1 - g2) / w2.stride + 1) * kiters : 0;
  uint8_t* wring = ring + size_t(warp) * SLICE;
  // a1's copies from the start; a2's once the warp's a1 groups are done (on a
  // drained ring; one cursor live at a time keeps the loops within the registers)
  PipeCursor<F1, R1, S1> cur1;
  constexpr int E1 = S1 - 1 < kPipeEarly ? S1 - 1 : kPipeEarly;
  cur1.init(w1, kiters, smem_addr(wring));
  pipe_issue(cur1, a1, n1, E1);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  stage_x<F1, NW, XS>(a1, xq, [&] { pipe_issue(cur1, a1, n1, S1 - 1 - E1); });
  const float scale = x_scale<XS>(a1, xq);
  asm volatile("griddepcontrol.launch_dependents;");
  Top2 t2;
  pipe_loop_w<F1, R1, S1, EPI, NW>(a1, n1, w1, xq, wring, scale, cur1, t2);
  PipeCursor<F2, R2, S2> cur2;
  cur2.init(w2, kiters, smem_addr(wring));
  pipe_issue(cur2, a2, n2, S2 - 1);
  pipe_loop_w<F2, R2, S2, EPI, NW>(a2, n2, w2, xq, wring, scale, cur2, t2);
  if (EPI == EPI_LOGITS) cta_top2<NW>(a1, blockIdx.x, t2.best, t2.best_i, t2.second);
}

// ---- multi-token launches (the verification of a speculative cycle) ---------
// One GEMV for up to kBatchMax tokens with the same weights: each warp's weight
// tiles are copied once and multiplied by every token's staged x.  Every
// token's result is bit for bit the single-token kernel's with the same R and
// epilogue: the same x staging and RMS factor, the same per-lane tile order, the
// same warp reduction and epilogue.
constexpr int kBatchMax = 4;
struct BatchTok {
  const float* x = nullptr;      // the token's input
  float* y = nullptr;            // the token's output (EPI_QKV: its q rows; EPI_ADD: its residual; EPI_SWIGLU: u)
  const int32_t* pos = nullptr;  // the token's position counter (EPI_QKV)
};
struct GemvBatch {
  BatchTok tok[kBatchMax];
  int32_t n = 0;
};

template <int FMT, int R, int S, int EPI, int NW>
__global__ void __launch_bounds__(NW * 32, 16 / NW) k_gemv_pipe_batch(const __grid_constant__ GemvArgs a,
                                                                      const __grid_constant__ GemvBatch b,
                                                                      const int64_t nrows) {
  using P = Pipe<FMT>;
  constexpr int E = S - 1 < kPipeEarly ? S - 1 : kPipeEarly;
  constexpr int XS = x_slices(EPI), XU = x_unit<XS>();
  extern __shared__ float4 smem4[];
  uint8_t* xq = reinterpret_cast<uint8_t*>(smem4);
  const size_t xbytes = size_t(a.ncols / 32) * XU;   // one token's staged x (a multiple of 16 bytes)
  uint8_t* ring = xq + size_t(b.n) * xbytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, kiters = int(a.ncols / 1024);
  const WarpTiles w = warp_tiles(nrows, R, kiters, warp, NW, blockIdx.x, gridDim.x);
  uint8_t* wring = ring + size_t(warp) * pipe_slice<FMT, R, S, 0>();
  PipeCursor<FMT, R, S> cur;
  cur.init(w, kiters, smem_addr(wring));
  pipe_issue(cur, a, nrows, E);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int j = 0; j < b.n; j++) {
    if (j == 0)
      stage_x_from<FMT, NW, XS>(b.tok[0].x + a.col0, a.ncols, xq, a.norm != 0,
                                   [&] { pipe_issue(cur, a, nrows, S - 1 - E); });
    else stage_x_from<FMT, NW, XS>(b.tok[j].x + a.col0, a.ncols, xq + size_t(j) * xbytes, a.norm != 0, NoOp());
  }
  __syncthreads();
  float scale[kBatchMax];
#pragma unroll
  for (int j = 0; j < kBatchMax; j++) scale[j] = j < b.n ? x_scale_n<XS>(a.norm, a.ncols, a.eps, xq + size_t(j) * xbytes) : 1.f;
  asm volatile("griddepcontrol.launch_dependents;");
  if (w.ntiles == 0) return;

  float acc[kBatchMax][R];
#pragma unroll
  for (int j = 0; j < kBatchMax; j++)
#pragma unroll
    for (int r = 0; r < R; r++) acc[j][r] = 0.f;
  float best = -INFINITY, second = -INFINITY;
  int best_i = 0x7fffffff;
  int64_t c_grp = w.g0;
  int c_it = 0;
  const uint8_t* rd = wring;
  const uint8_t* const rd_end = wring + S * R * P::RB;
  const uint8_t* xp = xq + size_t(lane) * XU;   // this lane's x block of the tile (token 0)
  typename P::Frag fr[R];
  cp_wait<S - 2>();
  __syncwarp();
#pragma unroll
  for (int r = 0; r < R; r++) P::load(rd + r * P::RB, lane, fr[r]);
#pragma unroll 1
  for (int t = 0; t < w.ntiles; t++) {
#pragma unroll
    for (int j = 0; j < kBatchMax; j++) {
      if (j < b.n) {
        XBlock xb;
        load_xblock<XS>(xp + size_t(j) * xbytes, xb);
#pragma unroll
        for (int r = 0; r < R; r++) acc[j][r] = __fmaf_rn(xb.sx, P::template compute<XS>(fr[r], lane, xb), acc[j][r]);
      }
    }
    rd += R * P::RB;
    if (rd == rd_end) rd = wring;
    xp += 32 * XU;
    if (++c_it == kiters) {
      c_it = 0;
      xp = xq + size_t(lane) * XU;
#pragma unroll
      for (int j = 0; j < kBatchMax; j++) {
        if (j < b.n) {
          float kk = warp_reduce_rows<R>(acc[j], lane);
          kk = __fmul_rn(kk, scale[j]);
          epilogue_to<R, EPI>(a, b.tok[j].y, b.tok[j].pos, c_grp, nrows, lane, kk, best, best_i, second);
        }
#pragma unroll
        for (int r = 0; r < R; r++) acc[j][r] = 0.f;
      }
      c_grp += w.stride;
    }
    cp_wait<S - 3>();
    __syncwarp();
#pragma unroll
    for (int r = 0; r < R; r++) P::load(rd + r * P::RB, lane, fr[r]);
    cur.template step<true>(a, nrows, lane);
  }
  cp_wait<0>();
  __syncwarp();
}

inline size_t pipe_x_bytes(int64_t cols, int epi) {
  return size_t(cols / 32) * size_t(x_slices(epi) == 3 ? x_unit<3>() : x_unit<2>());
}
inline int pipe_row_bytes(int fmt) {
  switch (fmt) {
    case NT_Q8_0: return Pipe<NT_Q8_0>::RB;
    case NT_Q4_0: return Pipe<NT_Q4_0>::RB;
    case NT_Q4_K: return Pipe<NT_Q4_K>::RB;
    case NT_Q5_K: return Pipe<NT_Q5_K>::RB;
    default: return Pipe<NT_Q6_K>::RB;
  }
}

template <int FMT, int R, int S, int EPI, int NW>
cudaError_t launch_gemv_pipe_t(const GemvArgs& a, cudaStream_t s, bool pdl, int* grid_used) {
  const int64_t nrows = gemv_logical_rows(a);
  const size_t smem = pipe_x_bytes(a.ncols, EPI) + size_t(NW) * S * R * Pipe<FMT>::RB;
  if (smem > size_t(kPipeMaxSmem)) return cudaErrorInvalidValue;
  auto kern = k_gemv_pipe<FMT, R, S, EPI, NW>;
  static const KernelSetup setup = kernel_setup(kern, kPipeMaxSmem);
  if (setup.err != cudaSuccess) return setup.err;
  const int s_sms = setup.sms;
  thread_local size_t s_occ_smem = ~size_t(0);   // occupancy of the last shared-memory size (per thread)
  thread_local int s_occ = 0;
  if (s_occ_smem != smem) {
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NW * 32, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    s_occ = occ;
    s_occ_smem = smem;
  }
  // one wave, no more CTAs than the work fills (but at least one per SM while
  // there are groups for it); groups are spread warp-major over the CTAs
  int64_t grid = int64_t(s_sms) * s_occ;
  const int64_t groups = (nrows + R - 1) / R;
  int64_t want = (groups + NW - 1) / NW;
  if (want < s_sms) want = groups < s_sms ? groups : s_sms;
  if (grid > want) grid = want;
  if (grid > a.max_grid) grid = a.max_grid;
  if (grid < 1) grid = 1;
  if (grid_used) *grid_used = int(grid);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(NW * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, nrows);
}

template <int FMT, int R, int S, int NW>
cudaError_t launch_gemv_pipe_rs(const GemvArgs& a, int epi, cudaStream_t s, bool pdl, int* grid_used) {
  switch (epi) {
    case EPI_STORE: return launch_gemv_pipe_t<FMT, R, S, EPI_STORE, NW>(a, s, pdl, grid_used);
    case EPI_ADD: return launch_gemv_pipe_t<FMT, R, S, EPI_ADD, NW>(a, s, pdl, grid_used);
    case EPI_QKV: return launch_gemv_pipe_t<FMT, R, S, EPI_QKV, NW>(a, s, pdl, grid_used);
    case EPI_SWIGLU: return launch_gemv_pipe_t<FMT, R, S, EPI_SWIGLU, NW>(a, s, pdl, grid_used);
    case EPI_LOGITS: return launch_gemv_pipe_t<FMT, R, S, EPI_LOGITS, NW>(a, s, pdl, grid_used);
  }
  return cudaErrorInvalidValue;
}

// Formats with a four-row kernel (the 4-bit ones; the shapes' chooser takes four
// rows for no other).
template <int FMT>
constexpr bool kFourRows = FMT == NT_Q4_0 || FMT == NT_Q4_K || FMT == NT_Q5_K;

template <int FMT, int R, int S, int EPI>
cudaError_t launch_gemv_batch_t(const GemvArgs& a, const GemvBatch& b, cudaStream_t s, bool pdl) {
  constexpr int NW = kPipeWarps;
  const int64_t nrows = gemv_logical_rows(a);
  const size_t smem = size_t(b.n) * pipe_x_bytes(a.ncols, EPI) + size_t(NW) * S * R * Pipe<FMT>::RB;
  if (smem > size_t(kPipeMaxSmem) || b.n < 1 || b.n > kBatchMax) return cudaErrorInvalidValue;
  auto kern = k_gemv_pipe_batch<FMT, R, S, EPI, NW>;
  static const KernelSetup setup = kernel_setup(kern, kPipeMaxSmem);
  if (setup.err != cudaSuccess) return setup.err;
  // the grid of the single-token launch: one CTA per SM (capped by the groups)
  const int64_t groups = (nrows + R - 1) / R;
  int64_t want = (groups + NW - 1) / NW;
  if (want < setup.sms) want = groups < setup.sms ? groups : setup.sms;
  int64_t grid = setup.sms;
  if (grid > want) grid = want;
  if (grid > a.max_grid) grid = a.max_grid;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(NW * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, b, nrows);
}

// Multi-token launch of one format: R fixed by the caller (the single-token
// launch's), ring depth 3 or 4 (what fits beside the n staged x).
template <int FMT>
cudaError_t launch_gemv_batch_fmt(const GemvArgs& a, int epi, int R, int S, const GemvBatch& b, cudaStream_t s,
                                  bool pdl) {
#define NT_BATCH_EPI(RR, SS)                                                                  \
  switch (epi) {                                                                              \
    case EPI_ADD: return launch_gemv_batch_t<FMT, RR, SS, EPI_ADD>(a, b, s, pdl);             \
    case EPI_QKV: return launch_gemv_batch_t<FMT, RR, SS, EPI_QKV>(a, b, s, pdl);             \
    case EPI_SWIGLU: return launch_gemv_batch_t<FMT, RR, SS, EPI_SWIGLU>(a, b, s, pdl);       \
    case EPI_STORE: return launch_gemv_batch_t<FMT, RR, SS, EPI_STORE>(a, b, s, pdl);         \
  }
  if (R == 4) {
    if constexpr (kFourRows<FMT>) {
      if (S >= 4) { NT_BATCH_EPI(4, 4) } else { NT_BATCH_EPI(4, 3) }
    }
  } else if (R == 1) {   // the V rows of a two-format Q/K/V launch
    if constexpr (FMT == NT_Q6_K) {
      if (epi == EPI_QKV) {
        if (S >= 4) return launch_gemv_batch_t<FMT, 1, 4, EPI_QKV>(a, b, s, pdl);
        return launch_gemv_batch_t<FMT, 1, 3, EPI_QKV>(a, b, s, pdl);
      }
    }
  } else {
    if (S >= 4) { NT_BATCH_EPI(2, 4) } else { NT_BATCH_EPI(2, 3) }
  }
#undef NT_BATCH_EPI
  return cudaErrorInvalidValue;
}

// Instantiated shapes: 16 warps per CTA (one CTA per SM) with S in {3, 4, 6, 8}
// (R = 2) or {3, 4} (R = 4, 4-bit formats only).  S is rounded down to the
// nearest instantiated depth.
// (A depth of 5, which fits beside the x of 8192 and 28672 columns, measured 1%
// slower on the 70B Q4_K_M step and no faster on the down projection.)
template <int FMT>
cudaError_t launch_gemv_pipe_fmt(const GemvArgs& a, int epi, int R, int S, cudaStream_t s, bool pdl,
                                 int* grid_used) {
  if (R == 4) {
    if constexpr (kFourRows<FMT>) {
      if (S >= 4) return launch_gemv_pipe_rs<FMT, 4, 4, kPipeWarps>(a, epi, s, pdl, grid_used);
      return launch_gemv_pipe_rs<FMT, 4, 3, kPipeWarps>(a, epi, s, pdl, grid_used);
    }
    return cudaErrorInvalidValue;
  }
  if (S >= 8) return launch_gemv_pipe_rs<FMT, 2, 8, kPipeWarps>(a, epi, s, pdl, grid_used);
  if (S >= 6) return launch_gemv_pipe_rs<FMT, 2, 6, kPipeWarps>(a, epi, s, pdl, grid_used);
  if (S >= 4) return launch_gemv_pipe_rs<FMT, 2, 4, kPipeWarps>(a, epi, s, pdl, grid_used);
  return launch_gemv_pipe_rs<FMT, 2, 3, kPipeWarps>(a, epi, s, pdl, grid_used);
}

// Q4_K rows of a1 and Q6_K rows of a2 over one x (see k_gemv_pipe2), 16 warps
// per CTA, one CTA per SM, the ring depths that fit beside x.
template <int EPI>
cudaError_t launch_gemv_pipe2_q4k_q6k(const GemvArgs& a1, const GemvArgs& a2, cudaStream_t s, bool pdl) {
  constexpr int NW = kPipeWarps, R1 = 4, R2 = 1, S1 = 4, S2 = 8;
  auto kern = k_gemv_pipe2<NT_Q4_K, NT_Q6_K, R1, R2, S1, S2, EPI, NW>;
  constexpr size_t slice = pipe_slice<NT_Q4_K, R1, S1, 0>() > pipe_slice<NT_Q6_K, R2, S2, 0>()
                               ? pipe_slice<NT_Q4_K, R1, S1, 0>()
                               : pipe_slice<NT_Q6_K, R2, S2, 0>();
  const size_t smem = pipe_x_bytes(a1.ncols, EPI) + size_t(NW) * slice;
  if (smem > size_t(kPipeMaxSmem) || a1.ncols != a2.ncols || a1.col0 || a2.col0) return cudaErrorInvalidValue;
  static const KernelSetup setup = kernel_setup(kern, kPipeMaxSmem);
  if (setup.err != cudaSuccess) return setup.err;
  const int s_sms = setup.sms;
  const int64_t n1 = gemv_logical_rows(a1), n2 = gemv_logical_rows(a2);
  const int64_t groups = (n1 + R1 - 1) / R1 + (n2 + R2 - 1) / R2;
  int64_t grid = (groups + NW - 1) / NW;
  if (grid < s_sms) grid = groups < s_sms ? groups : s_sms;
  if (grid > s_sms) grid = s_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(NW * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a1, a2, n1, n2);
}

#define NT_DECLARE_GEMV_PIPE(NAME)                                                                          \
  cudaError_t NAME(const GemvArgs& a, int epi, int R, int S, cudaStream_t s, bool pdl, int* grid_used);        \
  cudaError_t NAME##_batch(const GemvArgs& a, int epi, int R, int S, const GemvBatch& b, cudaStream_t s, bool pdl);
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q8_0)
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q4_0)
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q4_k)
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q5_k)
NT_DECLARE_GEMV_PIPE(launch_gemv_pipe_q6_k)
#undef NT_DECLARE_GEMV_PIPE

}  // namespace nt
