// nt_internal.cuh -- shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/nt.h"

namespace nt {

// ---------------------------------------------------------------- errors --

void set_error(const std::string& msg);
nt_status fail(nt_status s, const std::string& msg);
nt_status cuda_fail(cudaError_t e, const char* what);

#define NT_CUDA(call)                                        \
  do {                                                       \
    cudaError_t e__ = (call);                                \
    if (e__ != cudaSuccess) return ::nt::cuda_fail(e__, #call); \
  } while (0)

// ------------------------------------------------------------ formats --

inline int block_elems(int t) {
  switch (t) {
    case NT_Q8_0: case NT_Q4_0: return 32;
    case NT_Q4_K: case NT_Q6_K: case NT_Q5_K: return 256;
  }
  return 0;
}
inline int block_bytes(int t) {
  switch (t) {
    case NT_Q8_0: return 34;
    case NT_Q4_0: return 18;
    case NT_Q4_K: return 144;
    case NT_Q6_K: return 210;
    case NT_Q5_K: return 176;
  }
  return 0;
}
inline bool supported_weight_type(int t) { return block_elems(t) != 0; }

// Device layout of one quantized matrix: separate streams in row-major element
// order, each starting on a 256-byte boundary.
//   Q8_0: q  = int8 code per element             d = f16 per 32 elements
//   Q4_0: q  = 4-bit codes, element k of a row at byte k/2 (low nibble for even k)
//                                                d = f16 per 32 elements
//   Q4_K: q  = 4-bit codes as Q4_0               meta = 16 B per 256 elements:
//         f16 d | f16 dmin | 8 B: byte j = sc_j | (m_j & 3) << 6 | 4 B: nibble j =
//         m_j >> 2 (the canonical header packs the same sixteen 6-bit fields
//         LSB-first; this arrangement gives each lane its sub-block's pair with a
//         byte permute and three logic ops)
//   Q6_K: q  = low 4 bits as Q4_0; qh = high 2 bits, 8 bytes per 32 elements
//         as two little-endian words G_0 (elements 0..15) and G_1 (16..31);
//         within G_p, element 8w+i of the unit (w = 2p + s, i = 2j + o) sits at
//         bit 8j + (o ? 0 : 4) + (s ? 2 : 0); meta = int8 sc per 16 elements,
//         d = f16 per 256.  (The canonical export order is rebuilt on the host.)
//   Q5_K: q  = low 4 bits as Q4_0; qh = one little-endian word H per 32 elements:
//         element 8w+2i+o of the unit (w < 4, i < 4, o < 2) has its fifth bit at
//         bit 8i + 2w + o, i.e. byte i of H serves byte i of the eight code words
//         v = 2w+o that the low/high nibbles of the unit's four words form;
//         meta = 16 B per 256 elements in Q4_K's device arrangement.
struct QMat {
  int32_t type = 0;
  int64_t rows = 0, cols = 0;
  uint8_t* q = nullptr;
  uint8_t* qh = nullptr;
  uint8_t* meta = nullptr;
  __half* d = nullptr;
};

struct StreamSizes {
  size_t q = 0, qh = 0, meta = 0, d = 0;
  size_t total() const { return q + qh + meta + d; }
  size_t padded_total() const;
};
StreamSizes stream_sizes(int type, int64_t rows, int64_t cols);

// Lays the streams out from base (which must be 256-byte aligned); returns
// the padded byte count used.
size_t layout_streams(QMat& m, uint8_t* base);

// Generation + quantization of a whole matrix into its device streams.
cudaError_t launch_generate(const QMat& m, uint64_t seed, uint32_t uid, float std, cudaStream_t s);
cudaError_t launch_dequant(const QMat& m, int64_t row0, int64_t nrows, float* out, cudaStream_t s);

// ------------------------------------------------------------- GEMV --

enum Epi : int {
  EPI_STORE = 0,     // y[r] = acc
  EPI_ADD = 1,       // y[r] += acc (residual stream)
  EPI_QKV = 2,       // q -> RoPE -> q buffer; k -> RoPE -> f16 cache; v -> f16 cache
  EPI_SWIGLU = 3,    // rows interleaved (gate_i, up_i): y[i] = silu(gate)*up
  EPI_LOGITS = 4,    // y[r] = acc and per-CTA top-2 partials for the argmax
};

struct EpiArgs {
  float* y = nullptr;
  int32_t row_base = 0;          // logical row of this launch's row 0 (EPI_QKV)
  // EPI_QKV
  int32_t q_rows = 0, k_rows = 0, head_dim = 0;
  const int32_t* pos = nullptr;  // device position counter
  const float2* rope = nullptr;  // [max_ctx][head_dim/2] (cos, sin)
  __half* k_cache = nullptr;     // this layer's K: [kv_head][max_ctx][head_dim]
  __half* v_cache = nullptr;
  int32_t max_ctx = 0;
  // EPI_LOGITS
  float4* top2 = nullptr;        // per CTA: (best value, best index as float bits, second value, -)
};

struct GemvArgs {
  QMat seg[3];                   // up to 3 row segments of one format, logical rows concatenated
  int32_t nseg = 1;
  int32_t interleave = 0;        // 2 segments of equal rows: logical row 2i+s -> segment s row i
  const float* x = nullptr;      // input [cols]
  int32_t norm = 0;              // 1: x <- x * rsqrt(mean(x^2) + eps) before the product
  float eps = 1e-5f;
  int64_t col0 = 0, ncols = 0;   // column window [col0, col0 + ncols) (set by launch_gemv)
  int32_t max_grid = 0;          // upper bound on CTAs (0: kMaxGemvGrid)
  EpiArgs epi;
};

int64_t gemv_logical_rows(const GemvArgs& a);
constexpr int kMaxGemvGrid = 152 * 8;   // upper bound of CTAs in one GEMV launch (partial buffers)
// grid_used (nullable) receives the number of CTAs launched.
cudaError_t launch_gemv(const GemvArgs& a, int epi, cudaStream_t s, bool pdl, int* grid_used);
// Two GEMVs over the same x in one launch where a kernel exists for the pair
// (a Q4_K a1 with a Q6_K a2, whole 1024-column tiles); else two launch_gemv calls.
// launches (nullable) receives 1 or 2.
cudaError_t launch_gemv_pair(const GemvArgs& a1, const GemvArgs& a2, int epi, cudaStream_t s, bool pdl,
                             int* launches);
// Several tokens through one GEMV (see launch_gemv_batch in nt_gemv.cu): token i
// reads toks[i].x and writes toks[i].y (its position: toks[i].pos), each with
// the arithmetic of its own single-token launch.
struct BatchTok;
// launches (nullable) receives the number of launches (per token when they do
// not fit two at a time).
cudaError_t launch_gemv_batch(const GemvArgs& a, int epi, const BatchTok* toks, int k, int R_single, cudaStream_t s,
                              bool pdl, int* launches);
cudaError_t launch_gemv_pair_batch(const GemvArgs& a1, const GemvArgs& a2, int epi, const BatchTok* toks1,
                                   const BatchTok* toks2, int k, cudaStream_t s, bool pdl, int* launches);
bool pipe_shape(int fmt, int64_t nrows, int64_t cols, int epi, int& R, int& S);

// ------------------------------------------------------------ generator --
// SplitMix64 output function (Steele, Lea, Flood, OOPSLA 2014) on the counter
// seed + gamma*(uid*2^40 + 3i + j + 1), j = 0..2; the twelve 16-bit lanes of the
// three outputs sum to an Irwin-Hall draw z = (sum - 393210)/65536 (mean 0, variance 1).
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float gen_normal(uint64_t seed, uint32_t uid, uint64_t i) {
  const uint64_t gamma = 0x9E3779B97F4A7C15ull;
  const uint64_t base = (uint64_t(uid) << 40) + 3ull * i;
  int s = 0;
#pragma unroll
  for (int j = 0; j < 3; j++) {
    const uint64_t r = mix64(seed + gamma * (base + uint64_t(j) + 1ull));
    s += int(r & 0xFFFF) + int((r >> 16) & 0xFFFF) + int((r >> 32) & 0xFFFF) + int(r >> 48);
  }
  // |s - 393210| < 2^19: the conversion and the power-of-two scale are exact
  return __fmul_rn(__int2float_rn(s - 393210), 1.0f / 65536.0f);
}

// One dequantized weight (flat element index e), bit-exact under the formats'
// fp32 formulas: Q8_0 d*q, Q4_0 d*(q-8), Q4_K and Q5_K fma(d*sc, q, -(dmin*m)),
// Q6_K (d*sc)*(q-32).
__device__ __forceinline__ int nib_at(const uint8_t* q, int64_t e) { return (q[e >> 1] >> ((e & 1) * 4)) & 15; }

// Two high bits of element e of a Q6_K tensor in the device layout (see QMat).
__host__ __device__ __forceinline__ int q6_hi_shift(int k) {   // k = e % 32
  const int w = k >> 3, i = k & 7;
  return 8 * (i >> 1) + ((i & 1) ? 0 : 4) + ((w & 1) ? 2 : 0);
}
__device__ __forceinline__ int q6_hi(const uint8_t* qh, int64_t e) {
  const int k = int(e & 31);
  const uint32_t g = *reinterpret_cast<const uint32_t*>(qh + ((e - k) >> 2) + 4 * (k >> 4));
  return int(g >> q6_hi_shift(k)) & 3;
}

// Fifth bit of element e of a Q5_K tensor in the device layout (see QMat).
__host__ __device__ __forceinline__ int q5_hi_bit(int k) {   // k = e % 32
  return 8 * ((k & 7) >> 1) + 2 * (k >> 3) + (k & 1);
}
__device__ __forceinline__ int q5_hi(const uint8_t* qh, int64_t e) {
  const int k = int(e & 31);
  const uint32_t h = *reinterpret_cast<const uint32_t*>(qh + ((e - k) >> 3));
  return int(h >> q5_hi_bit(k)) & 1;
}

// Scale sc_j and min m_j of sub-block j from a K-quant super-block header in
// the device arrangement (words x: d, dmin; y, z: bytes sc_j | (m_j & 3) << 6;
// w: nibbles m_j >> 2).
__device__ __forceinline__ void kquant_scale_min(const uint4 meta, int j, uint32_t& sc, uint32_t& m) {
  const uint32_t b = __byte_perm(meta.y, meta.z, uint32_t(j));   // byte j of y:z in the low byte
  sc = b & 63u;
  m = ((b >> 6) & 3u) | (((meta.w >> (4 * j)) & 15u) << 2);
}
__host__ __device__ __forceinline__ void kquant_scale_min_bytes(const uint8_t* meta, int j, int& sc, int& m) {
  sc = meta[4 + j] & 63;
  m = (meta[4 + j] >> 6) | (((meta[12 + (j >> 1)] >> (4 * (j & 1))) & 15) << 2);
}

__device__ __forceinline__ float dequant_elem(const QMat& m, int64_t e) {
  switch (m.type) {
    case NT_Q8_0:
      return __fmul_rn(__half2float(m.d[e / 32]), float(int8_t(m.q[e])));
    case NT_Q4_0:
      return __fmul_rn(__half2float(m.d[e / 32]), float(nib_at(m.q, e) - 8));
    case NT_Q4_K: {
      const uint8_t* meta = m.meta + (e / 256) * 16;
      const float d = __half2float(__ushort_as_half(uint16_t(meta[0] | (meta[1] << 8))));
      const float dmin = __half2float(__ushort_as_half(uint16_t(meta[2] | (meta[3] << 8))));
      int sc, mm;
      kquant_scale_min_bytes(meta, int((e % 256) / 32), sc, mm);
      const float a = __fmul_rn(d, float(sc));
      const float b = __fmul_rn(dmin, float(mm));
      return __fmaf_rn(a, float(nib_at(m.q, e)), -b);
    }
    case NT_Q5_K: {
      const uint8_t* meta = m.meta + (e / 256) * 16;
      const float d = __half2float(__ushort_as_half(uint16_t(meta[0] | (meta[1] << 8))));
      const float dmin = __half2float(__ushort_as_half(uint16_t(meta[2] | (meta[3] << 8))));
      int sc, mm;
      kquant_scale_min_bytes(meta, int((e % 256) / 32), sc, mm);
      const float a = __fmul_rn(d, float(sc));
      const float b = __fmul_rn(dmin, float(mm));
      return __fmaf_rn(a, float(nib_at(m.q, e) | (q5_hi(m.qh, e) << 4)), -b);
    }
    case NT_Q6_K: {
      const int q = nib_at(m.q, e) | (q6_hi(m.qh, e) << 4);
      const float a = __fmul_rn(__half2float(m.d[e / 256]), float(int8_t(m.meta[e / 16])));
      return __fmul_rn(a, float(q - 32));
    }
  }
  return 0.0f;
}

// ------------------------------------------------------------ helpers --

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// One-time launch setup of a kernel (thread-safe: a function-local static
// initialised once): the device's SM count and, for kernels that ask for more
// than 48 KB, the dynamic shared-memory limit.  A concurrent first launch from
// another thread waits for the setup instead of launching without the limit.
struct KernelSetup {
  int sms = 0;
  cudaError_t err = cudaSuccess;
};
template <class K>
inline KernelSetup kernel_setup(K kern, int max_dynamic_smem) {
  KernelSetup k;
  int dev = 0;
  k.err = cudaGetDevice(&dev);
  if (k.err == cudaSuccess) k.err = cudaDeviceGetAttribute(&k.sms, cudaDevAttrMultiProcessorCount, dev);
  if (k.err == cudaSuccess && max_dynamic_smem > 0)
    k.err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic_smem);
  return k;
}

}  // namespace nt

struct nt_qtensor {
  nt::QMat m;
  size_t nbytes = 0;       // sum of the stream sizes (= rows*cols*bpw)
  uint8_t* base = nullptr; // device allocation (owned when owns != 0)
  uint8_t* host = nullptr; // page-locked host copy when the tensor lives on the host
  int owns = 0;
  int on_host = 0;
};
