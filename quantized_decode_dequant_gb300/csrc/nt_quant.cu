// nt_quant.cu -- weight generation, block quantization, dequantization and the
// quantized-tensor entry points.
//
// Formats: hada "Überblick über NTransformer" lists Q4_0, Q8_0, Q4_K(_M), Q6_K;
// their dequantization formulas are w = d*q (Q8_0), d*(q-8) (Q4_0),
// d*sc*q - dmin*m (Q4_K) and d*sc*(q-32) (Q6_K).  The pages give neither the
// quantizer nor the byte packing; the rules implemented here are:
//   Q8_0  d32 = absmax/127, d = f16(d32), q = clamp(round(w/d32), -127, 127)
//   Q4_0  d32 = absmax/7,   d = f16(d32), q = clamp(round(w/d32)+8, 0, 15)
//   Q4_K  per 32: lo = min(0, min w), s = (max w - lo)/15, m* = -lo;
//         d = f16(max s/63), dmin = f16(max m*/63), sc = clamp(round(s/d), 0, 63),
//         m = clamp(round(m*/dmin), 0, 63), q = clamp(round((w + dmin*m)/(d*sc)), 0, 15)
//   Q6_K  per 16: s = absmax/31; d = f16(max s/127); sc = clamp(round(s/d), 0, 127);
//         q = clamp(round(w/(d*sc)) + 32, 0, 63)
// with round = half away from zero, IEEE division and binary16 round-to-nearest-even.
// Weights come from a counter-based generator: SplitMix64's output function
// (Steele, Lea, Flood, OOPSLA 2014) on the counter seed + gamma*(uid*2^40 + 3i + j + 1),
// j = 0..2, whose twelve 16-bit lanes sum to an Irwin-Hall normal draw.
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "nt_internal.cuh"

namespace nt {

static thread_local std::string g_err;

void set_error(const std::string& msg) { g_err = msg; }
nt_status fail(nt_status s, const std::string& msg) {
  g_err = msg;
  return s;
}
nt_status cuda_fail(cudaError_t e, const char* what) {
  char buf[512];
  snprintf(buf, sizeof buf, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  g_err = buf;
  return e == cudaErrorMemoryAllocation ? NT_E_NOMEM : NT_E_CUDA;
}

// ---------------------------------------------------------------- layout --

static size_t pad256(size_t n) { return (n + 255) & ~size_t(255); }

size_t StreamSizes::padded_total() const { return pad256(q) + pad256(qh) + pad256(meta) + pad256(d); }

StreamSizes stream_sizes(int type, int64_t rows, int64_t cols) {
  StreamSizes s;
  size_t n = size_t(rows) * size_t(cols);
  switch (type) {
    case NT_Q8_0: s.q = n; s.d = n / 32 * 2; break;
    case NT_Q4_0: s.q = n / 2; s.d = n / 32 * 2; break;
    case NT_Q4_K: s.q = n / 2; s.meta = n / 256 * 16; break;
    case NT_Q6_K: s.q = n / 2; s.qh = n / 4; s.meta = n / 16; s.d = n / 256 * 2; break;
    case NT_Q5_K: s.q = n / 2; s.qh = n / 8; s.meta = n / 256 * 16; break;
  }
  return s;
}

size_t layout_streams(QMat& m, uint8_t* base) {
  StreamSizes s = stream_sizes(m.type, m.rows, m.cols);
  uint8_t* p = base;
  m.q = p; p += pad256(s.q);
  m.qh = s.qh ? p : nullptr; p += pad256(s.qh);
  m.meta = s.meta ? p : nullptr; p += pad256(s.meta);
  m.d = s.d ? reinterpret_cast<__half*>(p) : nullptr; p += pad256(s.d);
  return size_t(p - base);
}

// ------------------------------------------------------------- generator --

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }
__device__ __forceinline__ int rnd(float v) { return int(roundf(v)); }   // half away from zero

// One warp quantizes 256 consecutive elements of a row; lane l owns 8 of them.
template <int T>
__global__ void __launch_bounds__(256) k_generate(QMat m, uint64_t seed, uint32_t uid, float std) {
  const int lane = threadIdx.x & 31;
  const int64_t chunks_per_row = (m.cols + 255) / 256;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (warp >= m.rows * chunks_per_row) return;   // whole warps exit together
  const int64_t row = warp / chunks_per_row;
  const int64_t e0 = (warp % chunks_per_row) * 256;
  const int64_t ebase = row * m.cols + e0 + 8 * lane;     // flat element index of this lane's first value
  const bool active = e0 + 8 * lane < m.cols;

  float w[8];
#pragma unroll
  for (int k = 0; k < 8; k++) w[k] = active ? __fmul_rn(gen_normal(seed, uid, uint64_t(ebase + k)), std) : 0.0f;

  if (T == NT_Q8_0 || T == NT_Q4_0) {
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; k++) amax = fmaxf(amax, fabsf(w[k]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d32 = __fdiv_rn(amax, T == NT_Q8_0 ? 127.0f : 7.0f);
    if (!active) return;
    if (T == NT_Q8_0) {
      uint32_t wd[2] = {0u, 0u};
#pragma unroll
      for (int k = 0; k < 8; k++) {
        int q = d32 == 0.0f ? 0 : clampi(rnd(__fdiv_rn(w[k], d32)), -127, 127);
        wd[k >> 2] |= uint32_t(q & 0xFF) << (8 * (k & 3));
      }
      *reinterpret_cast<uint2*>(m.q + ebase) = make_uint2(wd[0], wd[1]);
    } else {
      uint32_t wd = 0u;
#pragma unroll
      for (int k = 0; k < 8; k++) {
        int q = d32 == 0.0f ? 8 : clampi(rnd(__fdiv_rn(w[k], d32)) + 8, 0, 15);
        wd |= uint32_t(q) << (4 * k);
      }
      *reinterpret_cast<uint32_t*>(m.q + ebase / 2) = wd;
    }
    if ((lane & 3) == 0) m.d[ebase / 32] = __float2half_rn(d32);
  } else if (T == NT_Q4_K || T == NT_Q5_K) {
    constexpr float kLevels = T == NT_Q4_K ? 15.0f : 31.0f;
    constexpr int kMaxQ = T == NT_Q4_K ? 15 : 31;
    float lo = 0.0f, hi = w[0];
#pragma unroll
    for (int k = 0; k < 8; k++) { lo = fminf(lo, w[k]); hi = fmaxf(hi, w[k]); }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const float s = __fdiv_rn(__fsub_rn(hi, lo), kLevels);
    const float ms = __fsub_rn(0.0f, lo);
    float smax = s, mmax = ms;
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
      mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    }
    const __half dh = __float2half_rn(__fdiv_rn(smax, 63.0f));
    const __half mh = __float2half_rn(__fdiv_rn(mmax, 63.0f));
    const float d = __half2float(dh), dmin = __half2float(mh);
    const int sc = d == 0.0f ? 0 : clampi(rnd(__fdiv_rn(s, d)), 0, 63);
    const int mm = dmin == 0.0f ? 0 : clampi(rnd(__fdiv_rn(ms, dmin)), 0, 63);
    const float a = __fmul_rn(d, float(sc)), b = __fmul_rn(dmin, float(mm));
    uint32_t wd = 0u, hb = 0u;
    const int wi = lane & 3;   // this lane's code word within the 32-element unit
#pragma unroll
    for (int k = 0; k < 8; k++) {
      int q = a == 0.0f ? 0 : clampi(rnd(__fdiv_rn(__fadd_rn(w[k], b), a)), 0, kMaxQ);
      wd |= uint32_t(q & 15) << (4 * k);
      if (T == NT_Q5_K) hb |= uint32_t(q >> 4) << q5_hi_bit(8 * wi + k);
    }
    *reinterpret_cast<uint32_t*>(m.q + ebase / 2) = wd;
    if (T == NT_Q5_K) {   // the unit's four lanes share one fifth-bit word
      hb |= __shfl_xor_sync(0xffffffffu, hb, 1);
      hb |= __shfl_xor_sync(0xffffffffu, hb, 2);
      if (wi == 0) *reinterpret_cast<uint32_t*>(m.qh + ebase / 8) = hb;
    }
    // device header: bytes sc_j | (m_j & 3) << 6 (j = 0..7), then nibbles m_j >> 2
    uint32_t yz[2] = {0u, 0u}, wn = 0u;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const uint32_t scj = uint32_t(__shfl_sync(0xffffffffu, sc, 4 * j));
      const uint32_t mj = uint32_t(__shfl_sync(0xffffffffu, mm, 4 * j));
      yz[j >> 2] |= (scj | ((mj & 3u) << 6)) << (8 * (j & 3));
      wn |= (mj >> 2) << (4 * j);
    }
    if (lane == 0) {
      uint4 meta;
      meta.x = uint32_t(__half_as_ushort(dh)) | (uint32_t(__half_as_ushort(mh)) << 16);
      meta.y = yz[0];
      meta.z = yz[1];
      meta.w = wn;
      *reinterpret_cast<uint4*>(m.meta + (ebase / 256) * 16) = meta;
    }
  } else {  // NT_Q6_K
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; k++) amax = fmaxf(amax, fabsf(w[k]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const float s = __fdiv_rn(amax, 31.0f);
    float smax = s;
#pragma unroll
    for (int o = 2; o <= 16; o <<= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
    const __half dh = __float2half_rn(__fdiv_rn(smax, 127.0f));
    const float d = __half2float(dh);
    const int sc = d == 0.0f ? 0 : clampi(rnd(__fdiv_rn(s, d)), 0, 127);
    const float a = __fmul_rn(d, float(sc));
    // lane l holds elements 8(l%4)..8(l%4)+7 of a 32-element unit: code word l%4
    const int wi = lane & 3;
    uint32_t lo = 0u, g = 0u;
#pragma unroll
    for (int k = 0; k < 8; k++) {
      int q = a == 0.0f ? 32 : clampi(rnd(__fdiv_rn(w[k], a)) + 32, 0, 63);
      lo |= uint32_t(q & 15) << (4 * k);
      g |= uint32_t(q >> 4) << q6_hi_shift(8 * wi + k);
    }
    g |= __shfl_xor_sync(0xffffffffu, g, 1);   // code words 2p and 2p+1 share high-bit word G_p
    *reinterpret_cast<uint32_t*>(m.q + ebase / 2) = lo;
    if ((wi & 1) == 0) *reinterpret_cast<uint32_t*>(m.qh + (ebase - 8 * wi) / 4 + 4 * (wi >> 1)) = g;
    if ((lane & 1) == 0) m.meta[ebase / 16] = uint8_t(int8_t(sc));
    if (lane == 0) m.d[ebase / 256] = dh;
  }
}

cudaError_t launch_generate(const QMat& m, uint64_t seed, uint32_t uid, float std, cudaStream_t s) {
  const int64_t warps = m.rows * ((m.cols + 255) / 256);
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)blocks), block(256u);
  switch (m.type) {
    case NT_Q8_0: k_generate<NT_Q8_0><<<grid, block, 0, s>>>(m, seed, uid, std); break;
    case NT_Q4_0: k_generate<NT_Q4_0><<<grid, block, 0, s>>>(m, seed, uid, std); break;
    case NT_Q4_K: k_generate<NT_Q4_K><<<grid, block, 0, s>>>(m, seed, uid, std); break;
    case NT_Q6_K: k_generate<NT_Q6_K><<<grid, block, 0, s>>>(m, seed, uid, std); break;
    case NT_Q5_K: k_generate<NT_Q5_K><<<grid, block, 0, s>>>(m, seed, uid, std); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// --------------------------------------------------------------- dequant --

// The formats' fp32 formulas, one rounding per operation (Q4_K: one fused multiply-add).
__global__ void k_dequant(QMat m, int64_t row0, int64_t n, float* out) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
    out[i] = dequant_elem(m, row0 * m.cols + i);
}

cudaError_t launch_dequant(const QMat& m, int64_t row0, int64_t nrows, float* out, cudaStream_t s) {
  const int64_t n = nrows * m.cols;
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  k_dequant<<<unsigned(blocks), 256, 0, s>>>(m, row0, n, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- export --

// K-quant super-block header, device arrangement -> canonical bytes: d, dmin,
// then the sixteen 6-bit fields sc_0..7, m_0..7 packed least-significant bit first.
static void kquant_header_canonical(const uint8_t* dev, uint8_t* out) {
  memcpy(out, dev, 4);
  memset(out + 4, 0, 12);
  for (int j = 0; j < 8; j++) {
    int sc, m;
    kquant_scale_min_bytes(dev, j, sc, m);
    for (int f = 0; f < 2; f++) {
      const int v = f ? m : sc, base = 6 * (j + 8 * f);
      for (int bit = 0; bit < 6; bit++)
        if ((v >> bit) & 1) out[4 + ((base + bit) >> 3)] |= uint8_t(1u << ((base + bit) & 7));
    }
  }
}

// Interleaves the device streams of rows [row0, row0+nrows) into canonical
// block bytes on the host.
static nt_status export_rows(const nt_qtensor* t, int64_t row0, int64_t nrows, uint8_t* dst) {
  const QMat& m = t->m;
  const int64_t n = nrows * m.cols;
  if (n == 0) return NT_OK;
  StreamSizes full = stream_sizes(m.type, m.rows, m.cols);
  StreamSizes part = stream_sizes(m.type, nrows, m.cols);
  std::vector<uint8_t> q(part.q), qh(part.qh), meta(part.meta), d(part.d);
  auto fetch = [&](std::vector<uint8_t>& v, const uint8_t* src, size_t full_bytes) -> nt_status {
    if (v.empty()) return NT_OK;
    const size_t off = size_t(row0) * (full_bytes / size_t(m.rows));   // streams hold whole rows
    const uint8_t* p = src + off;
    if (t->on_host) memcpy(v.data(), p, v.size());
    else NT_CUDA(cudaMemcpy(v.data(), p, v.size(), cudaMemcpyDeviceToHost));
    return NT_OK;
  };
  nt_status st;
  if ((st = fetch(q, m.q, full.q)) || (st = fetch(qh, m.qh, full.qh)) || (st = fetch(meta, m.meta, full.meta)) ||
      (st = fetch(d, reinterpret_cast<const uint8_t*>(m.d), full.d)))
    return st;
  const int qk = block_elems(m.type), bb = block_bytes(m.type);
  for (int64_t b = 0; b < n / qk; b++) {
    uint8_t* out = dst + b * bb;
    const int64_t e = b * qk;   // element index relative to row0
    switch (m.type) {
      case NT_Q8_0:
        memcpy(out, &d[b * 2], 2);
        memcpy(out + 2, &q[e], 32);
        break;
      case NT_Q4_0:
        memcpy(out, &d[b * 2], 2);
        memcpy(out + 2, &q[e / 2], 16);
        break;
      case NT_Q4_K:
        kquant_header_canonical(&meta[b * 16], out);
        memcpy(out + 16, &q[e / 2], 128);
        break;
      case NT_Q5_K: {
        kquant_header_canonical(&meta[b * 16], out);
        // canonical fifth bits: element k of the block at byte k/8, bit k%8
        uint8_t* cqh = out + 16;
        memset(cqh, 0, 32);
        for (int k = 0; k < 256; k++) {
          const uint8_t* hp = &qh[(e + (k & ~31)) / 8];
          const uint32_t h = uint32_t(hp[0]) | (uint32_t(hp[1]) << 8) | (uint32_t(hp[2]) << 16) | (uint32_t(hp[3]) << 24);
          cqh[k >> 3] |= uint8_t(((h >> q5_hi_bit(k & 31)) & 1) << (k & 7));
        }
        memcpy(out + 48, &q[e / 2], 128);
      } break;
      case NT_Q6_K: {
        memcpy(out, &q[e / 2], 128);
        // canonical high bits: element k of the block at byte k/4, bits 2(k%4)
        uint8_t* cqh = out + 128;
        memset(cqh, 0, 64);
        for (int k = 0; k < 256; k++) {
          const int64_t ue = e + (k & ~31);            // first element of k's 32-element unit
          const int kk = k & 31;
          const uint8_t* gp = &qh[ue / 4 + 4 * (kk >> 4)];
          const uint32_t g = uint32_t(gp[0]) | (uint32_t(gp[1]) << 8) | (uint32_t(gp[2]) << 16) | (uint32_t(gp[3]) << 24);
          const int hi = int(g >> q6_hi_shift(kk)) & 3;
          cqh[k >> 2] |= uint8_t(hi << (2 * (k & 3)));
        }
        memcpy(out + 192, &meta[e / 16], 16);
        memcpy(out + 208, &d[b * 2], 2);
      } break;
    }
  }
  return NT_OK;
}

}  // namespace nt

using namespace nt;

extern "C" {

const char* nt_last_error(void) { return g_err.c_str(); }

nt_status nt_qtensor_create(nt_qtype type, int64_t rows, int64_t cols, uint64_t seed, uint32_t uid, float std,
                            nt_qtensor** out) {
  if (!out) return fail(NT_E_INVAL, "nt_qtensor_create: out is NULL");
  if (type == NT_F32 || type == NT_F16) return fail(NT_E_UNSUPPORTED, "nt_qtensor_create: F32/F16 weights are not implemented");
  if (!supported_weight_type(type)) return fail(NT_E_INVAL, "nt_qtensor_create: unknown type");
  if (rows <= 0 || cols <= 0 || cols % block_elems(type))
    return fail(NT_E_INVAL, "nt_qtensor_create: rows/cols must be positive and cols a multiple of the block size");
  if (uid >= (1u << 24)) return fail(NT_E_INVAL, "nt_qtensor_create: uid must be below 2^24");
  if (rows * cols > (int64_t(1) << 40)) return fail(NT_E_INVAL, "nt_qtensor_create: tensor too large");
  nt_qtensor* t = new (std::nothrow) nt_qtensor();
  if (!t) return fail(NT_E_NOMEM, "nt_qtensor_create: host allocation failed");
  t->m.type = type;
  t->m.rows = rows;
  t->m.cols = cols;
  StreamSizes s = stream_sizes(type, rows, cols);
  t->nbytes = s.total();
  cudaError_t e = cudaMalloc(&t->base, s.padded_total());
  if (e != cudaSuccess) {
    delete t;
    return cuda_fail(e, "nt_qtensor_create: cudaMalloc");
  }
  t->owns = 1;
  layout_streams(t->m, t->base);
  e = launch_generate(t->m, seed, uid, std, 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  if (e != cudaSuccess) {
    cudaFree(t->base);
    delete t;
    return cuda_fail(e, "nt_qtensor_create: generate");
  }
  *out = t;
  return NT_OK;
}

void nt_qtensor_destroy(nt_qtensor* t) {
  if (!t) return;
  if (t->owns && t->base) cudaFree(t->base);
  delete t;
}

nt_status nt_qtensor_info(const nt_qtensor* t, nt_qtype* type, int64_t* rows, int64_t* cols, size_t* device_bytes) {
  if (!t) return fail(NT_E_INVAL, "nt_qtensor_info: tensor is NULL");
  if (type) *type = nt_qtype(t->m.type);
  if (rows) *rows = t->m.rows;
  if (cols) *cols = t->m.cols;
  if (device_bytes) *device_bytes = t->nbytes;
  return NT_OK;
}

nt_status nt_qtensor_export(const nt_qtensor* t, int64_t row0, int64_t nrows, void* host_blocks, size_t nbytes) {
  if (!t || !host_blocks) return fail(NT_E_INVAL, "nt_qtensor_export: NULL argument");
  if (row0 < 0 || nrows < 0 || row0 + nrows > t->m.rows) return fail(NT_E_INVAL, "nt_qtensor_export: row range");
  const size_t need = size_t(nrows) * size_t(t->m.cols / block_elems(t->m.type)) * size_t(block_bytes(t->m.type));
  if (nbytes < need) return fail(NT_E_INVAL, "nt_qtensor_export: buffer too small");
  return export_rows(t, row0, nrows, static_cast<uint8_t*>(host_blocks));
}

nt_status nt_dequant(const nt_qtensor* t, int64_t row0, int64_t nrows, float* dev_out, void* stream) {
  if (!t || !dev_out) return fail(NT_E_INVAL, "nt_dequant: NULL argument");
  if (t->on_host) return fail(NT_E_STATE, "nt_dequant: tensor lives in host memory (streamed layer)");
  if (row0 < 0 || nrows < 0 || row0 + nrows > t->m.rows) return fail(NT_E_INVAL, "nt_dequant: row range");
  cudaError_t e = launch_dequant(t->m, row0, nrows, dev_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "nt_dequant");
  return NT_OK;
}

}  // extern "C"
