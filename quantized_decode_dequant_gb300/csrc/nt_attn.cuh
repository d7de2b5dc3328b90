// nt_attn.cuh -- GQA decode attention over the f16 KV cache (hada "Hauptfunktionen":
// GQA with a KV cache; "Architektur und Codestruktur": softmax kernel).
//
// Split context: item (kv head g, chunk c) attends the G = n_heads/n_kv_heads
// query heads that share g over the chunk's C cached positions.  It keeps the
// chunk's softmax statistics (max m_c, sum of exponentials l_c) and the
// unnormalised exp-weighted sum o_c of its values.  The chunks of g's heads
// are merged, M = max m_c, o = sum o_c e^(m_c - M) / sum l_c e^(m_c - M), in
// one of two ways with the same arithmetic: where the items of every kv head
// fit one thread-block cluster that the GPU can hold for all kv heads at once,
// warps of the cluster merge from the items' shared memory (k_attn_cl);
// otherwise the CTA that finishes the last chunk of kv head g (an atomic
// ticket per kv head) merges from partials in global memory.
//
// The two contractions of an item are small dense products, run on the tensor
// cores with mma.sync m16n8k16 (f16 operands, fp32 accumulation):
//   scores  S[h][t] = q_h . K_t        A = q (query heads), B = K^T
//   values  O[h][d] = sum_t P[h][t] V_t[d]   A = P, B = V
// K and V are f16 already, so they enter exactly.  q and P are fp32; each is
// split into two f16 terms, hi = f16(v) and lo = f16(v - hi), held as separate
// rows of the A operand, and the two rows' products are added in fp32
// afterwards: the operand keeps about 22 significant bits instead of 11.
// With G <= 8 one 16-row tile holds hi (rows 0..G-1) and lo (rows 8..8+G-1);
// with G = 16 two tiles hold hi and lo of all heads.
#pragma once

#include <cooperative_groups.h>

#include "nt_internal.cuh"

namespace nt {

constexpr int kAttnWarps = 8;
constexpr int kAttnThreads = 32 * kAttnWarps;

// Chunk length C, a multiple of 16 and at least 32, fixed per model: the
// context is cut into at most 8 items per kv head up to 2560 positions,
// C = max(32, 16 ceil(max_ctx / 128)), so that a kv head's items fit one
// thread-block cluster of 8 (k_attn_cl); beyond that into at most 16 items up
// to 5120 positions, C = 16 ceil(max_ctx / 256), at most 320 (the merge reads
// every chunk's partials in one round of loads); longer contexts take more
// items of 320.  The items a step uses split its positions evenly (see k_attn).
// (Measured on GB300: 70B step at ctx 4096, 8 kv heads: 19 items per kv head,
// one per SM, 0.6% slower, the O projection's CTAs then finding no free SM for
// their early weight copies; 14 items the same as 16, 12 items 1% slower.
// Scoring the chunk's rows block by block as their copies land, with an
// acquire-release ticket, did not change the step either.  8B step at ctx 512:
// 8 items with the ticket merge the same as 16, with the cluster merge 0.6%
// faster.)
inline int attn_chunk_len(int max_ctx) {
  if (max_ctx <= 8 * 320) {
    const int c8 = 16 * ((max_ctx + 127) / 128);
    return c8 < 32 ? 32 : c8;
  }
  const int c = 16 * ((max_ctx + 255) / 256);
  return c > 320 ? 320 : c;   // 320: the largest instantiated chunk (longer contexts: more items)
}
// Largest chunk a kernel instantiation holds (its shared-memory layout).
inline int attn_chunk_max(int chunk) { return chunk <= 64 ? 64 : (chunk <= 128 ? 128 : (chunk <= 256 ? 256 : 320)); }

struct AttnArgs {
  const float* q = nullptr;         // [n_heads][hd], RoPE applied
  const __half* kc = nullptr;       // this layer's K: [n_kv][max_ctx][hd]
  const __half* vc = nullptr;
  int max_ctx = 0;
  int chunk = 64;                   // C, a multiple of 16
  float scale = 1.f;                // 1/sqrt(hd)
  float* part_o = nullptr;          // [n_heads][n_chunks][hd]
  float2* part_ml = nullptr;        // [n_heads][n_chunks] (m_c, l_c)
  int n_chunks = 0;                 // chunk stride of the partials
  unsigned* tickets = nullptr;      // [n_kv]: finished chunks of the current layer (0 between layers)
  float* out = nullptr;             // [n_heads][hd]
};

// Shared memory of one item (CM: the largest chunk).  K and V rows are padded
// by 16 bytes so that the eight 16-byte rows one ldmatrix phase reads fall in
// distinct banks; P rows likewise.  Then the softmax reductions and the merge
// flag.
template <int HD, int G, int CM>
struct AttnLayout {
  static constexpr int KP = HD + 8;              // halves per padded K/V row
  static constexpr int MT = G > 8 ? 2 : 1;       // 16-row tiles of the A operand
  static constexpr int PP = CM + 8;              // halves per padded P row
  static constexpr size_t kK = 0;
  static constexpr size_t kV = kK + size_t(CM) * KP * 2;
  static constexpr size_t kP = kV + size_t(CM) * KP * 2;
  static constexpr size_t kRed = kP + size_t(MT) * 16 * PP * 2;        // [2][warps][G] floats
  static constexpr size_t kFlag = kRed + size_t(2) * kAttnWarps * G * 4;
  static constexpr size_t kBytes = kFlag + 16;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void attn_cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// D += A B for one 16x8x16 tile (f16 operands, fp32 accumulators)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (hi, lo) f16 pair terms of two fp32 values, packed as two f16x2 words
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(__fsub_rn(x0, hf.x), __fsub_rn(x1, hf.y));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Copies of rows [r0, r1) of the item's K and V (chunk-relative) into shared
// memory, 16 bytes per thread and copy.  (One bulk copy per row, by one warp,
// measured almost twice as slow: 512 copies of 256 bytes queue up.)
template <int HD, int CM>
__device__ __forceinline__ void attn_copy_rows(const AttnArgs& a, int g, int t0, int r0, int r1, uint8_t* sm) {
  constexpr int KP = HD + 8, VPR = HD / 8;
  const __half* kb = a.kc + (int64_t(g) * a.max_ctx + t0) * HD;
  const __half* vb = a.vc + (int64_t(g) * a.max_ctx + t0) * HD;
  const uint32_t ks = smem_u32(sm), vs = ks + uint32_t(CM * KP) * 2;
  for (int i = r0 * VPR + int(threadIdx.x); i < r1 * VPR; i += kAttnThreads) {
    const int r = i / VPR, c = i % VPR;
    attn_cp16(ks + uint32_t(r * KP + c * 8) * 2, kb + r * HD + c * 8);
    attn_cp16(vs + uint32_t(r * KP + c * 8) * 2, vb + r * HD + c * 8);
  }
}

// Merge of the `used` chunks of query head j by one warp (lane holds HD/32
// dimensions): M = max m_c, o = sum_c o_c e^(m_c - M) / sum_c l_c e^(m_c - M),
// sums over c in increasing order.  Up to 32 chunks (every context up to 16 x 320
// positions), the statistics of chunk `lane` and the partial outputs of 16
// chunks at a time are loaded before any of them is used.
template <int HD>
__device__ __forceinline__ void attn_combine_head(const AttnArgs& a, int j, int used, int lane) {
  constexpr int V = HD / 32, NB = 16;
  const float2* ml = a.part_ml + int64_t(j) * a.n_chunks;
  const float* pj = a.part_o + int64_t(j) * a.n_chunks * HD + lane * V;
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; v++) acc[v] = 0.f;
  auto load_batch = [&](int c0, float (&t)[NB][V]) {
#pragma unroll
    for (int i = 0; i < NB; i++) {
      if (c0 + i < used) {
        const float* po = pj + int64_t(c0 + i) * HD;
        if (V == 4) {
          const float4 u = __ldcg(reinterpret_cast<const float4*>(po));
          t[i][0] = u.x; t[i][1 % V] = u.y; t[i][2 % V] = u.z; t[i][3 % V] = u.w;
        } else {
          const float2 u = __ldcg(reinterpret_cast<const float2*>(po));
          t[i][0] = u.x; t[i][1 % V] = u.y;
        }
      }
    }
  };
  float L = 0.f;
  if (used <= 32) {
    const float2 mv = lane < used ? __ldcg(ml + lane) : make_float2(-INFINITY, 0.f);
    float t[NB][V];
    load_batch(0, t);
    float M = mv.x;
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = lane < used ? expf(mv.x - M) : 0.f;
    L = __fmul_rn(mv.y, w);
#pragma unroll
    for (int o = 16; o; o >>= 1) L = __fadd_rn(L, __shfl_xor_sync(0xffffffffu, L, o));
    for (int c0 = 0; c0 < used; c0 += NB) {
      if (c0) load_batch(c0, t);
#pragma unroll
      for (int i = 0; i < NB; i++) {
        const float wi = __shfl_sync(0xffffffffu, w, (c0 + i) & 31);
        if (c0 + i < used) {
#pragma unroll
          for (int v = 0; v < V; v++) acc[v] = __fmaf_rn(t[i][v], wi, acc[v]);
        }
      }
    }
  } else {
    float M = -INFINITY;
    for (int c = lane; c < used; c += 32) M = fmaxf(M, __ldcg(ml + c).x);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    for (int c0 = 0; c0 < used; c0 += NB) {
      float t[NB][V];
      load_batch(c0, t);
#pragma unroll
      for (int i = 0; i < NB; i++) {
        if (c0 + i < used) {
          const float2 m = __ldcg(ml + c0 + i);
          const float wi = expf(m.x - M);
          L = __fadd_rn(L, __fmul_rn(m.y, wi));
#pragma unroll
          for (int v = 0; v < V; v++) acc[v] = __fmaf_rn(t[i][v], wi, acc[v]);
        }
      }
    }
  }
  float* out = a.out + int64_t(j) * HD + lane * V;
  if (V == 4) {
    *reinterpret_cast<float4*>(out) = make_float4(acc[0] / L, acc[1 % V] / L, acc[2 % V] / L, acc[3 % V] / L);
  } else {
    *reinterpret_cast<float2*>(out) = make_float2(acc[0] / L, acc[1 % V] / L);
  }
}

// An item's partials when the items of a kv head run as one thread-block
// cluster: o_c of the G heads ([G][HD] floats), then (m_c, l_c) per head, in the
// item's own K rows, which no thread reads once the scores are formed.
template <int HD, int G, int CM>
__device__ __forceinline__ float* attn_cluster_o(uint8_t* sm) {
  static_assert(size_t(G) * HD * 4 + size_t(G) * 8 <= size_t(CM) * (HD + 8) * 2, "partials fit in the K rows");
  return reinterpret_cast<float*>(sm + AttnLayout<HD, G, CM>::kK);
}
template <int HD, int G, int CM>
__device__ __forceinline__ float2* attn_cluster_ml(uint8_t* sm) {
  return reinterpret_cast<float2*>(sm + AttnLayout<HD, G, CM>::kK + size_t(G) * HD * 4);
}

// Merge of query head g G + h from the partials of the `used` live items of
// kv head g, item c in the shared memory of cluster rank c, by one warp: the
// arithmetic and order of attn_combine_head (used <= 32), with the partials
// read from distributed shared memory instead of global memory.  Call after a
// cluster barrier that follows every item's partial stores.
template <int HD, int G, int CM>
__device__ __forceinline__ void attn_merge_cluster(const AttnArgs& a, int g, int h, int used, int lane,
                                                   uint8_t* sm) {
  namespace cg = cooperative_groups;
  constexpr int V = HD / 32;
  cg::cluster_group cl = cg::this_cluster();
  float2 mv = make_float2(-INFINITY, 0.f);
  if (lane < used) mv = cl.map_shared_rank(attn_cluster_ml<HD, G, CM>(sm), unsigned(lane))[h];
  float M = mv.x;
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w = lane < used ? expf(mv.x - M) : 0.f;
  float L = __fmul_rn(mv.y, w);
#pragma unroll
  for (int o = 16; o; o >>= 1) L = __fadd_rn(L, __shfl_xor_sync(0xffffffffu, L, o));
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; v++) acc[v] = 0.f;
  const float* own = attn_cluster_o<HD, G, CM>(sm) + h * HD + lane * V;
  for (int c = 0; c < used; c++) {
    const float wi = __shfl_sync(0xffffffffu, w, c);
    const float* po = cl.map_shared_rank(own, unsigned(c));
    float t[V];
    if (V == 4) {
      const float4 u = *reinterpret_cast<const float4*>(po);
      t[0] = u.x; t[1 % V] = u.y; t[2 % V] = u.z; t[3 % V] = u.w;
    } else {
      const float2 u = *reinterpret_cast<const float2*>(po);
      t[0] = u.x; t[1 % V] = u.y;
    }
#pragma unroll
    for (int v = 0; v < V; v++) acc[v] = __fmaf_rn(t[v], wi, acc[v]);
  }
  float* out = a.out + int64_t(g * G + h) * HD + lane * V;
  if (V == 4) {
    *reinterpret_cast<float4*>(out) = make_float4(acc[0] / L, acc[1 % V] / L, acc[2 % V] / L, acc[3 % V] / L);
  } else {
    *reinterpret_cast<float2*>(out) = make_float2(acc[0] / L, acc[1 % V] / L);
  }
}

// One item by the whole CTA: kv head g, chunk `chunk` of C positions; n =
// positions attended (pos + 1: the current one is stored by now), used =
// ceil(n / C) items of kv head g exist; rows [0, r_done) of the chunk are
// already being copied (cp.async groups the CTA committed before).  Every
// thread of the CTA must call it.  Returns true on the CTA that merged.
//
// Warp w scores key tiles w, w + 8, ... (8 keys each) against all heads; the
// chunk maximum and sum per head go through shared memory; P (hi and lo rows)
// is written to shared memory; warp w then forms output dimensions
// [8 HD/64 w, 8 HD/64 (w+1)) over all keys.  Sums of the hi and lo rows, of the
// per-warp softmax sums and of the k-steps run in a fixed order, so the result
// does not depend on timing.
template <int HD, int G, int CM, bool CL = false>
__device__ __forceinline__ bool attn_item(const AttnArgs& a, int g, int chunk, int t0, int cnt, int used,
                                          uint8_t* sm, int r_done) {
  using Lay = AttnLayout<HD, G, CM>;
  constexpr int KP = Lay::KP, MT = Lay::MT, PP = Lay::PP, NW = kAttnWarps;
  constexpr int KS = HD / 16;                          // k-steps of the scores (even)
  constexpr int NTW = CM / 8 / NW;                     // score tiles per warp
  constexpr int NVW = HD / 8 / NW;                     // output tiles per warp (1 or 2)
  constexpr int HPT = MT;                              // heads per thread: gi (and gi + 8)
  static_assert(KS % 2 == 0 && NTW >= 1 && (NVW == 1 || NVW == 2) && CM % 64 == 0, "attention tile shape");
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, gi = lane >> 2, tg = lane & 3;
  const uint32_t ks = smem_u32(sm + Lay::kK), vs = smem_u32(sm + Lay::kV), ps = smem_u32(sm + Lay::kP);
  float* red_max = reinterpret_cast<float*>(sm + Lay::kRed);
  float* red_sum = red_max + NW * G;

  // q of this thread's heads as hi/lo A fragments (loads first: the longest latency)
  float2 qv[HPT][KS][2];
  {
    const float* qb = a.q + int64_t(g) * G * HD;
#pragma unroll
    for (int h = 0; h < HPT; h++) {
      const int head = gi + 8 * h;
#pragma unroll
      for (int kk = 0; kk < KS; kk++) {
        if (head < G) {
          qv[h][kk][0] = __ldcg(reinterpret_cast<const float2*>(qb + head * HD + kk * 16 + 2 * tg));
          qv[h][kk][1] = __ldcg(reinterpret_cast<const float2*>(qb + head * HD + kk * 16 + 8 + 2 * tg));
        } else {
          qv[h][kk][0] = qv[h][kk][1] = make_float2(0.f, 0.f);
        }
      }
    }
  }
  // the rows not copied before the wait (the current position's)
  attn_copy_rows<HD, CM>(a, g, t0, r_done, cnt, sm);
  asm volatile("cp.async.commit_group;" ::: "memory");
  // V rows past cnt inside the last 16-key step enter P V with weight 0: make them finite
  {
    const int r1 = min(CM, (cnt + 15) & ~15);
    for (int i = cnt * (HD / 8) + t; i < r1 * (HD / 8); i += kAttnThreads) {
      const int r = i / (HD / 8), c = i % (HD / 8);
      *reinterpret_cast<uint4*>(sm + Lay::kV + size_t(r * KP + c * 8) * 2) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  uint32_t qa[MT][KS][4];
#pragma unroll
  for (int kk = 0; kk < KS; kk++) {
    if (MT == 1) {   // rows gi (hi) and gi + 8 (lo) of one tile
      split2(qv[0][kk][0].x, qv[0][kk][0].y, qa[0][kk][0], qa[0][kk][1]);
      split2(qv[0][kk][1].x, qv[0][kk][1].y, qa[0][kk][2], qa[0][kk][3]);
    } else {         // tile 0: hi of heads gi, gi + 8; tile 1: their lo
      split2(qv[0][kk][0].x, qv[0][kk][0].y, qa[0][kk][0], qa[MT - 1][kk][0]);
      split2(qv[HPT - 1][kk][0].x, qv[HPT - 1][kk][0].y, qa[0][kk][1], qa[MT - 1][kk][1]);
      split2(qv[0][kk][1].x, qv[0][kk][1].y, qa[0][kk][2], qa[MT - 1][kk][2]);
      split2(qv[HPT - 1][kk][1].x, qv[HPT - 1][kk][1].y, qa[0][kk][3], qa[MT - 1][kk][3]);
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // ---- scores of this warp's key tiles ---------------------------------------
  const int nt_live = (cnt + 7) >> 3;
  float s[HPT][NTW][2];
#pragma unroll
  for (int i = 0; i < NTW; i++) {
    const int nt = warp + NW * i;
    if (nt < nt_live) {   // warp-uniform
      float acc[MT][4];
#pragma unroll
      for (int m = 0; m < MT; m++) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
      const uint32_t rowa = ks + uint32_t((nt * 8 + (lane & 7)) * KP + (lane >> 3) * 8) * 2;
#pragma unroll
      for (int kk = 0; kk < KS; kk += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(rowa + uint32_t(kk * 16) * 2, b0, b1, b2, b3);
#pragma unroll
        for (int m = 0; m < MT; m++) {
          mma16816(acc[m], qa[m][kk], b0, b1);
          mma16816(acc[m], qa[m][kk + 1], b2, b3);
        }
      }
#pragma unroll
      for (int e = 0; e < 2; e++) {
        const bool live = nt * 8 + 2 * tg + e < cnt;
        const float v0 = MT == 1 ? __fadd_rn(acc[0][e], acc[0][e + 2]) : __fadd_rn(acc[0][e], acc[MT - 1][e]);
        s[0][i][e] = live ? __fmul_rn(v0, a.scale) : -INFINITY;
        if (HPT == 2) {
          const float v1 = __fadd_rn(acc[0][e + 2], acc[MT - 1][e + 2]);
          s[HPT - 1][i][e] = live ? __fmul_rn(v1, a.scale) : -INFINITY;
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < HPT; h++) s[h][i][0] = s[h][i][1] = -INFINITY;
    }
  }
  // per-warp maxima per head
#pragma unroll
  for (int h = 0; h < HPT; h++) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < NTW; i++) mx = fmaxf(mx, fmaxf(s[h][i][0], s[h][i][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int head = gi + 8 * h;
    if (tg == 0 && head < G) red_max[warp * G + head] = mx;
  }
  __syncthreads();

  // ---- exponentials against the chunk maximum; P rows to shared memory --------
#pragma unroll
  for (int h = 0; h < HPT; h++) {
    const int head = gi + 8 * h;
    float M = -INFINITY;
    if (head < G) {
#pragma unroll
      for (int w = 0; w < NW; w++) M = fmaxf(M, red_max[w * G + head]);
    }
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < NTW; i++) {
      const int key = (warp + NW * i) * 8 + 2 * tg;
      float p0 = 0.f, p1 = 0.f;
      if (head < G) {
        p0 = expf(s[h][i][0] - M);   // exp(-inf) = 0 past cnt
        p1 = expf(s[h][i][1] - M);
      }
      l = __fadd_rn(l, __fadd_rn(p0, p1));
      uint32_t hi, lo;
      split2(p0, p1, hi, lo);
      // MT == 1: row gi hi, row gi + 8 lo; MT == 2: rows head (hi) and 16 + head (lo)
      const int rhi = MT == 1 ? gi : head, rlo = MT == 1 ? gi + 8 : 16 + head;
      *reinterpret_cast<uint32_t*>(sm + Lay::kP + size_t(rhi * PP + key) * 2) = hi;
      *reinterpret_cast<uint32_t*>(sm + Lay::kP + size_t(rlo * PP + key) * 2) = lo;
    }
    l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, 1));
    l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, 2));
    if (tg == 0 && head < G) red_sum[warp * G + head] = l;
  }
  __syncthreads();
  if (t < G) {   // chunk statistics of head t, warps in order
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; w++) M = fmaxf(M, red_max[w * G + t]);
#pragma unroll
    for (int w = 0; w < NW; w++) L = __fadd_rn(L, red_sum[w * G + t]);
    if constexpr (CL) attn_cluster_ml<HD, G, CM>(sm)[t] = make_float2(M, L);   // K rows are read by now
    else a.part_ml[int64_t(g * G + t) * a.n_chunks + chunk] = make_float2(M, L);
  }

  // ---- P V: this warp's output dimension tiles over the live key steps ---------
  {
    const int kv_steps = (cnt + 15) >> 4;
    float acc[MT][NVW][4];
#pragma unroll
    for (int m = 0; m < MT; m++)
#pragma unroll
      for (int j = 0; j < NVW; j++) acc[m][j][0] = acc[m][j][1] = acc[m][j][2] = acc[m][j][3] = 0.f;
    const int n0 = warp * NVW * 8;   // first output dimension of this warp
    // A rows (lane & 7) + 8 ((lane >> 3) & 1), keys + 8 (lane >> 4); V rows likewise for .trans
    const uint32_t pa = ps + uint32_t(((lane & 7) + 8 * ((lane >> 3) & 1)) * PP + 8 * (lane >> 4)) * 2;
    // (with one dimension tile only lanes 0..15 address rows: keys 0..15 of the step)
    const uint32_t va = vs + uint32_t(((lane & 7) + 8 * ((lane >> 3) & 1)) * KP + n0 + (NVW == 2 ? 8 * (lane >> 4) : 0)) * 2;
#pragma unroll 4
    for (int kv = 0; kv < kv_steps; kv++) {
      uint32_t pf[MT][4];
#pragma unroll
      for (int m = 0; m < MT; m++)
        ldsm_x4(pa + uint32_t(m * 16 * PP + kv * 16) * 2, pf[m][0], pf[m][1], pf[m][2], pf[m][3]);
      if (NVW == 2) {   // two dimension tiles of one key step
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(va + uint32_t(kv * 16 * KP) * 2, b0, b1, b2, b3);
#pragma unroll
        for (int m = 0; m < MT; m++) {
          mma16816(acc[m][0], pf[m], b0, b1);
          mma16816(acc[m][NVW - 1], pf[m], b2, b3);
        }
      } else {          // one dimension tile
        uint32_t b0, b1;
        ldsm_x2_t(va + uint32_t(kv * 16 * KP) * 2, b0, b1);
#pragma unroll
        for (int m = 0; m < MT; m++) mma16816(acc[m][0], pf[m], b0, b1);
      }
    }
#pragma unroll
    for (int h = 0; h < HPT; h++) {
      const int head = gi + 8 * h;
      if (head >= G) continue;
      float* po = (CL ? attn_cluster_o<HD, G, CM>(sm) + head * HD
                      : a.part_o + (int64_t(g * G + head) * a.n_chunks + chunk) * HD) + n0 + 2 * tg;
#pragma unroll
      for (int j = 0; j < NVW; j++) {
        float o0, o1;
        if (MT == 1) {
          o0 = __fadd_rn(acc[0][j][0], acc[0][j][2]);
          o1 = __fadd_rn(acc[0][j][1], acc[0][j][3]);
        } else {
          o0 = __fadd_rn(acc[0][j][2 * h], acc[MT - 1][j][2 * h]);
          o1 = __fadd_rn(acc[0][j][2 * h + 1], acc[MT - 1][j][2 * h + 1]);
        }
        *reinterpret_cast<float2*>(po + 8 * j) = make_float2(o0, o1);
      }
    }
  }

  if constexpr (CL) return false;   // the cluster merges (attn_merge_cluster)

  // ---- the CTA that finishes kv head g's last chunk merges its heads --------
  // (the CTA barrier orders every thread's partials before thread 0's fence)
  int* flag = reinterpret_cast<int*>(sm + Lay::kFlag);
  __syncthreads();
  if (t == 0) {
    // release: the CTA's partials (ordered before this by the barrier); acquire:
    // every earlier item's, for the CTA that takes the last ticket
    unsigned ticket;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(a.tickets + g) : "memory");
    *flag = ticket == unsigned(used - 1);
  }
  __syncthreads();
  if (!*flag) return false;
  for (int h = warp; h < G; h += NW) attn_combine_head<HD>(a, g * G + h, used, lane);
  if (t == 0) a.tickets[g] = 0u;
  return true;
}

}  // namespace nt
