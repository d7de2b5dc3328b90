// nt_attn.cuh -- GQA decode attention over the f16 KV cache, as device
// functions for one CTA of kAttnThreads threads, so the per-launch kernel and
// the persistent step kernel run the same arithmetic.
//
// Split context: item (kv head g, chunk c) scores the G = n_heads/n_kv_heads
// query heads that share g against the chunk's C cached keys (C = 64, 128 or
// 256, fixed per model by its maximum context), keeps the chunk's softmax
// statistics (max m_c, sum of exp l_c) and the unnormalised exp-weighted sum o_c
// of its values.  The CTA that finishes the last chunk of kv head g (an atomic
// ticket per kv head) merges the chunks of g's heads, one warp per head:
// M = max m_c, o = sum o_c e^(m_c - M) / sum l_c e^(m_c - M).
#pragma once

#include <cstdlib>

#include "nt_internal.cuh"

namespace nt {

constexpr int kAttnThreads = 512;
constexpr int kAttnMaxChunk = 256;

// Cached positions per item: as short as keeps the items of a full context
// within about one per SM (at most 256); NT_ATTN_CHUNK (64, 128 or 256)
// overrides.  Fixed per model: every path of a model splits the same way.
inline int attn_chunk_len(int max_ctx) {
  if (const char* e = getenv("NT_ATTN_CHUNK")) {
    const int c = atoi(e);
    if (c == 64 || c == 128 || c == 256) return c;
  }
  return max_ctx <= 1024 ? 64 : (max_ctx <= 2048 ? 128 : 256);
}

struct AttnArgs {
  const float* q = nullptr;         // [n_heads][hd], RoPE applied
  const __half* kc = nullptr;       // this layer's K: [n_kv][max_ctx][hd]
  const __half* vc = nullptr;
  int max_ctx = 0;
  int chunk = 64;                   // C
  float scale = 1.f;                // 1/sqrt(hd)
  float* part_o = nullptr;          // [n_heads][n_chunks][hd]
  float2* part_ml = nullptr;        // [n_heads][n_chunks] (m_c, l_c)
  int n_chunks = 0;                 // chunk stride of the partials
  unsigned* tickets = nullptr;      // [n_kv]: finished chunks of the current layer (0 between layers)
  float* out = nullptr;             // [n_heads][hd]
};

// Shared memory of one item: K and V rows (padded: 16-byte reads of 8 rows hit
// distinct banks), q of the G heads, the G x C scores, the P V partial sums of
// the kAttnThreads/hd position slices, a flag.
__host__ __device__ constexpr size_t attn_item_smem(int hd, int G, int C) {
  return size_t(2 * C * (hd + 8)) * 2 + size_t(G * hd + G * C) * 4 + size_t(2 * kAttnThreads / hd) * G * hd * 4 + 16;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void attn_cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Copies of rows [r0, r1) of the item's K and V (chunk-relative) into shared memory.
template <int HD>
__device__ __forceinline__ void attn_copy_rows(const AttnArgs& a, int g, int t0, int r0, int r1, uint8_t* sm) {
  constexpr int KP = HD + 8, VPR = HD / 8;
  const __half* kb = a.kc + (int64_t(g) * a.max_ctx + t0) * HD;
  const __half* vb = a.vc + (int64_t(g) * a.max_ctx + t0) * HD;
  const uint32_t ks = smem_u32(sm), vs = ks + uint32_t(a.chunk * KP) * 2;
  for (int i = r0 * VPR + int(threadIdx.x); i < r1 * VPR; i += kAttnThreads) {
    const int r = i / VPR, c = i % VPR;
    attn_cp16(ks + uint32_t(r * KP + c * 8) * 2, kb + r * HD + c * 8);
    attn_cp16(vs + uint32_t(r * KP + c * 8) * 2, vb + r * HD + c * 8);
  }
}

// Before the current position is known to be written: the item's rows of the
// positions cached by earlier steps (t < pos).  attn_item(..., prefetched=true)
// then copies only the rest.
template <int HD>
__device__ __forceinline__ void attn_prefetch(const AttnArgs& a, int g, int chunk, int pos, uint8_t* sm) {
  const int t0 = chunk * a.chunk;
  const int r1 = min(a.chunk, pos - t0);
  if (r1 > 0) attn_copy_rows<HD>(a, g, t0, 0, r1, sm);
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Merge of the `used` chunks of query head j by one warp (lane holds HD/32
// dimensions); chunk loads are issued eight at a time; sums run over c in
// increasing order.
template <int HD>
__device__ __forceinline__ void attn_combine_head(const AttnArgs& a, int j, int used, int lane) {
  constexpr int V = HD / 32;
  const float2* ml = a.part_ml + int64_t(j) * a.n_chunks;
  float M = -INFINITY;
  for (int c = lane; c < used; c += 32) M = fmaxf(M, __ldcg(ml + c).x);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; v++) acc[v] = 0.f;
  float L = 0.f;
  const float* pj = a.part_o + int64_t(j) * a.n_chunks * HD + lane * V;
  for (int c0 = 0; c0 < used; c0 += 32) {
    const int c = c0 + lane;
    float w = 0.f, lw = 0.f;
    if (c < used) {
      const float2 m = __ldcg(ml + c);
      w = expf(m.x - M);
      lw = __fmul_rn(m.y, w);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) lw = __fadd_rn(lw, __shfl_xor_sync(0xffffffffu, lw, o));
    L = __fadd_rn(L, lw);
    const int n = min(32, used - c0);
    for (int i0 = 0; i0 < n; i0 += 8) {
      float t[8][V];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        if (i0 + i < n) {
          const float* po = pj + int64_t(c0 + i0 + i) * HD;
          if (V == 4) {
            const float4 u = __ldcg(reinterpret_cast<const float4*>(po));
            t[i][0] = u.x; t[i][1 % V] = u.y; t[i][2 % V] = u.z; t[i][3 % V] = u.w;
          } else {
            const float2 u = __ldcg(reinterpret_cast<const float2*>(po));
            t[i][0] = u.x; t[i][1 % V] = u.y;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const float wi = __shfl_sync(0xffffffffu, w, (i0 + i) & 31);
        if (i0 + i < n) {
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

// One item by the whole CTA (C = a.chunk, a compile-time copy).  n = cached
// positions attended (pos + 1; the current one is already stored), used =
// ceil(n / C) items of kv head g exist.  Scores: threads 2c and 2c+1 hold the
// two halves of key c in registers and score it against every head (q read as
// broadcast float4s; even and odd dimensions in the two lanes of packed f32x2
// FMAs, added at the end).  P V: the CTA's threads are 2*kAttnThreads/HD
// position slices x HD/2 dimension pairs (packed f32x2 FMAs on a pair); slice s
// sums its contiguous share of the chunk for all G heads, and the slices are
// added in order.  Every thread of the CTA must call it.
template <int HD, int G, int C>
__device__ __forceinline__ bool attn_item(const AttnArgs& a, int g, int chunk, int n, int used, uint8_t* sm,
                                          bool prefetched) {
  constexpr int KP = HD + 8, NS = 2 * kAttnThreads / HD;
  __half* Ks = reinterpret_cast<__half*>(sm);
  __half* Vs = Ks + C * KP;
  float* qs = reinterpret_cast<float*>(Vs + C * KP);
  float* S = qs + G * HD;                      // [G][C]
  float* P = S + G * C;                        // [NS][G][HD]
  int* flag = reinterpret_cast<int*>(P + NS * G * HD);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int t0 = chunk * C;
  const int cnt = min(C, n - t0);
  const int pos = n - 1;
  // every copy of the chunk issued before any is waited for: one memory latency
  attn_copy_rows<HD>(a, g, t0, prefetched ? max(0, min(cnt, pos - t0)) : 0, cnt, sm);
  {
    const uint32_t qss = smem_u32(qs);
    for (int i = t; i < G * HD / 4; i += kAttnThreads) attn_cp16(qss + i * 16, a.q + int64_t(g) * G * HD + i * 4);
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // ---- scores: two threads per key (measured faster than spreading a key over
  // more threads when C < 256), each half of its dimensions ----
  if (t < 2 * C) {
    constexpr int TPK = 2, DPT = HD / TPK;
    const int c = t / TPK, part = t % TPK;
    float2 kf[DPT / 2];
    const uint4* kr = reinterpret_cast<const uint4*>(Ks + c * KP + part * DPT);
#pragma unroll
    for (int i = 0; i < DPT / 8; i++) {
      const uint4 v = kr[i];
      const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
      for (int j = 0; j < 4; j++) kf[i * 4 + j] = __half22float2(h2[j]);
    }
#pragma unroll
    for (int h = 0; h < G; h++) {
      const float4* qh = reinterpret_cast<const float4*>(qs + h * HD + part * DPT);
      float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);   // two chains: dimensions 8i..8i+3, 8i+4..8i+7
#pragma unroll
      for (int i = 0; i < DPT / 4; i += 2) {
        const float4 qv = qh[i], qw = qh[i + 1];
        a0 = __ffma2_rn(make_float2(qv.x, qv.y), kf[2 * i], a0);
        a1 = __ffma2_rn(make_float2(qw.x, qw.y), kf[2 * i + 2], a1);
        a0 = __ffma2_rn(make_float2(qv.z, qv.w), kf[2 * i + 1], a0);
        a1 = __ffma2_rn(make_float2(qw.z, qw.w), kf[2 * i + 3], a1);
      }
      float acc = __fadd_rn(__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y));
#pragma unroll
      for (int o = 1; o < TPK; o <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
      if (part == 0) S[h * C + c] = c < cnt ? __fmul_rn(acc, a.scale) : -INFINITY;
    }
  }
  __syncthreads();

  // ---- chunk softmax statistics (max, sum of exp), weights in place ---------
  for (int h = warp; h < G; h += kAttnThreads / 32) {
    float mx = -INFINITY;
    for (int c = lane; c < C; c += 32) mx = fmaxf(mx, S[h * C + c]);
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float l = 0.f;
    for (int c = lane; c < C; c += 32) {
      const float e = c < cnt ? expf(S[h * C + c] - mx) : 0.f;
      S[h * C + c] = e;
      l = __fadd_rn(l, e);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, o));
    if (lane == 0) a.part_ml[int64_t(g * G + h) * a.n_chunks + chunk] = make_float2(mx, l);
  }
  __syncthreads();

  // ---- P V: slice s of the positions, dimension pair (2dp, 2dp+1) -------------------
  {
    const int dp = t % (HD / 2), s = t / (HD / 2);
    const int span = C / NS;                   // positions per slice (a multiple of 4)
    const int c_lo = s * span, c_hi = min(c_lo + span, cnt);
    float2 acc[G];
#pragma unroll
    for (int h = 0; h < G; h++) acc[h] = make_float2(0.f, 0.f);
    for (int c = c_lo; c < c_hi; c += 4) {     // weights past cnt are 0; rows past cnt are finite smem
      float2 v[4];
#pragma unroll
      for (int j = 0; j < 4; j++)
        v[j] = c + j < cnt ? __half22float2(*reinterpret_cast<const __half2*>(Vs + (c + j) * KP + 2 * dp))
                           : make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < G; h++) {
        const float4 w = *reinterpret_cast<const float4*>(S + h * C + c);
        acc[h] = __ffma2_rn(make_float2(w.w, w.w), v[3], acc[h]);
        acc[h] = __ffma2_rn(make_float2(w.z, w.z), v[2], acc[h]);
        acc[h] = __ffma2_rn(make_float2(w.y, w.y), v[1], acc[h]);
        acc[h] = __ffma2_rn(make_float2(w.x, w.x), v[0], acc[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < G; h++) *reinterpret_cast<float2*>(P + (s * G + h) * HD + 2 * dp) = acc[h];
  }
  __syncthreads();
  for (int i = t; i < G * HD; i += kAttnThreads) {
    float o = P[i];
#pragma unroll
    for (int s = 1; s < NS; s++) o = __fadd_rn(o, P[s * G * HD + i]);
    const int h = i / HD, d = i % HD;
    a.part_o[(int64_t(g * G + h) * a.n_chunks + chunk) * HD + d] = o;
  }

  // ---- the CTA that finishes kv head g's last chunk merges its heads --------
  // (the CTA barrier orders every thread's partials before thread 0's fence)
  __syncthreads();
  if (t == 0) {
    __threadfence();
    const unsigned ticket = atomicAdd(a.tickets + g, 1u);
    *flag = ticket == unsigned(used - 1);
    __threadfence();
  }
  __syncthreads();
  const bool last = *flag;
  __syncthreads();   // the flag slot is free again before any later item writes it
  if (!last) return false;
  for (int h = warp; h < G; h += kAttnThreads / 32) attn_combine_head<HD>(a, g * G + h, used, lane);
  if (t == 0) a.tickets[g] = 0u;
  return true;
}

}  // namespace nt
