// nt_step.cuh -- one whole decode step as a single persistent kernel.
//
// One CTA of kStepWarps warps per SM, all co-resident (cooperative launch).
// Every CTA walks the phases of the step in order:
//
//   embed | per layer: RMSNorm+QKV+RoPE+KV append | attention (+ merge) | O + residual
//         | RMSNorm+gate/up+SwiGLU | down + residual |  RMSNorm+output+top-2 | argmax
//
// There is no grid-wide barrier between phases.  Each phase's input vector is
// consumed in 1024-column tiles, and a tile is used as soon as the rows that
// produce it are written: every finished row group of a producer adds its row
// count to the tile's counter (a release add), a consumer waits until the
// counter reaches the value that phase implies (an acquire load) and one warp
// per CTA then converts the tile into shared memory for all its warps.  So a CTA
// starts a phase while other CTAs still finish the previous one, and HBM stays
// busy across phase changes.  Attention items wait on a per kv head counter of
// the Q/K/V rows written; the CTA that merges a kv head's chunks releases the
// attention output tiles.  Counters only grow: each phase's target is derived
// from the number of completed steps (the epoch) and the layer.  One grid
// barrier remains, before the argmax over the CTAs' top-2 summaries.
//
// Each GEMV is the ring GEMV of nt_gemv_pipe.cuh (same device functions, hence
// the same results bit for bit as the per-launch kernels), and each warp copies
// its first ring tiles of the next GEMV as soon as it has finished its share of
// the current one.  Attention items use the whole CTA and its whole shared
// memory; their rows cached by earlier steps are copied before the wait for
// the current position's K and V.
//
// Every wait (counter, shared-memory flag, barrier) gives up after about a
// second: it sets the error word, which makes every later wait return at once,
// so the kernel runs to its end on stale data and the host reports the step as
// abandoned.  A launch that starts with the error word set does nothing.
#pragma once

#include <mutex>

#include "nt_attn.cuh"
#include "nt_gemv_pipe.cuh"

namespace nt {

constexpr int kStepWarps = 16;
constexpr int kStepThreads = kStepWarps * 32;
static_assert(kStepThreads == kAttnThreads, "attention items use the whole CTA");
constexpr int kStepMaxTiles = 32;          // 1024-column tiles of the widest vector (32768 columns)

// Every warp owns a fixed ring slice for all GEMVs of the step (the size of four
// Q8_0 tiles of two rows), so it can copy the next GEMV's first tiles as soon
// as it has finished its own share of the current one.  Ring depth per format:
// as many two-row tiles as fit, at most 8.
constexpr int kStepSlice = 4 * 2 * (32 * 32 + 64);
template <int FMT>
struct StepRing {
  static constexpr int S = int(kStepSlice / (2 * Pipe<FMT>::RB)) < 8 ? int(kStepSlice / (2 * Pipe<FMT>::RB)) : 8;
};
constexpr size_t kStepRingBytes = size_t(kStepWarps) * kStepSlice;

// Device sync state of the step kernel (unsigned words): the final barrier's
// arrivals and base, the epoch (completed steps), then the readiness counters.
enum : int {
  SYNC_ARRIVE = 0, SYNC_BASE = 1, SYNC_EPOCH = 2,
  SYNC_X = 32,                         // per tile of x: rows written (embedding, O, down)
  SYNC_U = SYNC_X + kStepMaxTiles,     // per tile of u: elements written (SwiGLU)
  SYNC_ATT = SYNC_U + kStepMaxTiles,   // per tile of the attention output: elements merged
  SYNC_KV = SYNC_ATT + kStepMaxTiles,  // per kv head: Q/K/V rows written
  SYNC_WORDS = SYNC_KV + kStepMaxTiles
};

struct StepGemv {
  GemvArgs a;
  int64_t nrows = 0;
};

// GEMV table per layer: QK (or QKV when v shares the format), V, O, gate/up, down.
enum : int { SG_QK = 0, SG_V = 1, SG_O = 2, SG_GU = 3, SG_DOWN = 4, SG_PER_LAYER = 5 };

struct StepArgs {
  // GEMVs of layer 0 (SG_* order) and the output head (index SG_PER_LAYER); the
  // GEMVs of layer l read weights layer_delta[l] bytes further on (every layer
  // blob has the same layout) and layer l's K/V cache.
  const StepGemv* gemv = nullptr;
  const int64_t* layer_delta = nullptr;   // [n_layers]
  int n_layers = 0;
  int split_v = 0;                  // v has its own format: QK and V are two GEMVs
  // embedding
  QMat embd;
  float* x = nullptr;
  int hidden = 0;
  // attention (kc/vc set per layer from the cache base)
  AttnArgs attn;
  const __half* kv = nullptr;       // [layer][K|V][n_kv][max_ctx][hd]
  int64_t kv_layer_elems = 0;
  int n_kv = 0;
  int attn_qd = 0, attn_kd = 0;     // rows of q and of k in the QKV GEMV
  // head and bookkeeping
  float4* top2 = nullptr;           // [gridDim.x]
  int32_t* small = nullptr;         // pos, token, next, margin bits, error word
  int32_t* hist = nullptr;
  int max_ctx = 0, vocab = 0;
  unsigned* bar = nullptr;          // SYNC_WORDS words of sync state
  long long* stamps = nullptr;      // nullable: clock64 of CTA 0 at the start and after every phase
  uint32_t ring_off = 0;            // dynamic shared memory: [x staging / attention | ring]
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait of the calling thread until *ctr has reached target (modulo 2^32).
// On the time limit it sets the error word; with the error word set it returns
// at once.
__device__ __forceinline__ void wait_count(const unsigned* ctr, unsigned target, volatile int32_t* err) {
  if (int(ld_acquire_u32(ctr) - target) >= 0) return;
  const unsigned long long t0 = globaltimer_ns();
  for (unsigned it = 0;; it++) {
    __nanosleep(32);
    if (int(ld_acquire_u32(ctr) - target) >= 0) return;
    if (*err) return;
    if ((it & 63u) == 63u && (globaltimer_ns() - t0 > 1000000000ull || it > (1u << 26))) {
      *err = 1;
      return;
    }
  }
}

// Signal kinds of a GEMV's finished row groups.
enum : int { SIG_NONE = 0, SIG_X = 1, SIG_U = 2, SIG_KV = 3 };

// Hooks of the step kernel's GEMVs (see pipe_loop): on-demand staging of the
// input tiles after their readiness counters, and release of the output rows.
struct StepHooks {
  static constexpr bool kAllStaged = false;
  const unsigned* ready = nullptr;   // input tile counters (nullptr: input complete)
  unsigned target = 0;
  unsigned* signal = nullptr;        // output counters
  int kind = SIG_NONE;
  int qd = 0, kd = 0, hd = 1, G = 1;  // SIG_KV: row -> kv head
  unsigned* tstate = nullptr;        // shared: per input tile, 2*tag (claimed) / 2*tag+1 (staged)
  unsigned tag = 0;
  volatile int32_t* err = nullptr;

  template <int FMT, int XS>
  __device__ __forceinline__ void tile(const GemvArgs& a, uint8_t* xq, int k) {
    const int lane = threadIdx.x & 31;
    volatile unsigned* st = tstate + k;
    const unsigned staged = 2 * tag + 1, claimed = 2 * tag;
    int mine = 0;
    if (lane == 0) {
      unsigned v = *st;
      if (v != staged && v != claimed) mine = atomicCAS(tstate + k, v, claimed) == v;
    }
    mine = __shfl_sync(0xffffffffu, mine, 0);
    if (mine) {
      if (lane == 0 && ready) wait_count(ready + k, target, err);
      __syncwarp();
      stage_tile<FMT, XS>(a.x + a.col0, k, xq);
      __syncwarp();
      __threadfence_block();
      if (lane == 0) atomicExch(tstate + k, staged);
    } else {
      if (lane == 0 && *st != staged) {
        const unsigned long long t0 = globaltimer_ns();
        for (unsigned it = 0; *st != staged; it++) {
          __nanosleep(32);
          if (*err) break;
          if ((it & 63u) == 63u && (globaltimer_ns() - t0 > 1000000000ull || it > (1u << 26))) {
            *err = 1;
            break;
          }
        }
      }
      __syncwarp();
      __threadfence_block();
    }
  }

  // At the start of a GEMV: warp w claims and stages tiles w, w + 16, ... as their
  // inputs become ready, so the tiles are staged in parallel rather than in the
  // order the first row group reaches them.
  template <int FMT, int XS>
  __device__ __forceinline__ void prestage(const GemvArgs& a, uint8_t* xq) {
    const int kt = int(a.ncols / 1024);
    for (int k = threadIdx.x >> 5; k < kt; k += kStepWarps) tile<FMT, XS>(a, xq, k);
  }

  __device__ __forceinline__ void group_done(const GemvArgs& a, int64_t grp, int nlive) {
    if (kind == SIG_NONE) return;
    __syncwarp();   // the epilogue's stores of every lane before lane 0's release
    if ((threadIdx.x & 31) != 0) return;
    const int row = int(grp * 2);   // R = 2
    int idx;
    unsigned amount = unsigned(nlive);
    if (kind == SIG_X) {
      idx = row >> 10;
    } else if (kind == SIG_U) {
      idx = (row >> 1) >> 10;
      amount = unsigned(nlive >> 1);
    } else {
      const int L = a.epi.row_base + row;
      idx = L < qd ? (L / hd) / G : (L < qd + kd ? (L - qd) / hd : (L - qd - kd) / hd);
    }
    red_release_add(signal + idx, amount);
  }
};

struct GridBarrier {
  unsigned* cnt;
  volatile int32_t* err;
  unsigned target;
  unsigned n;

  __device__ __forceinline__ void sync() {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(cnt, 1u);
      target += n;
      wait_count(cnt, target, err);
      __threadfence();
    }
    __syncthreads();
  }
};

// The phases are separate (not inlined) functions so that each gets its own
// register allocation under the kernel's 128-register cap.
template <int FMT, int EPI>
__device__ __noinline__ void step_prologue(const StepGemv& g, uint8_t* ring) {
  pipe_prologue<FMT, 2, StepRing<FMT>::S, kStepWarps, kStepSlice>(g.a, g.nrows, blockIdx.x, gridDim.x, ring);
}
template <int FMT, int EPI>
__device__ __noinline__ void step_gemv(const StepGemv& g, uint8_t* xq, uint8_t* ring, StepHooks& h) {
  h.template prestage<FMT, x_slices(EPI)>(g.a, xq);
  pipe_loop<FMT, 2, StepRing<FMT>::S, EPI, kStepWarps, kStepSlice>(g.a, g.nrows, blockIdx.x, gridDim.x, xq, ring,
                                                                   1.0f, h);
}

// Attention items of this CTA for one layer: items c, c + ncta, ... of the
// n_kv x used (kv head, chunk) items.  Each copies its rows cached by earlier
// steps, waits for its kv head's Q/K/V rows, runs; the CTA that merged a kv
// head releases that head's attention output.
template <int HD, int G>
__device__ __noinline__ void step_attention(const AttnArgs& aa, int n_kv, int n_ctx, uint8_t* sm,
                                            const unsigned* kv_ready, unsigned kv_target, unsigned* att_ready,
                                            volatile int32_t* err) {
  const int used = (n_ctx + aa.chunk - 1) / aa.chunk;
  const int items = n_kv * used, ncta = gridDim.x;
  for (int it = blockIdx.x; it < items; it += ncta) {
    const int g = it / used, chunk = it % used;
    attn_prefetch<HD>(aa, g, chunk, n_ctx - 1, sm);
    if (threadIdx.x == 0) wait_count(kv_ready + g, kv_target, err);
    __syncthreads();
    const bool merged = aa.chunk == 64    ? attn_item<HD, G, 64>(aa, g, chunk, n_ctx, used, sm, true)
                        : aa.chunk == 128 ? attn_item<HD, G, 128>(aa, g, chunk, n_ctx, used, sm, true)
                                          : attn_item<HD, G, 256>(aa, g, chunk, n_ctx, used, sm, true);
    if (merged) {
      __syncthreads();   // every head of kv head g merged
      if (threadIdx.x == 0) {
        __threadfence();
        const int r0 = g * G * HD, r1 = r0 + G * HD;
        for (int t = r0 >> 10; t <= (r1 - 1) >> 10; t++)
          red_release_add(att_ready + t, unsigned(min(r1, (t + 1) << 10) - max(r0, t << 10)));
      }
    }
    __syncthreads();   // shared memory reused by the next item
  }
}

// Layer l's copy of a layer-0 GEMV: weight streams moved by delta bytes, its
// own K/V cache for the QKV epilogue.
__device__ __forceinline__ void rebase_gemv(GemvArgs& dst, const GemvArgs& src, int64_t delta, __half* kc,
                                            __half* vc) {
  dst = src;
  for (int i = 0; i < src.nseg; i++) {
    QMat& q = dst.seg[i];
    if (q.q) q.q += delta;
    if (q.qh) q.qh += delta;
    if (q.meta) q.meta += delta;
    if (q.d) q.d = reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(q.d) + delta);
  }
  dst.epi.k_cache = kc;
  dst.epi.v_cache = vc;
}

__device__ __forceinline__ AttnArgs layer_attn(const StepArgs& s, int l) {
  AttnArgs aa = s.attn;
  aa.kc = s.kv + (int64_t(l) * 2 + 0) * s.kv_layer_elems;
  aa.vc = s.kv + (int64_t(l) * 2 + 1) * s.kv_layer_elems;
  return aa;
}

// Largest entry over the CTA summaries (ties to the lowest row), the gap to the
// second largest, then the step's bookkeeping.  Run by the first 256 threads
// of one CTA; bit-identical to the per-launch argmax kernel's result.
__device__ __forceinline__ void argmax_finish(const float4* top2, int n, int32_t* small, int32_t* hist, int max_ctx,
                                              int vocab, uint8_t* scratch) {
  float* sb = reinterpret_cast<float*>(scratch);
  float* ss = sb + 256;
  int* si = reinterpret_cast<int*>(ss + 256);
  const int t = threadIdx.x;
  float b = -INFINITY, s = -INFINITY;
  int bi = 0x7fffffff;
  if (t < 256) {
    for (int i = t; i < n; i += 256) {
      const float4 v = __ldcg(top2 + i);
      top2_merge(v.x, __float_as_int(v.y), v.z, b, bi, s);
    }
    sb[t] = b;
    ss[t] = s;
    si[t] = bi;
  }
  __syncthreads();
  if (t == 0) {
    for (int u = 1; u < 256; u++) top2_merge(sb[u], si[u], ss[u], b, bi, s);
    if (bi < 0 || bi >= vocab) bi = 0;     // no finite logit at all: keep the id in range
    const int p = small[0];
    small[2] = bi;
    reinterpret_cast<float*>(small)[3] = b - s;
    if (p < max_ctx) hist[p] = bi;
    small[1] = bi;
    small[0] = p + 1;
  }
}

template <int F_QK, int F_V, int F_O, int F_GU, int F_D, int F_OUT, int HD, int G>
__global__ void __launch_bounds__(kStepThreads, 1) k_step(const __grid_constant__ StepArgs s) {
  static_assert((F_V == NT_Q8_0) == (F_QK == NT_Q8_0), "a separate V GEMV reuses the staged x of Q/K");
  extern __shared__ float4 smem4[];
  uint8_t* const xq = reinterpret_cast<uint8_t*>(smem4);
  uint8_t* const ring = xq + s.ring_off;
  const int cta = blockIdx.x, ncta = gridDim.x, tid = threadIdx.x;
  volatile int32_t* err = s.small + 4;
  if (__ldcg(s.small + 4)) return;   // an earlier step was abandoned

  // GEMV arguments live in shared memory: the head's, and those of two layers
  // (the current one and the next, prepared a phase ahead) by five threads of warp 1
  __shared__ StepGemv s_head;
  __shared__ StepGemv s_layer[2][SG_PER_LAYER];
  __shared__ unsigned s_tile[kStepMaxTiles];
  auto prepare_layer = [&](int l) {
    const int r = tid - 32;
    if (r >= 0 && r < SG_PER_LAYER && l < s.n_layers) {
      StepGemv& d = s_layer[l & 1][r];
      rebase_gemv(d.a, s.gemv[r].a, __ldg(s.layer_delta + l),
                  const_cast<__half*>(s.kv) + (int64_t(l) * 2 + 0) * s.kv_layer_elems,
                  const_cast<__half*>(s.kv) + (int64_t(l) * 2 + 1) * s.kv_layer_elems);
      d.nrows = s.gemv[r].nrows;
    }
  };
  if (tid == SG_PER_LAYER) s_head = s.gemv[SG_PER_LAYER];
  if (tid < kStepMaxTiles) s_tile[tid] = 0u;
  prepare_layer(0);

  const unsigned epoch = __ldcg(s.bar + SYNC_EPOCH);
  const unsigned L = unsigned(s.n_layers);
  const unsigned kv_rows = unsigned((G + 2) * HD);
  const unsigned x_base = epoch * (2 * L + 1) * 1024u, u_base = epoch * L * 1024u;
  const unsigned kv_base = epoch * L * kv_rows;
  unsigned* const x_ready = s.bar + SYNC_X;
  unsigned* const u_ready = s.bar + SYNC_U;
  unsigned* const att_ready = s.bar + SYNC_ATT;
  unsigned* const kv_ready = s.bar + SYNC_KV;
  unsigned tag = 0;
  auto hooks = [&](const unsigned* ready, unsigned target, unsigned* signal, int kind) {
    StepHooks h;
    h.ready = ready;
    h.target = target;
    h.signal = signal;
    h.kind = kind;
    h.qd = s.attn_qd;
    h.kd = s.attn_kd;
    h.hd = HD;
    h.G = G;
    h.tstate = s_tile;
    h.tag = ++tag;
    h.err = err;
    return h;
  };
  auto stamp = [&](int k) {
    if (s.stamps && cta == 0 && tid == 0) s.stamps[k] = clock64();
  };
  stamp(0);
  __syncthreads();

  // ---- embedding row of the current token; releases x ----------------------------
  {
    int64_t tok = __ldcg(s.small + 1);
    if (tok < 0 || tok >= s.embd.rows) tok = 0;   // ids come validated from the host or from the argmax
    const int i0 = cta * kStepThreads;
    if (i0 < s.hidden) {
      if (i0 + tid < s.hidden) s.x[i0 + tid] = dequant_elem(s.embd, tok * s.embd.cols + i0 + tid);
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        red_release_add(x_ready + (i0 >> 10), unsigned(min(kStepThreads, s.hidden - i0)));
      }
    }
  }
  if (s.n_layers > 0) step_prologue<F_QK, EPI_QKV>(s_layer[0][SG_QK], ring);
  else step_prologue<F_OUT, EPI_LOGITS>(s_head, ring);
  __syncthreads();
  stamp(1);

  const int n_ctx = __ldcg(s.small + 0) + 1;
  for (int l = 0; l < s.n_layers; l++) {
    const StepGemv* lg = s_layer[l & 1];
    const unsigned ul = unsigned(l);
    // ---- RMSNorm -> Q|K|V -> RoPE -> cache; releases the kv heads' rows -------------
    {
      StepHooks h = hooks(x_ready, x_base + (2 * ul + 1) * 1024u, kv_ready, SIG_KV);
      step_gemv<F_QK, EPI_QKV>(lg[SG_QK], xq, ring, h);
      if (s.split_v) {   // same staged x (both nibble formats), same tag
        step_prologue<F_V, EPI_QKV>(lg[SG_V], ring);
        step_gemv<F_V, EPI_QKV>(lg[SG_V], xq, ring, h);
      }
    }
    __syncthreads();
    stamp(2 + 5 * l);

    // ---- attention over positions 0..pos, merged by the last CTA per kv head ----
    step_attention<HD, G>(layer_attn(s, l), s.n_kv, n_ctx, xq, kv_ready, kv_base + (ul + 1) * kv_rows, att_ready,
                          err);
    prepare_layer(l + 1);   // published by the next __syncthreads
    step_prologue<F_O, EPI_ADD>(lg[SG_O], ring);
    __syncthreads();
    stamp(3 + 5 * l);

    // ---- O + residual; releases x ---------------------------------------------------
    {
      StepHooks h = hooks(att_ready, u_base + (ul + 1) * 1024u, x_ready, SIG_X);
      step_gemv<F_O, EPI_ADD>(lg[SG_O], xq, ring, h);
    }
    step_prologue<F_GU, EPI_SWIGLU>(lg[SG_GU], ring);
    __syncthreads();
    stamp(4 + 5 * l);

    // ---- RMSNorm -> gate|up -> SwiGLU; releases u ---------------------------------------
    {
      StepHooks h = hooks(x_ready, x_base + (2 * ul + 2) * 1024u, u_ready, SIG_U);
      step_gemv<F_GU, EPI_SWIGLU>(lg[SG_GU], xq, ring, h);
    }
    step_prologue<F_D, EPI_ADD>(lg[SG_DOWN], ring);
    __syncthreads();
    stamp(5 + 5 * l);

    // ---- down + residual; releases x --------------------------------------------------
    {
      StepHooks h = hooks(u_ready, u_base + (ul + 1) * 1024u, x_ready, SIG_X);
      step_gemv<F_D, EPI_ADD>(lg[SG_DOWN], xq, ring, h);
    }
    if (l + 1 < s.n_layers) step_prologue<F_QK, EPI_QKV>(s_layer[(l + 1) & 1][SG_QK], ring);
    else step_prologue<F_OUT, EPI_LOGITS>(s_head, ring);
    __syncthreads();
    stamp(6 + 5 * l);
  }

  // ---- final RMSNorm -> output -> per-CTA top-2, then the one grid barrier -----------
  {
    StepHooks h = hooks(x_ready, x_base + (2 * L + 1) * 1024u, nullptr, SIG_NONE);
    step_gemv<F_OUT, EPI_LOGITS>(s_head, xq, ring, h);
  }
  GridBarrier bar;
  bar.cnt = s.bar + SYNC_ARRIVE;
  bar.err = err;
  bar.n = unsigned(ncta);
  bar.target = __ldcg(s.bar + SYNC_BASE);
  bar.sync();
  stamp(2 + 5 * s.n_layers);
  if (cta == 0) {
    argmax_finish(s.top2, ncta, s.small, s.hist, s.max_ctx, s.vocab, xq);
    if (tid == 0) {
      s.bar[SYNC_BASE] = bar.target;    // base of the next launch's barrier
      s.bar[SYNC_EPOCH] = epoch + 1u;
      stamp(3 + 5 * s.n_layers);
    }
  }
}

// Host side -------------------------------------------------------------------

// Cooperative launch of one instantiation: one CTA per SM.
template <int F_QK, int F_V, int F_O, int F_GU, int F_D, int F_OUT, int HD, int G>
cudaError_t launch_step_t(const StepArgs& a, size_t smem, cudaStream_t s) {
  auto kern = k_step<F_QK, F_V, F_O, F_GU, F_D, F_OUT, HD, G>;
  static const KernelSetup setup = kernel_setup(kern, 0);
  if (setup.err != cudaSuccess) return setup.err;
  const int sms = setup.sms;
  {   // the kernel's shared-memory limit only grows, so a launch never finds it below its own request
    static std::mutex mu;
    static size_t set_smem = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (set_smem < smem) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e != cudaSuccess) return e;
      set_smem = smem;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(sms));
  cfg.blockDim = dim3(unsigned(kStepThreads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Whether one CTA per SM with `smem` bytes of dynamic shared memory can be
// resident (a cooperative launch needs every CTA resident at once).
template <int F_QK, int F_V, int F_O, int F_GU, int F_D, int F_OUT, int HD, int G>
cudaError_t step_fits_t(size_t smem, bool* ok) {
  auto kern = k_step<F_QK, F_V, F_O, F_GU, F_D, F_OUT, HD, G>;
  *ok = false;
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  int dev = 0, optin = 0;
  if ((e = cudaGetDevice(&dev))) return e;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev))) return e;
  if (smem + fa.sharedSizeBytes > size_t(optin)) return cudaSuccess;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)))) return e;
  int occ = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kStepThreads, smem))) return e;
  *ok = occ >= 1;
  return cudaSuccess;
}

struct StepPlan {
  int f_qk, f_v, f_o, f_gu, f_d, f_out, hd, G;
};

// Dynamic shared memory of k_step for a plan: x staging of the widest GEMV then
// the warps' ring slices, or an attention item if that is larger (the two are
// never live at once).
size_t step_smem(const StepPlan& p, int64_t max_cols, int64_t qkv_cols, int attn_chunk, size_t* ring_off);

// Launches k_step for the plan (cooperative, one CTA per SM); whether it fits
// with `smem` bytes.  Both return cudaErrorNotSupported when no instantiation
// matches the plan.
cudaError_t launch_step(const StepPlan& p, const StepArgs& a, size_t smem, cudaStream_t s);
cudaError_t step_fits(const StepPlan& p, size_t smem, bool* ok);

#define NT_STEP_PLAN_DECL(NAME)                                                      \
  cudaError_t launch_step_##NAME(const StepArgs& a, size_t smem, cudaStream_t s); \
  cudaError_t step_fits_##NAME(size_t smem, bool* ok);
NT_STEP_PLAN_DECL(q8_0_g4)
NT_STEP_PLAN_DECL(q4_k_m_g8)
#undef NT_STEP_PLAN_DECL

}  // namespace nt
