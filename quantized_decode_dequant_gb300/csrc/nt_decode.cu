// nt_decode.cu -- the batch-1 Llama decode step, its model object, the layer
// streaming pipeline and the measurement entry points.
//
// Step (hada "Hauptfunktionen": Llama with RoPE, GQA, SwiGLU, RMSNorm, KV cache;
// "Architektur und Codestruktur": GEMV, RMSNorm, RoPE, SwiGLU, softmax kernels):
//   x = dequant(embd[token])
//   per layer:  [RMSNorm -> Q|K|V GEMV -> RoPE -> K,V to the f16 cache]   one GEMV launch
//               split-context GQA attention + combine                      two launches
//               [O GEMV + residual]                                        one GEMV launch
//               [RMSNorm -> gate|up GEMV -> SwiGLU]                        one GEMV launch
//               [down GEMV + residual]                                     one GEMV launch
//   [RMSNorm -> output GEMV -> per-CTA top-2] -> argmax                   two launches
// Resident models replay the step as one CUDA graph with programmatic
// dependent launch between consecutive GEMVs.
//
// Streaming (hada "3-stufiges adaptives Caching", "SLEP-Streaming ... Double
// Buffering"; hotdry "gpu-nvme-direct的实现架构": two staging buffers, copy and
// compute overlapped on CUDA streams): layers >= n_resident live in page-locked
// host memory; each step copies layer l into staging buffer (l - n_resident) % 2
// on a copy stream while layer l-1 computes; the copy into a buffer waits for
// the compute that last read it.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <thread>
#include <vector>

#include "nt_attn.cuh"
#include "nt_gemv_pipe.cuh"

namespace nt {

constexpr uint32_t kUidEmbd = 0x100000u, kUidOutput = 0x100001u, kUidKv = 0x200000u;

// ---------------------------------------------------------------- kernels --

__global__ void k_embed(const QMat e, const int32_t* __restrict__ d_token, float* __restrict__ x) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= e.cols) return;
  int64_t tok = *d_token;
  if (tok < 0 || tok >= e.rows) tok = 0;   // ids come validated from the host or from k_argmax
  x[i] = dequant_elem(e, tok * e.cols + i);
}

// One CTA per (kv head, chunk).  The n = pos + 1 positions of a step are split
// into per = max(32, ceil(n / chunks of the grid)) <= C positions per item, the
// last item taking the rest, over used = ceil(n / per) items of each kv head
// (items past those have nothing to do).  Launched as a programmatic dependent of the QKV GEMV: the
// rows cached by earlier steps (and the position, written by the previous
// step's argmax) are final before that GEMV starts, so they are copied before
// waiting for it; q and the current position's K and V only after.
template <int HD, int G, int CM>
__global__ void __launch_bounds__(kAttnThreads, 1) k_attn(const __grid_constant__ AttnArgs a,
                                                          const int32_t* __restrict__ d_pos) {
  extern __shared__ uint4 smem_u4[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(smem_u4);
  const int n = __ldcg(d_pos) + 1;
  const int per = max(32, (n + int(gridDim.y) - 1) / int(gridDim.y));   // positions per item, <= C
  const int used = (n + per - 1) / per;
  // the O projection may start its weight prefetch; it waits for this grid before reading its output
  asm volatile("griddepcontrol.launch_dependents;");
  if (int(blockIdx.y) >= used) return;
  const int t0 = int(blockIdx.y) * per, cnt = min(per, n - t0);
  const int r_done = max(0, min(cnt, n - 1 - t0));          // rows of positions cached by earlier steps
  attn_copy_rows<HD, CM>(a, blockIdx.x, t0, 0, r_done, sm);
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  attn_item<HD, G, CM>(a, blockIdx.x, blockIdx.y, t0, cnt, used, sm, r_done);
}

// The same items with the items of each kv head launched as one thread-block
// cluster (cluster rank = item): the items keep their partials in shared
// memory, and after a cluster barrier the G heads are merged by warps spread
// over the cluster, reading the partials across it (no global partials, fence
// or ticket).  Every CTA takes part in both cluster barriers, items with no
// positions included; the second keeps each CTA's partials in place until the
// merges that read them are done.
template <int HD, int G, int CM>
__global__ void __launch_bounds__(kAttnThreads, 1) k_attn_cl(const __grid_constant__ AttnArgs a,
                                                             const int32_t* __restrict__ d_pos) {
  namespace cg = cooperative_groups;
  extern __shared__ uint4 smem_u4[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(smem_u4);
  cg::cluster_group cl = cg::this_cluster();
  const int items = int(cl.num_blocks()), item = int(cl.block_rank());
  const int n = __ldcg(d_pos) + 1;
  const int per = max(32, (n + items - 1) / items);   // positions per item, <= C
  const int used = (n + per - 1) / per;
  asm volatile("griddepcontrol.launch_dependents;");
  const bool live = item < used;
  int t0 = 0, cnt = 0, r_done = 0;
  if (live) {
    t0 = item * per;
    cnt = min(per, n - t0);
    r_done = max(0, min(cnt, n - 1 - t0));
    attn_copy_rows<HD, CM>(a, blockIdx.x, t0, 0, r_done, sm);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (live) attn_item<HD, G, CM, true>(a, blockIdx.x, item, t0, cnt, used, sm, r_done);
  cl.sync();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int h = item + items * warp; h < G; h += items * kAttnWarps)
    attn_merge_cluster<HD, G, CM>(a, blockIdx.x, h, used, lane, sm);
  cl.sync();
}

// Greedy choice over the per-CTA top-2 summaries of the output GEMV (ties to the
// lowest id), then the step's bookkeeping: next input token, history, position.
__global__ void k_argmax(const float4* __restrict__ top2, int n, int32_t* d_pos, int32_t* d_token,
                         int32_t* d_next, float* d_margin, int32_t* d_hist, int max_ctx, int vocab) {
  __shared__ float sb[256], ss[256];
  __shared__ int si[256];
  float b = -INFINITY, s = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const float4 v = top2[i];
    top2_merge(v.x, __float_as_int(v.y), v.z, b, bi, s);
  }
  sb[threadIdx.x] = b;
  ss[threadIdx.x] = s;
  si[threadIdx.x] = bi;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int t = 1; t < blockDim.x; t++) top2_merge(sb[t], si[t], ss[t], b, bi, s);
    if (bi < 0 || bi >= vocab) bi = 0;     // no finite logit at all: keep the id in range
    const int p = *d_pos;
    *d_next = bi;
    *d_margin = b - s;
    if (p < max_ctx) d_hist[p] = bi;
    *d_token = bi;
    *d_pos = p + 1;
  }
}

// cos[l] = <a, b> / (|a| |b|) for a = hs[l], b = hs[l + 1] (0 when either is zero):
// one CTA per layer, fp64 partial sums in a fixed order.
__global__ void __launch_bounds__(256) k_layer_cos(const float* __restrict__ hs, int n, double* __restrict__ cos) {
  const float* a = hs + size_t(blockIdx.x) * n;
  const float* b = a + n;
  double ab = 0, aa = 0, bb = 0;
  for (int i = threadIdx.x; i < n; i += 256) {
    const double u = a[i], v = b[i];
    ab = fma(u, v, ab);
    aa = fma(u, u, aa);
    bb = fma(v, v, bb);
  }
  __shared__ double red[3][8];
  for (int o = 16; o; o >>= 1) {
    ab += __shfl_xor_sync(0xffffffffu, ab, o);
    aa += __shfl_xor_sync(0xffffffffu, aa, o);
    bb += __shfl_xor_sync(0xffffffffu, bb, o);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red[0][w] = ab;
    red[1][w] = aa;
    red[2][w] = bb;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double s0 = 0, s1 = 0, s2 = 0;
    for (int i = 0; i < 8; i++) {
      s0 += red[0][i];
      s1 += red[1][i];
      s2 += red[2][i];
    }
    cos[blockIdx.x] = (s1 == 0 || s2 == 0) ? 0.0 : s0 / (sqrt(s1) * sqrt(s2));
  }
}

// f16 N(0,1) prefill; counter index of (t, kv head g, d) is (t*n_kv + g)*hd + d.
__global__ void k_kv_prefill(__half* kv, int n_layers, int n_kv, int max_ctx, int hd, int n_ctx, uint64_t seed) {
  const int64_t per = int64_t(n_ctx) * n_kv * hd;
  const int64_t total = int64_t(n_layers) * 2 * per;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t lk = i / per, r = i % per;    // lk = layer*2 + kv
    const int64_t t = r / (int64_t(n_kv) * hd);
    const int g = int((r / hd) % n_kv), d = int(r % hd);
    const float z = __fmul_rn(gen_normal(seed, kUidKv + uint32_t(lk), uint64_t(r)), 1.0f);
    kv[((lk * n_kv + g) * max_ctx + t) * hd + d] = __float2half_rn(z);
  }
}

// ------------------------------------------------------------------ model --

struct Layer {
  uint8_t* dev = nullptr;    // device blob (resident layers)
  uint8_t* host = nullptr;   // page-locked host blob (streamed layers)
  size_t bytes = 0;          // padded blob bytes
  size_t off[7] = {};        // per-role offset inside the blob
  int64_t rows[7] = {}, cols[7] = {};
  int type[7] = {};
  nt_qtensor view[7];        // what nt_model_tensor hands out
};

struct Prof {
  struct Rec {
    int kind;
    double bytes;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  cudaEvent_t ev() {
    if (used == pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[used++];
  }
  ~Prof() {
    for (auto e : pool) cudaEventDestroy(e);
  }
};

}  // namespace nt

struct nt_model {
  nt_config c{};
  std::vector<nt::Layer> layers;
  nt_qtensor embd, output;
  __half* kv = nullptr;
  float *x = nullptr, *q = nullptr, *att = nullptr, *u = nullptr, *logits = nullptr;
  float* part_o = nullptr;
  float2* part_ml = nullptr;
  float2* rope = nullptr;
  float4* top2 = nullptr;
  unsigned* tickets = nullptr;       // attention: finished chunks per kv head
  int32_t* small = nullptr;          // pos, token, next, margin(float bits)
  int32_t* hist = nullptr;           // produced ids by position
  int32_t* h_io = nullptr;           // pinned host mirror of small; [32, 56): speculative step
  float* sp_x = nullptr;             // speculative step: residual of each draft token after the draft layers
  float *sp_q = nullptr, *sp_att = nullptr, *sp_u = nullptr;   // speculative step: per-token q, attention output, u
  int32_t* sp_i = nullptr;           // speculative step: positions [0, 8), full-model tokens [8, 16), draft tokens [16, 24)
  float* cur_x = nullptr;            // residual the enqueue helpers use (nullptr: x)
  int32_t* cur_pos = nullptr;        // device position the enqueue helpers use (nullptr: the step's)
  int n_chunks = 0;
  cudaStream_t stream = nullptr, copy_stream = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  // graph of a resident model's speculative cycle (draft and verification) for
  // one draft depth, k and skip mask; verification weight bytes it reads
  cudaGraphExec_t sp_exec = nullptr;
  int sp_n_draft = -1, sp_k = -1;
  std::vector<uint8_t> sp_skip;
  double sp_vwb = 0;
  int out_grid = 0;
  int32_t pos = 0;
  int n_resident = 0;
  uint8_t* staging[2] = {nullptr, nullptr};
  cudaEvent_t ev_copy_done[2] = {}, ev_compute_done[2] = {};
  std::vector<cudaEvent_t> ev_cs, ev_ce, ev_ls, ev_le;
  cudaEvent_t ev_step0 = nullptr, ev_step1 = nullptr;
  cudaEvent_t ev_io = nullptr;       // after a step's result copies to the host
  nt_stats stats{};
  std::vector<uint8_t> skip;         // per layer: 1 = skipped (empty: none)
  std::vector<uint8_t> ran;          // per layer: evaluated in the last streamed step
  float* hs = nullptr;               // similarity step: residual before each layer and after the last
  double* d_cos = nullptr;           // similarity step: per-layer cosine
  size_t dev_bytes = 0, dev_limit = 0;
  std::vector<std::pair<void*, size_t>> dev_allocs;   // live device allocations and their sizes
};

namespace nt {

static int32_t* d_pos(nt_model* m) { return m->small + 0; }
static int32_t* d_token(nt_model* m) { return m->small + 1; }
static int32_t* d_next(nt_model* m) { return m->small + 2; }
static float* d_margin(nt_model* m) { return reinterpret_cast<float*>(m->small + 3); }
// Residual vector and device position of the token being enqueued: the step's
// own, or one token of a speculative verification pass.
static float* xres(nt_model* m) { return m->cur_x ? m->cur_x : m->x; }
static int32_t* xpos(nt_model* m) { return m->cur_pos ? m->cur_pos : d_pos(m); }

static cudaError_t dev_alloc(nt_model* m, void** p, size_t bytes) {
  if (m->dev_limit && m->dev_bytes + bytes > m->dev_limit) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(p, bytes ? bytes : 1);
  if (e == cudaSuccess) {
    m->dev_bytes += bytes;
    m->dev_allocs.emplace_back(*p, bytes);
  }
  return e;
}

static void dev_free(nt_model* m, void* p) {
  if (!p) return;
  for (size_t i = 0; i < m->dev_allocs.size(); i++)
    if (m->dev_allocs[i].first == p) {
      m->dev_bytes -= m->dev_allocs[i].second;
      m->dev_allocs.erase(m->dev_allocs.begin() + long(i));
      break;
    }
  cudaFree(p);
}

static QMat view_at(const Layer& L, int role, uint8_t* base) {
  QMat q;
  q.type = L.type[role];
  q.rows = L.rows[role];
  q.cols = L.cols[role];
  layout_streams(q, base + L.off[role]);
  return q;
}

static int64_t kv_layer_elems(const nt_config& c) { return int64_t(c.n_kv_heads) * c.max_ctx * c.head_dim; }
static __half* k_cache(nt_model* m, int l) { return m->kv + (int64_t(l) * 2 + 0) * kv_layer_elems(m->c); }
static __half* v_cache(nt_model* m, int l) { return m->kv + (int64_t(l) * 2 + 1) * kv_layer_elems(m->c); }

static bool skipped(const nt_model* m, int l) { return !m->skip.empty() && m->skip[size_t(l)]; }

static double qbytes(const QMat& q) { return double(stream_sizes(q.type, q.rows, q.cols).total()); }

// Launch helper: optional event pair around each launch for nt_profile_steps.
struct Launcher {
  Prof* prof = nullptr;
  cudaStream_t s = nullptr;
  template <class F>
  cudaError_t run(int kind, double bytes, F&& f) {
    cudaEvent_t a = nullptr, b = nullptr;
    if (prof) {
      a = prof->ev();
      b = prof->ev();
      if (!a || !b) return cudaErrorMemoryAllocation;
      cudaError_t e = cudaEventRecord(a, s);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = f();
    if (e != cudaSuccess) return e;
    if (prof) {
      e = cudaEventRecord(b, s);
      if (e != cudaSuccess) return e;
      prof->recs.push_back({kind, bytes, a, b});
    }
    return cudaSuccess;
  }
};

constexpr size_t kAttnMinSmem = 116 * 1024;   // more than half of an SM's shared memory

// Whether the clusters of `items` CTAs of k_attn_cl<HD, G, CM> can all be
// resident at once for n_kv kv heads (one cluster each), from the occupancy
// query; cached per cluster size.  Sizes above 8 need the non-portable cluster
// attribute.
template <int HD, int G, int CM>
static bool attn_clusters_fit(int items, int n_kv, size_t smem) {
  static std::atomic<int> fit[17] = {};   // 0: not asked yet; else 1 + clusters resident at once
  if (items < 2 || items > 16) return false;
  int v = fit[items].load(std::memory_order_relaxed);
  if (v == 0) {
    auto kern = k_attn_cl<HD, G, CM>;
    int clusters = 0;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(unsigned(n_kv), unsigned(items));
      cfg.blockDim = dim3(kAttnThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = unsigned(items);
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    }
    if (e != cudaSuccess) {
      (void)cudaGetLastError();   // a refused query only means: no clusters
      clusters = 0;
    }
    v = 1 + clusters;
    fit[items].store(v, std::memory_order_relaxed);
  }
  return v - 1 >= n_kv;
}

template <int HD, int G, int CM>
static cudaError_t launch_attn_cm(dim3 grid, cudaStream_t s, const AttnArgs& a, const int32_t* pos, bool pdl) {
  auto kern = k_attn<HD, G, CM>;
  // one item per SM: the block scheduler would otherwise pack several small items
  // onto the first SMs the Q/K/V GEMV frees instead of spreading them
  size_t smem = AttnLayout<HD, G, CM>::kBytes;
  if (smem < kAttnMinSmem) smem = kAttnMinSmem;
  static const KernelSetup setup = kernel_setup(kern, int(smem));
  if (setup.err != cudaSuccess) return setup.err;
  const bool cluster = attn_clusters_fit<HD, G, CM>(int(grid.y), int(grid.x), smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cluster) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = grid.y;
    attr[na].val.clusterDim.z = 1;
    na++;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
  }
  cfg.attrs = attr;
  cfg.numAttrs = unsigned(na);
  return cluster ? cudaLaunchKernelEx(&cfg, k_attn_cl<HD, G, CM>, a, pos) : cudaLaunchKernelEx(&cfg, kern, a, pos);
}

template <int HD, int G>
static cudaError_t launch_attn_t(dim3 grid, cudaStream_t s, const AttnArgs& a, const int32_t* pos, bool pdl) {
  switch (attn_chunk_max(a.chunk)) {
    case 64: return launch_attn_cm<HD, G, 64>(grid, s, a, pos, pdl);
    case 128: return launch_attn_cm<HD, G, 128>(grid, s, a, pos, pdl);
    case 256: return launch_attn_cm<HD, G, 256>(grid, s, a, pos, pdl);
    case 320: return launch_attn_cm<HD, G, 320>(grid, s, a, pos, pdl);
  }
  return cudaErrorInvalidValue;
}

static cudaError_t launch_attn(int hd, int G, dim3 grid, cudaStream_t s, const AttnArgs& a, const int32_t* pos,
                               bool pdl) {
#define NT_ATTN_G(HD)                                                  \
  switch (G) {                                                         \
    case 1: return launch_attn_t<HD, 1>(grid, s, a, pos, pdl);         \
    case 2: return launch_attn_t<HD, 2>(grid, s, a, pos, pdl);         \
    case 4: return launch_attn_t<HD, 4>(grid, s, a, pos, pdl);         \
    case 8: return launch_attn_t<HD, 8>(grid, s, a, pos, pdl);         \
    case 16: return launch_attn_t<HD, 16>(grid, s, a, pos, pdl);       \
  }
  if (hd == 128) {
    NT_ATTN_G(128)
  } else {
    NT_ATTN_G(64)
  }
#undef NT_ATTN_G
  return cudaErrorInvalidValue;
}

static AttnArgs attn_args(nt_model* m, int l) {
  AttnArgs a;
  a.q = m->q;
  a.kc = k_cache(m, l);
  a.vc = v_cache(m, l);
  a.max_ctx = m->c.max_ctx;
  a.chunk = attn_chunk_len(m->c.max_ctx);
  a.scale = 1.0f / sqrtf(float(m->c.head_dim));
  a.part_o = m->part_o;
  a.part_ml = m->part_ml;
  a.n_chunks = m->n_chunks;
  a.tickets = m->tickets;
  a.out = m->att;
  return a;
}

// The GEMVs of layer l with its weights at base: QK (QKV when v shares the
// format; then v_split is false and `v` unused), V, O, gate/up, down.
struct LayerGemvs {
  GemvArgs qk, v, o, gu, down;
  bool v_split = false;
};

static LayerGemvs layer_gemvs(nt_model* m, int l, uint8_t* base) {
  const nt_config& c = m->c;
  const Layer& ly = m->layers[size_t(l)];
  const int hd = c.head_dim, qd = c.n_heads * hd, kd = c.n_kv_heads * hd;
  LayerGemvs g;
  // RMSNorm -> Q|K|V -> RoPE -> cache
  GemvArgs& a = g.qk;
  a.x = xres(m);
  a.norm = 1;
  a.eps = c.rms_eps;
  a.epi.y = m->q;
  a.epi.q_rows = qd;
  a.epi.k_rows = kd;
  a.epi.head_dim = hd;
  a.epi.pos = xpos(m);
  a.epi.rope = m->rope;
  a.epi.k_cache = k_cache(m, l);
  a.epi.v_cache = v_cache(m, l);
  a.epi.max_ctx = c.max_ctx;
  a.seg[0] = view_at(ly, NT_ROLE_Q, base);
  a.seg[1] = view_at(ly, NT_ROLE_K, base);
  if (c.t_v == c.t_q) {
    a.seg[2] = view_at(ly, NT_ROLE_V, base);
    a.nseg = 3;
  } else {
    a.nseg = 2;
    g.v = a;
    g.v.seg[0] = view_at(ly, NT_ROLE_V, base);
    g.v.nseg = 1;
    g.v.epi.row_base = qd + kd;
    g.v_split = true;
  }
  // O + residual
  g.o.seg[0] = view_at(ly, NT_ROLE_O, base);
  g.o.x = m->att;
  g.o.epi.y = xres(m);
  // RMSNorm -> gate|up (rows interleaved) -> SwiGLU
  g.gu.seg[0] = view_at(ly, NT_ROLE_GATE, base);
  g.gu.seg[1] = view_at(ly, NT_ROLE_UP, base);
  g.gu.nseg = 2;
  g.gu.interleave = 1;
  g.gu.x = xres(m);
  g.gu.norm = 1;
  g.gu.eps = c.rms_eps;
  g.gu.epi.y = m->u;
  // down + residual
  g.down.seg[0] = view_at(ly, NT_ROLE_DOWN, base);
  g.down.x = m->u;
  g.down.epi.y = xres(m);
  return g;
}

static GemvArgs head_gemv(nt_model* m) {
  GemvArgs a;
  a.seg[0] = m->output.m;
  a.x = xres(m);
  a.norm = 1;
  a.eps = m->c.rms_eps;
  a.epi.y = m->logits;
  a.epi.top2 = m->top2;
  return a;
}

static double gemv_bytes(const GemvArgs& a, double out_bytes) {
  double b = 0;
  for (int i = 0; i < a.nseg; i++) b += qbytes(a.seg[i]);
  return b + 4.0 * double(a.seg[0].cols) + out_bytes;
}

static cudaError_t enqueue_layer(nt_model* m, int l, uint8_t* base, Launcher& L, bool pdl) {
  const nt_config& c = m->c;
  const int hd = c.head_dim, G = c.n_heads / c.n_kv_heads;
  const int qd = c.n_heads * hd, kd = c.n_kv_heads * hd;
  cudaStream_t s = L.s;
  cudaError_t e;
  const LayerGemvs g = layer_gemvs(m, l, base);

  if (!g.v_split) {
    const double by = gemv_bytes(g.qk, 4.0 * qd + 4.0 * kd);
    if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv(g.qk, EPI_QKV, s, pdl, nullptr); }))) return e;
  } else {   // v in its own format: one launch for both where a kernel exists for the pair
    const double by = gemv_bytes(g.qk, 4.0 * qd + 2.0 * kd) + gemv_bytes(g.v, 2.0 * kd) - 4.0 * c.hidden;
    if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv_pair(g.qk, g.v, EPI_QKV, s, pdl, nullptr); }))) return e;
  }

  // split-context GQA attention over positions 0..pos, merged by the last chunk's CTA
  {
    const int n_used = m->pos + 1;   // host mirror (exact for profiled and streamed steps)
    const double by = 2.0 * 2.0 * double(c.n_kv_heads) * n_used * hd + 8.0 * qd;
    dim3 grid(unsigned(c.n_kv_heads), unsigned(m->n_chunks));
    const AttnArgs aa = attn_args(m, l);
    e = L.run(NT_KC_ATTN, by, [&] { return launch_attn(hd, G, grid, s, aa, xpos(m), pdl); });
    if (e) return e;
  }

  double by = gemv_bytes(g.o, 8.0 * c.hidden);
  if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv(g.o, EPI_ADD, s, pdl, nullptr); }))) return e;
  by = gemv_bytes(g.gu, 4.0 * c.ffn_dim);
  if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv(g.gu, EPI_SWIGLU, s, pdl, nullptr); }))) return e;
  by = gemv_bytes(g.down, 8.0 * c.hidden);
  if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv(g.down, EPI_ADD, s, pdl, nullptr); }))) return e;
  return cudaSuccess;
}

// Output GEMV and greedy choice; next_out (device) receives the token instead
// of the step's next-token word when given.
static cudaError_t enqueue_head(nt_model* m, Launcher& L, bool pdl, int32_t* next_out = nullptr) {
  const nt_config& c = m->c;
  cudaStream_t s = L.s;
  const GemvArgs a = head_gemv(m);
  const double by = gemv_bytes(a, 4.0 * c.vocab);
  cudaError_t e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv(a, EPI_LOGITS, s, pdl, &m->out_grid); });
  if (e) return e;
  return L.run(NT_KC_OTHER, 0.0, [&] {
    k_argmax<<<1, 256, 0, s>>>(m->top2, m->out_grid, xpos(m), d_token(m), next_out ? next_out : d_next(m),
                               d_margin(m), m->hist, c.max_ctx, c.vocab);
    return cudaGetLastError();
  });
}

static cudaError_t enqueue_embed(nt_model* m, Launcher& L) {
  return L.run(NT_KC_OTHER, 0.0, [&] {
    k_embed<<<unsigned((m->c.hidden + 255) / 256), 256, 0, L.s>>>(m->embd.m, d_token(m), m->x);
    return cudaGetLastError();
  });
}

// Whole step for a model whose layers are all resident.
static cudaError_t enqueue_resident(nt_model* m, Launcher& L, bool pdl) {
  cudaError_t e = enqueue_embed(m, L);
  for (int l = 0; l < m->c.n_layers && !e; l++)
    if (!skipped(m, l)) e = enqueue_layer(m, l, m->layers[size_t(l)].dev, L, pdl);
  if (!e) e = enqueue_head(m, L, pdl);
  return e;
}

// Copy of layer l's host blob into staging buffer b on the copy stream, once the
// buffer's last reader (ev_compute_done[b]) is done; records ev_copy_done[b]
// (and the layer's copy start/end events when `timed`).  One copy per layer:
// splitting it over several copy streams was measured slower on GB300's
// host link (168 GB/s with one stream, 148 with two, 115 with four).
static cudaError_t issue_layer_copy(nt_model* m, int l, int b, bool timed) {
  const Layer& ly = m->layers[size_t(l)];
  cudaStream_t cs = m->copy_stream;
  cudaError_t e = cudaStreamWaitEvent(cs, m->ev_compute_done[b], 0);
  if (!e && timed) e = cudaEventRecord(m->ev_cs[size_t(l)], cs);
  if (!e) e = cudaMemcpyAsync(m->staging[b], ly.host, ly.bytes, cudaMemcpyHostToDevice, cs);
  if (!e && timed) e = cudaEventRecord(m->ev_ce[size_t(l)], cs);
  if (!e) e = cudaEventRecord(m->ev_copy_done[b], cs);
  return e;
}

// Whole step with layers [n_resident, n_layers) copied through the staging
// buffers (with none streamed it is the resident step without PDL).  Skipped
// layers are neither copied nor run; the staging buffers alternate over the
// streamed layers that do run.  With hs set (similarity step) every layer runs
// and the residual is copied to hs[l] before layer l and to hs[n_layers] after
// the last.
static cudaError_t enqueue_streamed(nt_model* m, Launcher& L, float* hs, float* x_out = nullptr) {
  const int nl = m->c.n_layers, nr = m->n_resident;
  const size_t xbytes = size_t(m->c.hidden) * 4;
  cudaStream_t s = L.s;
  cudaError_t e;
  m->ran.assign(size_t(nl), 0);
  for (int l = 0; l < nl; l++) m->ran[size_t(l)] = (hs || !skipped(m, l)) ? 1 : 0;
  std::vector<int> sl;   // streamed layers that run, in order; sl[k] uses buffer k % 2
  for (int l = nr; l < nl; l++)
    if (m->ran[size_t(l)]) sl.push_back(l);
  auto issue_copy = [&](size_t k) -> cudaError_t { return issue_layer_copy(m, sl[k], int(k & 1), true); };
  for (size_t k = 0; k < sl.size() && k < 2; k++)
    if ((e = issue_copy(k))) return e;
  // programmatic dependent launch when only resident layers run and no copy or
  // event sits between the launches (a speculative draft); per-layer events otherwise
  const bool pdl = sl.empty() && !hs;
  if ((e = enqueue_embed(m, L))) return e;
  size_t k = 0;
  for (int l = 0; l < nl; l++) {
    if (!m->ran[size_t(l)]) continue;
    const bool streamed = l >= nr;
    const int b = int(k & 1);
    uint8_t* base = streamed ? m->staging[b] : m->layers[size_t(l)].dev;
    if (hs && (e = cudaMemcpyAsync(hs + size_t(l) * m->c.hidden, m->x, xbytes, cudaMemcpyDeviceToDevice, s)))
      return e;
    if (streamed && (e = cudaStreamWaitEvent(s, m->ev_copy_done[b], 0))) return e;
    if (!pdl && (e = cudaEventRecord(m->ev_ls[size_t(l)], s))) return e;
    if ((e = enqueue_layer(m, l, base, L, pdl))) return e;
    if (!pdl && (e = cudaEventRecord(m->ev_le[size_t(l)], s))) return e;
    if (streamed) {
      if ((e = cudaEventRecord(m->ev_compute_done[b], s))) return e;
      if (k + 2 < sl.size() && (e = issue_copy(k + 2))) return e;
      k++;
    }
  }
  if (x_out && (e = cudaMemcpyAsync(x_out, m->x, xbytes, cudaMemcpyDeviceToDevice, s))) return e;
  if (hs) {
    if ((e = cudaMemcpyAsync(hs + size_t(nl) * m->c.hidden, m->x, xbytes, cudaMemcpyDeviceToDevice, s))) return e;
    if (nl > 0) {
      k_layer_cos<<<unsigned(nl), 256, 0, s>>>(hs, m->c.hidden, m->d_cos);
      if ((e = cudaGetLastError())) return e;
    }
  }
  return enqueue_head(m, L, pdl);
}

static double watchdog_ms() {
  const char* v = getenv("NT_WATCHDOG_MS");
  return v ? atof(v) : 120000.0;
}

// Waits for an event with a host-side time limit (NT_E_TIMEOUT when it expires).
static nt_status wait_event(cudaEvent_t ev, const char* what) {
  const auto t0 = std::chrono::steady_clock::now();
  const double limit = watchdog_ms();
  for (;;) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return NT_OK;
    if (e != cudaErrorNotReady) return cuda_fail(e, what);
    const double ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    if (ms > limit) return fail(NT_E_TIMEOUT, std::string(what) + ": device did not finish within the watchdog limit");
    // a decode step takes milliseconds: poll without sleeping for the first 20 ms
    // (a sleep of a few microseconds returns only after the timer slack, tens of
    // microseconds, which a step would pay every token), then back off
    if (ms < 20.0) std::this_thread::yield();
    else std::this_thread::sleep_for(std::chrono::microseconds(200));
  }
}

static void drop_graph(nt_model* m) {
  if (m->exec) cudaGraphExecDestroy(m->exec);
  if (m->graph) cudaGraphDestroy(m->graph);
  m->exec = nullptr;
  m->graph = nullptr;
  if (m->sp_exec) cudaGraphExecDestroy(m->sp_exec);
  m->sp_exec = nullptr;
  m->sp_n_draft = m->sp_k = -1;
}

static nt_status ensure_graph(nt_model* m) {
  if (m->exec) return NT_OK;
  Launcher L;
  L.s = m->stream;
  NT_CUDA(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal));
  cudaError_t e = enqueue_resident(m, L, true);
  cudaGraph_t g = nullptr;
  cudaError_t e2 = cudaStreamEndCapture(m->stream, &g);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return cuda_fail(e, "decode step capture");
  }
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaStreamEndCapture");
  m->graph = g;
  e = cudaGraphInstantiate(&m->exec, g, 0);
  if (e != cudaSuccess) {
    drop_graph(m);
    return cuda_fail(e, "cudaGraphInstantiate");
  }
  return NT_OK;
}

static void free_model(nt_model* m) {
  if (!m) return;
  if (m->stream) cudaStreamSynchronize(m->stream);
  if (m->copy_stream) cudaStreamSynchronize(m->copy_stream);
  drop_graph(m);
  for (auto& L : m->layers)
    if (L.host) cudaFreeHost(L.host);
  for (auto& a : m->dev_allocs) cudaFree(a.first);
  m->dev_allocs.clear();
  if (m->h_io) cudaFreeHost(m->h_io);
  for (int b = 0; b < 2; b++) {
    if (m->ev_copy_done[b]) cudaEventDestroy(m->ev_copy_done[b]);
    if (m->ev_compute_done[b]) cudaEventDestroy(m->ev_compute_done[b]);
  }
  for (auto* v : {&m->ev_cs, &m->ev_ce, &m->ev_ls, &m->ev_le})
    for (auto e : *v) cudaEventDestroy(e);
  if (m->ev_step0) cudaEventDestroy(m->ev_step0);
  if (m->ev_step1) cudaEventDestroy(m->ev_step1);
  if (m->ev_io) cudaEventDestroy(m->ev_io);
  if (m->stream) cudaStreamDestroy(m->stream);
  if (m->copy_stream) cudaStreamDestroy(m->copy_stream);
  delete m;
}

static nt_status validate(const nt_config* c) {
  if (c->n_layers < 0 || c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->ffn_dim <= 0 || c->vocab <= 0 || c->max_ctx <= 0)
    return fail(NT_E_INVAL, "nt_model_create: sizes must be positive");
  if (c->n_heads % c->n_kv_heads) return fail(NT_E_INVAL, "nt_model_create: n_heads must be a multiple of n_kv_heads");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(NT_E_UNSUPPORTED, "nt_model_create: head_dim must be 64 or 128");
  {
    const int G = c->n_heads / c->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
      return fail(NT_E_UNSUPPORTED, "nt_model_create: query heads per kv head must be 1, 2, 4, 8 or 16");
  }
  const nt_qtype ts[9] = {c->t_embd, c->t_q, c->t_k, c->t_v, c->t_o, c->t_gate, c->t_up, c->t_down, c->t_out};
  for (nt_qtype t : ts) {
    if (t == NT_F32 || t == NT_F16) return fail(NT_E_UNSUPPORTED, "nt_model_create: F32/F16 weights are not implemented");
    if (!supported_weight_type(t)) return fail(NT_E_INVAL, "nt_model_create: unknown weight type");
  }
  if (c->t_q != c->t_k) return fail(NT_E_UNSUPPORTED, "nt_model_create: q and k must share a format");
  if (c->t_gate != c->t_up) return fail(NT_E_UNSUPPORTED, "nt_model_create: gate and up must share a format");
  const int64_t h = c->hidden, qd = int64_t(c->n_heads) * c->head_dim, f = c->ffn_dim;
  auto ok = [](nt_qtype t, int64_t cols) { return cols % block_elems(t) == 0 && cols <= 32768 && cols % 32 == 0; };
  if (!ok(c->t_embd, h) || !ok(c->t_out, h) || !ok(c->t_q, h) || !ok(c->t_v, h) || !ok(c->t_gate, h) ||
      !ok(c->t_o, qd) || !ok(c->t_down, f))
    return fail(NT_E_INVAL, "nt_model_create: a column count is not a multiple of its format's block (or > 32768)");
  if (int64_t(c->vocab) * h >= (int64_t(1) << 40)) return fail(NT_E_INVAL, "nt_model_create: vocab too large");
  if (c->n_layers * 16 + 16 >= 0x100000) return fail(NT_E_INVAL, "nt_model_create: too many layers");
  return NT_OK;
}

}  // namespace nt

using namespace nt;

// Workspace of the isolated attention entry: kv-head tickets, the position the
// kernel reads, then the chunk statistics and partial outputs, each 16-byte
// aligned.
struct AttnWorkspace {
  int chunk = 0, n_chunks = 0;
  size_t off_tickets = 0, off_pos = 0, off_ml = 0, off_o = 0, bytes = 0;
};

static nt_status attn_workspace(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx,
                                AttnWorkspace* w) {
  if (n_heads <= 0 || n_kv_heads <= 0 || max_ctx <= 0) return fail(NT_E_INVAL, "nt_attention: sizes must be positive");
  if (n_heads % n_kv_heads) return fail(NT_E_INVAL, "nt_attention: n_heads must be a multiple of n_kv_heads");
  if (head_dim != 64 && head_dim != 128) return fail(NT_E_UNSUPPORTED, "nt_attention: head_dim must be 64 or 128");
  const int G = n_heads / n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(NT_E_UNSUPPORTED, "nt_attention: query heads per kv head must be 1, 2, 4, 8 or 16");
  if (n_kv_heads > 65535) return fail(NT_E_INVAL, "nt_attention: more than 65535 kv heads");
  w->chunk = attn_chunk_len(max_ctx);
  w->n_chunks = (max_ctx + w->chunk - 1) / w->chunk;
  if (w->n_chunks > 65535) return fail(NT_E_INVAL, "nt_attention: max_ctx needs more than 65535 items per kv head");
  auto up = [](size_t b) { return (b + 15) & ~size_t(15); };
  w->off_tickets = 0;
  w->off_pos = up(size_t(n_kv_heads) * 4);
  w->off_ml = w->off_pos + 16;
  w->off_o = w->off_ml + up(size_t(n_heads) * size_t(w->n_chunks) * 8);
  w->bytes = w->off_o + size_t(n_heads) * size_t(w->n_chunks) * size_t(head_dim) * 4;
  return NT_OK;
}

// Clears the kv-head tickets and stores the position p (= n_ctx - 1) that the
// attention kernel reads.
__global__ void k_attn_setup(unsigned* tickets, int n_kv, int32_t* d_pos, int p) {
  for (int i = threadIdx.x; i < n_kv; i += blockDim.x) tickets[i] = 0u;
  if (threadIdx.x == 0) *d_pos = p;
}

extern "C" {

nt_status nt_model_create(const nt_config* cfg, nt_model** out) {
  if (!cfg || !out) return fail(NT_E_INVAL, "nt_model_create: NULL argument");
  nt_status st = validate(cfg);
  if (st) return st;
  nt_model* m = new (std::nothrow) nt_model();
  if (!m) return fail(NT_E_NOMEM, "nt_model_create: host allocation failed");
  m->c = *cfg;
  const nt_config& c = m->c;
  if (const char* lim = getenv("NT_DEVICE_BYTES_LIMIT")) m->dev_limit = size_t(strtoull(lim, nullptr, 10));
  cudaError_t e;
#define NT_TRY(call, what)            \
  do {                                \
    e = (call);                       \
    if (e != cudaSuccess) {           \
      nt_status s_ = cuda_fail(e, what); \
      free_model(m);                  \
      return s_;                      \
    }                                 \
  } while (0)
  NT_TRY(cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking), "cudaStreamCreate");
  NT_TRY(cudaStreamCreateWithFlags(&m->copy_stream, cudaStreamNonBlocking), "cudaStreamCreate");
  for (int b = 0; b < 2; b++) {
    NT_TRY(cudaEventCreateWithFlags(&m->ev_copy_done[b], cudaEventDisableTiming), "cudaEventCreate");
    NT_TRY(cudaEventCreateWithFlags(&m->ev_compute_done[b], cudaEventDisableTiming), "cudaEventCreate");
  }
  NT_TRY(cudaEventCreate(&m->ev_step0), "cudaEventCreate");
  NT_TRY(cudaEventCreate(&m->ev_step1), "cudaEventCreate");
  NT_TRY(cudaEventCreateWithFlags(&m->ev_io, cudaEventDisableTiming), "cudaEventCreate");
  for (auto* v : {&m->ev_cs, &m->ev_ce, &m->ev_ls, &m->ev_le}) {
    v->resize(size_t(c.n_layers));
    for (auto& ev : *v) NT_TRY(cudaEventCreate(&ev), "cudaEventCreate");
  }

  const int64_t h = c.hidden, hd = c.head_dim, qd = int64_t(c.n_heads) * hd, kd = int64_t(c.n_kv_heads) * hd;
  // weights
  m->layers.resize(size_t(c.n_layers));
  const nt_qtype types[7] = {c.t_q, c.t_k, c.t_v, c.t_o, c.t_gate, c.t_up, c.t_down};
  const int64_t rows[7] = {qd, kd, kd, h, c.ffn_dim, c.ffn_dim, h};
  const int64_t colsv[7] = {h, h, h, qd, h, h, c.ffn_dim};
  for (int l = 0; l < c.n_layers; l++) {
    Layer& L = m->layers[size_t(l)];
    size_t off = 0;
    for (int r = 0; r < 7; r++) {
      L.type[r] = types[r];
      L.rows[r] = rows[r];
      L.cols[r] = colsv[r];
      L.off[r] = off;
      off += stream_sizes(types[r], rows[r], colsv[r]).padded_total();
    }
    L.bytes = off;
    NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&L.dev), L.bytes), "nt_model_create: layer allocation");
    for (int r = 0; r < 7; r++) {
      nt_qtensor& v = L.view[r];
      v.m = view_at(L, r, L.dev);
      v.nbytes = stream_sizes(types[r], rows[r], colsv[r]).total();
      NT_TRY(launch_generate(v.m, c.seed, uint32_t(l * 16 + r), c.init_std, m->stream), "generate layer");
    }
  }
  auto make_big = [&](nt_qtensor& t, nt_qtype ty, uint32_t uid) -> cudaError_t {
    t.m.type = ty;
    t.m.rows = c.vocab;
    t.m.cols = h;
    StreamSizes ss = stream_sizes(ty, c.vocab, h);
    t.nbytes = ss.total();
    cudaError_t er = dev_alloc(m, reinterpret_cast<void**>(&t.base), ss.padded_total());
    if (er) return er;
    layout_streams(t.m, t.base);
    return launch_generate(t.m, c.seed, uid, c.init_std, m->stream);
  };
  NT_TRY(make_big(m->embd, c.t_embd, kUidEmbd), "nt_model_create: token_embd");
  NT_TRY(make_big(m->output, c.t_out, kUidOutput), "nt_model_create: output");

  // cache, activations, partials
  const size_t kv_elems = size_t(c.n_layers) * 2 * size_t(kv_layer_elems(c));
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->kv), kv_elems * 2), "nt_model_create: KV cache");
  NT_TRY(cudaMemsetAsync(m->kv, 0, kv_elems * 2, m->stream), "cudaMemset");
  m->n_chunks = int((c.max_ctx + attn_chunk_len(c.max_ctx) - 1) / attn_chunk_len(c.max_ctx));
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->x), size_t(h) * 4), "alloc x");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->q), size_t(qd) * 4), "alloc q");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->att), size_t(qd) * 4), "alloc att");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->u), size_t(c.ffn_dim) * 4), "alloc u");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->logits), size_t(c.vocab) * 4), "alloc logits");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->part_o), size_t(qd) * m->n_chunks * 4), "alloc partials");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->part_ml), size_t(c.n_heads) * m->n_chunks * 8), "alloc partials");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->top2), size_t(kMaxGemvGrid) * 16), "alloc top2");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->tickets), size_t(c.n_kv_heads) * 4), "alloc tickets");
  NT_TRY(cudaMemsetAsync(m->tickets, 0, size_t(c.n_kv_heads) * 4, m->stream), "cudaMemset");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->small), 16 * 4), "alloc small");
  NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->hist), size_t(c.max_ctx) * 4), "alloc hist");
  NT_TRY(cudaMemsetAsync(m->small, 0, 16 * 4, m->stream), "cudaMemset");
  NT_TRY(cudaMemsetAsync(m->hist, 0xff, size_t(c.max_ctx) * 4, m->stream), "cudaMemset");
  NT_TRY(cudaHostAlloc(reinterpret_cast<void**>(&m->h_io), 64 * 4, cudaHostAllocDefault), "cudaHostAlloc");
  // RoPE table in double: angle p * theta^(-2i/head_dim)
  {
    NT_TRY(dev_alloc(m, reinterpret_cast<void**>(&m->rope), size_t(c.max_ctx) * (hd / 2) * 8), "alloc rope");
    std::vector<float2> tab(size_t(c.max_ctx) * size_t(hd / 2));
    for (int p = 0; p < c.max_ctx; p++)
      for (int i = 0; i < hd / 2; i++) {
        const double ang = double(p) * std::pow(double(c.rope_theta), -2.0 * i / double(hd));
        tab[size_t(p) * (hd / 2) + i] = make_float2(float(std::cos(ang)), float(std::sin(ang)));
      }
    NT_TRY(cudaMemcpyAsync(m->rope, tab.data(), tab.size() * 8, cudaMemcpyHostToDevice, m->stream), "rope upload");
    NT_TRY(cudaStreamSynchronize(m->stream), "nt_model_create");
  }
  m->n_resident = c.n_layers;
  m->stats.n_resident = c.n_layers;
#undef NT_TRY
  *out = m;
  return NT_OK;
}

void nt_model_destroy(nt_model* m) { free_model(m); }

static nt_status set_pos(nt_model* m, int32_t p) {
  m->h_io[0] = p;
  NT_CUDA(cudaMemcpyAsync(d_pos(m), m->h_io, 4, cudaMemcpyHostToDevice, m->stream));
  NT_CUDA(cudaStreamSynchronize(m->stream));
  m->pos = p;
  return NT_OK;
}

nt_status nt_kv_reset(nt_model* m) {
  if (!m) return fail(NT_E_INVAL, "nt_kv_reset: model is NULL");
  m->stats.steps = 0;
  return set_pos(m, 0);
}

nt_status nt_kv_prefill(nt_model* m, int32_t n_ctx, uint64_t seed) {
  if (!m) return fail(NT_E_INVAL, "nt_kv_prefill: model is NULL");
  if (n_ctx < 0 || n_ctx > m->c.max_ctx) return fail(NT_E_INVAL, "nt_kv_prefill: n_ctx outside [0, max_ctx]");
  if (n_ctx > 0 && m->c.n_layers > 0) {
    const nt_config& c = m->c;
    k_kv_prefill<<<152 * 16, 256, 0, m->stream>>>(m->kv, c.n_layers, c.n_kv_heads, c.max_ctx, c.head_dim, n_ctx, seed);
    NT_CUDA(cudaGetLastError());
  }
  return set_pos(m, n_ctx);
}

// One synchronous decode step.  cos_out (similarity step): every layer runs on
// the launch-by-launch path and the per-layer cosines are copied out.
static nt_status run_step(nt_model* m, int32_t token, int32_t* next_token, float* logits_host, float* top2_margin,
                          double* cos_out, const char* who) {
  if (!m || !next_token) return fail(NT_E_INVAL, std::string(who) + ": NULL argument");
  if (token < 0 || token >= m->c.vocab) return fail(NT_E_INVAL, std::string(who) + ": token outside [0, vocab)");
  if (m->pos >= m->c.max_ctx) return fail(NT_E_INVAL, std::string(who) + ": position reached max_ctx");
  const nt_config& c = m->c;
  const bool streamed = m->n_resident < c.n_layers;
  const bool calib = cos_out != nullptr;
  if (calib && !m->hs) {
    NT_CUDA(dev_alloc(m, reinterpret_cast<void**>(&m->hs), size_t(c.n_layers + 1) * c.hidden * 4));
    NT_CUDA(dev_alloc(m, reinterpret_cast<void**>(&m->d_cos), size_t(c.n_layers > 0 ? c.n_layers : 1) * 8));
  }
  if (!calib && !streamed) {
    nt_status st = ensure_graph(m);
    if (st) return st;
  }
  m->h_io[1] = token;
  NT_CUDA(cudaMemcpyAsync(d_token(m), m->h_io + 1, 4, cudaMemcpyHostToDevice, m->stream));
  NT_CUDA(cudaEventRecord(m->ev_step0, m->stream));
  if (streamed || calib) {
    Launcher L;
    L.s = m->stream;
    cudaError_t e = enqueue_streamed(m, L, calib ? m->hs : nullptr);
    if (e) return cuda_fail(e, (std::string(who) + ": launch-by-launch step").c_str());
  } else {
    NT_CUDA(cudaGraphLaunch(m->exec, m->stream));
  }
  NT_CUDA(cudaEventRecord(m->ev_step1, m->stream));
  // next id and margin
  NT_CUDA(cudaMemcpyAsync(m->h_io + 2, d_next(m), 8, cudaMemcpyDeviceToHost, m->stream));
  if (logits_host)
    NT_CUDA(cudaMemcpyAsync(logits_host, m->logits, size_t(c.vocab) * 4, cudaMemcpyDeviceToHost, m->stream));
  if (calib && c.n_layers > 0)
    NT_CUDA(cudaMemcpyAsync(cos_out, m->d_cos, size_t(c.n_layers) * 8, cudaMemcpyDeviceToHost, m->stream));
  NT_CUDA(cudaEventRecord(m->ev_io, m->stream));   // the step and its result copies
  nt_status st = wait_event(m->ev_io, who);
  if (st) return st;
  float ms = 0.f;
  NT_CUDA(cudaEventElapsedTime(&ms, m->ev_step0, m->ev_step1));
  m->stats.last_step_ms = ms;
  m->stats.steps++;
  m->stats.h2d_layer_min_GBs = m->stats.h2d_layer_max_GBs = 0;
  m->stats.h2d_layer_min_idx = -1;
  if (streamed || calib) {
    double h2d = 0, cms = 0, bytes = 0;
    for (int l = 0; l < c.n_layers; l++) {
      if (!m->ran[size_t(l)]) continue;
      float t = 0.f;
      NT_CUDA(cudaEventElapsedTime(&t, m->ev_ls[size_t(l)], m->ev_le[size_t(l)]));
      cms += t;
      if (l >= m->n_resident) {
        NT_CUDA(cudaEventElapsedTime(&t, m->ev_cs[size_t(l)], m->ev_ce[size_t(l)]));
        h2d += t;
        bytes += double(m->layers[size_t(l)].bytes);
        if (t > 0.f) {
          const double r = double(m->layers[size_t(l)].bytes) / (double(t) * 1e6);
          if (m->stats.h2d_layer_min_idx < 0 || r < m->stats.h2d_layer_min_GBs) {
            m->stats.h2d_layer_min_GBs = r;
            m->stats.h2d_layer_min_idx = l;
          }
          if (r > m->stats.h2d_layer_max_GBs) m->stats.h2d_layer_max_GBs = r;
        }
      }
    }
    m->stats.h2d_ms = h2d;
    m->stats.h2d_bytes = bytes;
    m->stats.compute_ms = cms;
    const double mn = h2d < cms ? h2d : cms;
    double ov = mn > 0 ? (h2d + cms - ms) / mn : 0.0;
    m->stats.overlap = ov < 0 ? 0 : (ov > 1 ? 1 : ov);
  } else {
    m->stats.h2d_ms = m->stats.h2d_bytes = m->stats.overlap = 0;
    m->stats.compute_ms = ms;
  }
  m->pos++;
  *next_token = m->h_io[2];
  if (top2_margin) memcpy(top2_margin, m->h_io + 3, 4);
  return NT_OK;
}

nt_status nt_decode_step(nt_model* m, int32_t token, int32_t* next_token, float* logits_host, float* top2_margin) {
  return run_step(m, token, next_token, logits_host, top2_margin, nullptr, "nt_decode_step");
}

nt_status nt_layer_similarity(nt_model* m, int32_t token, int32_t* next_token, double* cos_out) {
  if (!cos_out) return fail(NT_E_INVAL, "nt_layer_similarity: NULL argument");
  return run_step(m, token, next_token, nullptr, nullptr, cos_out, "nt_layer_similarity");
}

nt_status nt_set_layer_skip(nt_model* m, const uint8_t* mask) {
  if (!m) return fail(NT_E_INVAL, "nt_set_layer_skip: model is NULL");
  NT_CUDA(cudaStreamSynchronize(m->stream));
  drop_graph(m);
  m->skip.clear();
  if (mask) {
    m->skip.assign(size_t(m->c.n_layers), 0);
    for (int l = 0; l < m->c.n_layers; l++) m->skip[size_t(l)] = mask[l] ? 1 : 0;
  }
  return NT_OK;
}

// The draft's tokens d_1..d_k of a speculative cycle from the token history at
// positions sp_i[0] .. sp_i[0] + k - 1 into sp_i[16 .. 16 + k) (one warp; the
// position comes from device memory, so a captured cycle replays at any position).
__global__ void k_draft_tokens(const int32_t* __restrict__ hist, int32_t* sp_i, int k) {
  const int j = int(threadIdx.x);
  if (j < k) sp_i[16 + j] = hist[sp_i[0] + j];
}

// Verification pass of a speculative cycle: layers [n_draft, n_layers) that the
// skip mask keeps, layer by layer, each for the k draft tokens (token i at
// position p + i from its residual after the draft layers, enqueue_layer_batch:
// a layer's weights are read once per multi-token launch); a host-tier layer is
// copied once for all k.  Then the head for each token; token i's greedy
// choice goes to sp_i[8 + i].  Returns the bytes copied from the host tier.
// Layer l (weights at base) for the k tokens of a verification pass (pdl: its
// GEMVs with programmatic dependent launch, for resident layers): token i
// enters with residual sp_x[i] at position sp_i[i].  Each GEMV runs once for
// several tokens (launch_gemv_batch: the weights are read once per launch, with
// each token's single-token arithmetic); attention runs once per token, token i
// over positions [0, p + i], after every token's K/V row of the layer is stored.
// Bit for bit the same as k enqueue_layer calls in token order.
static cudaError_t enqueue_layer_batch(nt_model* m, int l, uint8_t* base, Launcher& L, int k, bool pdl) {
  const nt_config& c = m->c;
  const int hd = c.head_dim, G = c.n_heads / c.n_kv_heads;
  const size_t qd = size_t(c.n_heads) * hd, kd = size_t(c.n_kv_heads) * hd, h = size_t(c.hidden);
  const size_t F = size_t(c.ffn_dim);
  cudaStream_t s = L.s;
  cudaError_t e;
  const LayerGemvs g = layer_gemvs(m, l, base);
  BatchTok qkv[8], o[8], gu[8], dn[8];
  int nq = 0, no = 0, ng = 0, nd = 0;   // launches of each GEMV (each reads the GEMV's weights once)
  for (int i = 0; i < k; i++) {
    float* xi = m->sp_x + size_t(i) * h;
    qkv[i] = {xi, m->sp_q + size_t(i) * qd, m->sp_i + i};
    o[i] = {m->sp_att + size_t(i) * qd, xi, nullptr};
    gu[i] = {xi, m->sp_u + size_t(i) * F, nullptr};
    dn[i] = {m->sp_u + size_t(i) * F, xi, nullptr};
  }
  if (!g.v_split) {
    const double by = gemv_bytes(g.qk, 4.0 * qd + 4.0 * kd);
    if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv_batch(g.qk, EPI_QKV, qkv, k, 0, s, pdl, &nq); }))) return e;
  } else {
    const double by = gemv_bytes(g.qk, 4.0 * qd + 2.0 * kd) + gemv_bytes(g.v, 2.0 * kd) - 4.0 * c.hidden;
    if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv_pair_batch(g.qk, g.v, EPI_QKV, qkv, qkv, k, s, pdl, &nq); })))
      return e;
  }
  for (int i = 0; i < k; i++) {
    const int n_used = m->pos + i + 1;
    const double by = 2.0 * 2.0 * double(c.n_kv_heads) * n_used * hd + 8.0 * qd;
    dim3 grid(unsigned(c.n_kv_heads), unsigned(m->n_chunks));
    AttnArgs aa = attn_args(m, l);
    aa.q = m->sp_q + size_t(i) * qd;
    aa.out = m->sp_att + size_t(i) * qd;
    const int32_t* pos = m->sp_i + i;
    // no programmatic dependent launch here: an attention item copies the rows
    // below its position before its dependency wait, and for token i > 0 rows
    // p .. p + i - 1 come from this layer's Q/K/V launch, which the previous
    // attention launch (it lets its dependents start at once) does not wait for
    if ((e = L.run(NT_KC_ATTN, by, [&] { return launch_attn(hd, G, grid, s, aa, pos, false); }))) return e;
  }
  double by = gemv_bytes(g.o, 8.0 * c.hidden);
  if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv_batch(g.o, EPI_ADD, o, k, 0, s, pdl, &no); }))) return e;
  by = gemv_bytes(g.gu, 4.0 * c.ffn_dim);
  if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv_batch(g.gu, EPI_SWIGLU, gu, k, 0, s, pdl, &ng); }))) return e;
  by = gemv_bytes(g.down, 8.0 * c.hidden);
  if ((e = L.run(NT_KC_GEMV, by, [&] { return launch_gemv_batch(g.down, EPI_ADD, dn, k, 0, s, pdl, &nd); }))) return e;
  // weight bytes the layer's launches read
  const Layer& ly = m->layers[size_t(l)];
  double wb = 0;
  const int nl_[7] = {nq, nq, nq, no, ng, ng, nd};
  for (int r = 0; r < 7; r++) wb += double(nl_[r]) * qbytes(view_at(ly, r, base));
  m->stats.verify_weight_bytes += wb;
  return cudaSuccess;
}

static cudaError_t enqueue_verify(nt_model* m, Launcher& L, int n_draft, int k, double* h2d_bytes) {
  const int nl = m->c.n_layers, nr = m->n_resident;
  const size_t h = size_t(m->c.hidden);
  cudaStream_t s = L.s;
  cudaError_t e;
  std::vector<int> run, sl;
  for (int l = n_draft; l < nl; l++)
    if (!skipped(m, l)) {
      run.push_back(l);
      if (l >= nr) sl.push_back(l);
    }
  *h2d_bytes = 0;
  auto issue_copy = [&](size_t j) -> cudaError_t {
    *h2d_bytes += double(m->layers[size_t(sl[j])].bytes);
    return issue_layer_copy(m, sl[j], int(j & 1), false);
  };
  for (size_t j = 0; j < sl.size() && j < 2; j++)
    if ((e = issue_copy(j))) return e;
  size_t j = 0;
  for (int l : run) {
    const bool streamed = l >= nr;
    const int b = int(j & 1);
    uint8_t* base = streamed ? m->staging[b] : m->layers[size_t(l)].dev;
    if (streamed && (e = cudaStreamWaitEvent(s, m->ev_copy_done[b], 0))) return e;
    if ((e = enqueue_layer_batch(m, l, base, L, k, sl.empty()))) return e;
    if (streamed) {
      if ((e = cudaEventRecord(m->ev_compute_done[b], s))) return e;
      if (j + 2 < sl.size() && (e = issue_copy(j + 2))) return e;
      j++;
    }
  }
  for (int i = 0; i < k && !e; i++) {
    m->cur_x = m->sp_x + size_t(i) * h;
    m->cur_pos = m->sp_i + i;
    e = enqueue_head(m, L, sl.empty(), m->sp_i + 8 + i);
  }
  m->cur_x = nullptr;
  m->cur_pos = nullptr;
  return e;
}

// One speculative cycle's device work from position sp_i[0]: k draft steps over
// the layers below n_draft (and the head; each token's residual after them is
// kept for the verification), the draft's tokens, then the verification.  h2d
// receives the bytes copied from the host tier.
static cudaError_t enqueue_cycle(nt_model* m, int n_draft, int k, double* h2d) {
  const nt_config& c = m->c;
  const size_t h = size_t(c.hidden);
  *h2d = 0;
  const std::vector<uint8_t> user = m->skip;
  std::vector<uint8_t> dmask(size_t(c.n_layers), 0);
  for (int l = 0; l < c.n_layers; l++) dmask[size_t(l)] = (l >= n_draft || (!user.empty() && user[size_t(l)])) ? 1 : 0;
  m->skip = dmask;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < k && !e; i++) {
    Launcher L;
    L.s = m->stream;
    e = enqueue_streamed(m, L, nullptr, m->sp_x + size_t(i) * h);
    for (int l = 0; l < c.n_layers; l++)
      if (m->ran[size_t(l)] && l >= m->n_resident) *h2d += double(m->layers[size_t(l)].bytes);
  }
  m->skip = user;
  if (e) return e;
  k_draft_tokens<<<1, 32, 0, m->stream>>>(m->hist, m->sp_i, k);
  if ((e = cudaGetLastError())) return e;
  Launcher L;
  L.s = m->stream;
  double vb = 0;
  m->stats.verify_weight_bytes = 0;
  e = enqueue_verify(m, L, n_draft, k, &vb);
  *h2d += vb;
  return e;
}

nt_status nt_speculative_step(nt_model* m, int32_t token, int32_t n_draft, int32_t k, int32_t* out_tokens,
                              int32_t* n_out, int32_t* n_accepted) {
  if (!m || !out_tokens || !n_out) return fail(NT_E_INVAL, "nt_speculative_step: NULL argument");
  const nt_config& c = m->c;
  if (token < 0 || token >= c.vocab) return fail(NT_E_INVAL, "nt_speculative_step: token outside [0, vocab)");
  if (k < 1 || k > 8 || n_draft < 0 || n_draft > c.n_layers)
    return fail(NT_E_INVAL, "nt_speculative_step: k outside [1, 8] or n_draft outside [0, n_layers]");
  if (m->pos + k > c.max_ctx) return fail(NT_E_INVAL, "nt_speculative_step: the cycle would pass max_ctx");
  const size_t h = size_t(c.hidden);
  if (!m->sp_x) {
    const size_t qd = size_t(c.n_heads) * c.head_dim;
    NT_CUDA(dev_alloc(m, reinterpret_cast<void**>(&m->sp_x), 8 * h * 4));
    NT_CUDA(dev_alloc(m, reinterpret_cast<void**>(&m->sp_i), 32 * 4));
    NT_CUDA(dev_alloc(m, reinterpret_cast<void**>(&m->sp_q), 8 * qd * 4));
    NT_CUDA(dev_alloc(m, reinterpret_cast<void**>(&m->sp_att), 8 * qd * 4));
    NT_CUDA(dev_alloc(m, reinterpret_cast<void**>(&m->sp_u), 8 * size_t(c.ffn_dim) * 4));
  }
  NT_CUDA(cudaStreamSynchronize(m->stream));
  const int32_t p = m->pos;
  int32_t* hs = m->h_io + 32;            // positions, full-model tokens, draft tokens
  for (int i = 0; i < k; i++) hs[i] = p + i;
  m->h_io[0] = p;
  m->h_io[1] = token;
  NT_CUDA(cudaMemcpyAsync(d_pos(m), m->h_io, 8, cudaMemcpyHostToDevice, m->stream));   // pos, token
  NT_CUDA(cudaMemcpyAsync(m->sp_i, hs, 8 * 4, cudaMemcpyHostToDevice, m->stream));
  NT_CUDA(cudaEventRecord(m->ev_step0, m->stream));

  // on failure the cycle may have moved the device position: put it back
  auto resync = [&](nt_status st) {
    m->h_io[0] = m->pos;
    cudaMemcpyAsync(d_pos(m), m->h_io, 4, cudaMemcpyHostToDevice, m->stream);
    cudaStreamSynchronize(m->stream);
    return st;
  };
  double h2d = 0;
  cudaError_t e = cudaSuccess;
  if (m->n_resident >= c.n_layers) {
    // resident: the cycle's launches as one cached graph (they read positions and
    // tokens from device memory, so it replays at any position)
    if (!m->sp_exec || m->sp_n_draft != n_draft || m->sp_k != k || m->sp_skip != m->skip) {
      if (m->sp_exec) cudaGraphExecDestroy(m->sp_exec);
      m->sp_exec = nullptr;
      e = cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal);
      if (e) return resync(cuda_fail(e, "nt_speculative_step: cycle capture"));
      double h2d_c = 0;
      cudaError_t ec = enqueue_cycle(m, n_draft, k, &h2d_c);
      cudaGraph_t g = nullptr;
      const cudaError_t e2 = cudaStreamEndCapture(m->stream, &g);   // always leaves the capture
      if (!ec && !e2) ec = cudaGraphInstantiate(&m->sp_exec, g, 0);
      if (g) cudaGraphDestroy(g);
      if (ec || e2) {
        m->sp_exec = nullptr;
        return resync(cuda_fail(ec ? ec : e2, "nt_speculative_step: cycle capture"));
      }
      m->sp_n_draft = n_draft;
      m->sp_k = k;
      m->sp_skip = m->skip;
      m->sp_vwb = m->stats.verify_weight_bytes;
    }
    m->stats.verify_weight_bytes = m->sp_vwb;
    if ((e = cudaGraphLaunch(m->sp_exec, m->stream))) return resync(cuda_fail(e, "nt_speculative_step: cycle"));
  } else if ((e = enqueue_cycle(m, n_draft, k, &h2d))) {
    return resync(cuda_fail(e, "nt_speculative_step: cycle"));
  }
  NT_CUDA(cudaEventRecord(m->ev_step1, m->stream));
  NT_CUDA(cudaMemcpyAsync(hs + 8, m->sp_i + 8, 16 * 4, cudaMemcpyDeviceToHost, m->stream));
  nt_status st = wait_event(m->ev_step1, "nt_speculative_step");
  if (st) return resync(st);
  NT_CUDA(cudaStreamSynchronize(m->stream));
  const int32_t* y = hs + 8;
  const int32_t* d = hs + 16;
  int j = 0;
  while (j < k && y[j] == d[j]) j++;
  const int n = j < k ? j + 1 : k;
  for (int i = 0; i < j; i++) out_tokens[i] = d[i];
  if (j < k) out_tokens[j] = y[j];
  // the history at p..p+n-1 already holds the full model's choices; position and
  // next input move to the end of the emitted run
  m->pos = p + n;
  m->h_io[0] = m->pos;
  m->h_io[1] = out_tokens[n - 1];
  NT_CUDA(cudaMemcpyAsync(d_pos(m), m->h_io, 8, cudaMemcpyHostToDevice, m->stream));
  NT_CUDA(cudaStreamSynchronize(m->stream));
  float ms = 0.f;
  NT_CUDA(cudaEventElapsedTime(&ms, m->ev_step0, m->ev_step1));
  m->stats.last_step_ms = ms;
  m->stats.steps += n;
  m->stats.h2d_bytes = h2d;
  m->stats.h2d_ms = 0;
  m->stats.compute_ms = ms;
  m->stats.overlap = 0;
  *n_out = n;
  if (n_accepted) *n_accepted = j;
  return NT_OK;
}

nt_status nt_plan_layer_skip(const double* cos, int32_t n_layers, double threshold, int32_t max_skip,
                             uint8_t* mask_out, int32_t* n_skipped) {
  if (n_layers < 0 || (n_layers > 0 && (!cos || !mask_out)))
    return fail(NT_E_INVAL, "nt_plan_layer_skip: NULL array or negative n_layers");
  std::vector<int> cand;
  for (int l = 0; l < n_layers; l++)
    if (cos[l] >= threshold) cand.push_back(l);
  // most similar first, lower layer first among equals
  std::stable_sort(cand.begin(), cand.end(), [&](int a, int b) { return cos[a] > cos[b]; });
  if (max_skip > 0 && int(cand.size()) > max_skip) cand.resize(size_t(max_skip));
  for (int l = 0; l < n_layers; l++) mask_out[l] = 0;
  for (int l : cand) mask_out[l] = 1;
  if (n_skipped) *n_skipped = int32_t(cand.size());
  return NT_OK;
}

nt_status nt_decode_run(nt_model* m, int32_t token, int32_t n_steps, void* stream) {
  if (!m) return fail(NT_E_INVAL, "nt_decode_run: model is NULL");
  if (n_steps < 0 || token < 0 || token >= m->c.vocab) return fail(NT_E_INVAL, "nt_decode_run: bad token or n_steps");
  if (m->pos + n_steps > m->c.max_ctx) return fail(NT_E_INVAL, "nt_decode_run: would pass max_ctx");
  if (m->n_resident < m->c.n_layers) return fail(NT_E_STATE, "nt_decode_run: model has streamed layers");
  nt_status st = ensure_graph(m);
  if (st) return st;
  cudaStream_t us = static_cast<cudaStream_t>(stream);
  NT_CUDA(cudaEventRecord(m->ev_step0, us));
  NT_CUDA(cudaStreamWaitEvent(m->stream, m->ev_step0, 0));
  m->h_io[1] = token;
  NT_CUDA(cudaMemcpyAsync(d_token(m), m->h_io + 1, 4, cudaMemcpyHostToDevice, m->stream));
  for (int i = 0; i < n_steps; i++) NT_CUDA(cudaGraphLaunch(m->exec, m->stream));
  NT_CUDA(cudaEventRecord(m->ev_step1, m->stream));
  NT_CUDA(cudaStreamWaitEvent(us, m->ev_step1, 0));
  m->pos += n_steps;
  m->stats.steps += n_steps;
  return NT_OK;
}

nt_status nt_get_tokens(nt_model* m, int32_t t0, int32_t n, int32_t* host_out) {
  if (!m || !host_out) return fail(NT_E_INVAL, "nt_get_tokens: NULL argument");
  if (t0 < 0 || n < 0 || t0 + n > m->c.max_ctx) return fail(NT_E_INVAL, "nt_get_tokens: range");
  NT_CUDA(cudaStreamSynchronize(m->stream));
  NT_CUDA(cudaMemcpy(host_out, m->hist + t0, size_t(n) * 4, cudaMemcpyDeviceToHost));
  return NT_OK;
}

nt_status nt_kv_export(nt_model* m, int32_t layer, int32_t kv, int32_t kv_head, int32_t t0, int32_t n,
                       uint16_t* host_out) {
  if (!m || !host_out) return fail(NT_E_INVAL, "nt_kv_export: NULL argument");
  const nt_config& c = m->c;
  if (layer < 0 || layer >= c.n_layers || kv < 0 || kv > 1 || kv_head < 0 || kv_head >= c.n_kv_heads || t0 < 0 ||
      n < 0 || t0 + n > c.max_ctx)
    return fail(NT_E_INVAL, "nt_kv_export: index out of range");
  NT_CUDA(cudaStreamSynchronize(m->stream));
  const __half* src = (kv ? v_cache(m, layer) : k_cache(m, layer)) + (int64_t(kv_head) * c.max_ctx + t0) * c.head_dim;
  NT_CUDA(cudaMemcpy(host_out, src, size_t(n) * c.head_dim * 2, cudaMemcpyDeviceToHost));
  return NT_OK;
}

nt_status nt_stream_layers(nt_model* m, int32_t n_resident, int32_t n_staging) {
  if (!m) return fail(NT_E_INVAL, "nt_stream_layers: model is NULL");
  if (n_staging != 2) return fail(NT_E_UNSUPPORTED, "nt_stream_layers: n_staging must be 2 (double buffering)");
  if (n_resident < 0 || n_resident > m->c.n_layers) return fail(NT_E_INVAL, "nt_stream_layers: n_resident range");
  NT_CUDA(cudaStreamSynchronize(m->stream));
  NT_CUDA(cudaStreamSynchronize(m->copy_stream));
  drop_graph(m);
  size_t max_bytes = 0;
  for (int l = 0; l < m->c.n_layers; l++) {
    Layer& L = m->layers[size_t(l)];
    const bool want_dev = l < n_resident;
    if (want_dev && !L.dev) {
      cudaError_t e = dev_alloc(m, reinterpret_cast<void**>(&L.dev), L.bytes);
      if (e) return cuda_fail(e, "nt_stream_layers: device allocation");
      NT_CUDA(cudaMemcpy(L.dev, L.host, L.bytes, cudaMemcpyHostToDevice));
      cudaFreeHost(L.host);
      L.host = nullptr;
    } else if (!want_dev && !L.host) {
      cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&L.host), L.bytes, cudaHostAllocDefault);
      if (e) return cuda_fail(e, "nt_stream_layers: cudaHostAlloc (page-locked tier)");
      NT_CUDA(cudaMemcpy(L.host, L.dev, L.bytes, cudaMemcpyDeviceToHost));
      dev_free(m, L.dev);
      L.dev = nullptr;
    }
    for (int r = 0; r < 7; r++) {
      L.view[r].m = view_at(L, r, L.dev ? L.dev : L.host);
      L.view[r].on_host = L.dev ? 0 : 1;
    }
    if (!want_dev && L.bytes > max_bytes) max_bytes = L.bytes;
  }
  for (int b = 0; b < 2; b++) {
    if (m->staging[b]) {
      dev_free(m, m->staging[b]);
      m->staging[b] = nullptr;
    }
    if (max_bytes) {
      cudaError_t e = dev_alloc(m, reinterpret_cast<void**>(&m->staging[b]), max_bytes);
      if (e) return cuda_fail(e, "nt_stream_layers: staging buffer");
    }
  }
  m->n_resident = n_resident;
  m->stats.n_resident = n_resident;
  return NT_OK;
}

// Device bytes of one layer blob and of everything else a model allocates (see
// nt_model_create), both with the 256-byte stream padding.
static void model_bytes(const nt_config& c, int64_t* layer, int64_t* fixed) {
  const int64_t h = c.hidden, hd = c.head_dim, qd = int64_t(c.n_heads) * hd, kd = int64_t(c.n_kv_heads) * hd;
  const nt_qtype types[7] = {c.t_q, c.t_k, c.t_v, c.t_o, c.t_gate, c.t_up, c.t_down};
  const int64_t rows[7] = {qd, kd, kd, h, c.ffn_dim, c.ffn_dim, h};
  const int64_t colsv[7] = {h, h, h, qd, h, h, c.ffn_dim};
  int64_t lb = 0;
  for (int r = 0; r < 7; r++) lb += int64_t(stream_sizes(types[r], rows[r], colsv[r]).padded_total());
  const int chunk = attn_chunk_len(c.max_ctx);
  const int64_t n_chunks = (c.max_ctx + chunk - 1) / chunk;
  int64_t f = int64_t(stream_sizes(c.t_embd, c.vocab, h).padded_total()) +
              int64_t(stream_sizes(c.t_out, c.vocab, h).padded_total());
  f += int64_t(c.n_layers) * 2 * kd * c.max_ctx * 2;                      // K/V cache
  f += 4 * (h + 2 * qd + c.ffn_dim + c.vocab);                            // x, q, att, u, logits
  f += qd * n_chunks * 4 + int64_t(c.n_heads) * n_chunks * 8;              // attention partials
  f += int64_t(kMaxGemvGrid) * 16 + int64_t(c.n_kv_heads) * 4 + 16 * 4;
  f += int64_t(c.max_ctx) * 4 + int64_t(c.max_ctx) * (hd / 2) * 8;        // token history, RoPE table
  f += int64_t(c.n_layers) * 256 * 16;                                    // allocation rounding
  *layer = lb;
  *fixed = f;
}

nt_status nt_get_stats(const nt_model* m, nt_stats* out) {
  if (!m || !out) return fail(NT_E_INVAL, "nt_get_stats: NULL argument");
  *out = m->stats;
  out->pos = m->pos;
  if (out->h2d_layer_max_GBs <= 0) out->h2d_layer_min_idx = -1;   // no layer copied in the last step
  int64_t wb = int64_t(m->output.nbytes) + int64_t(m->embd.m.cols) * 0;
  for (const auto& L : m->layers)
    for (int r = 0; r < 7; r++) wb += int64_t(L.view[r].nbytes);
  out->weight_bytes = wb;
  out->kv_bytes_per_pos = int64_t(m->c.n_layers) * 2 * m->c.n_kv_heads * m->c.head_dim * 2;
  return NT_OK;
}

nt_status nt_profile_steps(nt_model* m, int32_t token, int32_t n_steps, nt_kernel_times* out) {
  if (!m || !out) return fail(NT_E_INVAL, "nt_profile_steps: NULL argument");
  if (token < 0 || token >= m->c.vocab || n_steps < 1) return fail(NT_E_INVAL, "nt_profile_steps: bad token or n_steps");
  if (m->pos + n_steps > m->c.max_ctx) return fail(NT_E_INVAL, "nt_profile_steps: would pass max_ctx");
  if (m->n_resident < m->c.n_layers) return fail(NT_E_STATE, "nt_profile_steps: model has streamed layers");
  nt_kernel_times t{};
  double wall = 0;
  m->h_io[1] = token;
  NT_CUDA(cudaMemcpyAsync(d_token(m), m->h_io + 1, 4, cudaMemcpyHostToDevice, m->stream));
  for (int i = 0; i < n_steps; i++) {
    Prof prof;
    Launcher L;
    L.s = m->stream;
    L.prof = &prof;
    NT_CUDA(cudaEventRecord(m->ev_step0, m->stream));
    cudaError_t e = enqueue_resident(m, L, false);
    if (e) return cuda_fail(e, "nt_profile_steps");
    NT_CUDA(cudaEventRecord(m->ev_step1, m->stream));
    nt_status st = wait_event(m->ev_step1, "nt_profile_steps");
    if (st) return st;
    float ms;
    NT_CUDA(cudaEventElapsedTime(&ms, m->ev_step0, m->ev_step1));
    wall += ms;
    for (auto& r : prof.recs) {
      NT_CUDA(cudaEventElapsedTime(&ms, r.a, r.b));
      t.kernel_launches++;
      t.launches[r.kind]++;
      t.ms[r.kind] += ms;
      t.bytes[r.kind] += r.bytes;
    }
    m->pos++;
    m->stats.steps++;
  }
  t.step_ms = wall / n_steps;
  *out = t;
  return NT_OK;
}

nt_status nt_profile_gemvs(nt_model* m, int32_t n_reps, double* ms_per_launch, double* bytes_per_launch,
                           int32_t* launches_per_step) {
  if (!m || !ms_per_launch || !bytes_per_launch || !launches_per_step)
    return fail(NT_E_INVAL, "nt_profile_gemvs: NULL argument");
  if (n_reps < 1) return fail(NT_E_INVAL, "nt_profile_gemvs: n_reps < 1");
  if (m->n_resident < m->c.n_layers) return fail(NT_E_STATE, "nt_profile_gemvs: model has streamed layers");
  if (m->pos >= m->c.max_ctx) return fail(NT_E_INVAL, "nt_profile_gemvs: position reached max_ctx");
  const nt_config& c = m->c;
  const int hd = c.head_dim, qd = c.n_heads * hd, kd = c.n_kv_heads * hd;
  cudaStream_t s = m->stream;
  double bytes = 0;
  int n = 0;
  // the step's GEMV launches, in order, programmatic dependent launches as in the step graph
  auto enqueue = [&]() -> cudaError_t {
    bytes = 0;
    n = 0;
    cudaError_t e;
    for (int l = 0; l < c.n_layers; l++) {
      const LayerGemvs g = layer_gemvs(m, l, m->layers[size_t(l)].dev);
      if (!g.v_split) {
        if ((e = launch_gemv(g.qk, EPI_QKV, s, true, nullptr))) return e;
        bytes += gemv_bytes(g.qk, 4.0 * qd + 4.0 * kd);
      } else {
        int nl = 0;
        if ((e = launch_gemv_pair(g.qk, g.v, EPI_QKV, s, true, &nl))) return e;
        bytes += gemv_bytes(g.qk, 4.0 * qd + 2.0 * kd) + gemv_bytes(g.v, 2.0 * kd) - 4.0 * c.hidden;
        n += nl - 1;
      }
      if ((e = launch_gemv(g.o, EPI_ADD, s, true, nullptr))) return e;
      if ((e = launch_gemv(g.gu, EPI_SWIGLU, s, true, nullptr))) return e;
      if ((e = launch_gemv(g.down, EPI_ADD, s, true, nullptr))) return e;
      bytes += gemv_bytes(g.o, 8.0 * c.hidden) + gemv_bytes(g.gu, 4.0 * c.ffn_dim) + gemv_bytes(g.down, 8.0 * c.hidden);
      n += 4;
    }
    const GemvArgs h = head_gemv(m);
    if ((e = launch_gemv(h, EPI_LOGITS, s, true, &m->out_grid))) return e;
    bytes += gemv_bytes(h, 4.0 * c.vocab);
    return cudaSuccess;
  };
  n = 0;
  NT_CUDA(cudaStreamSynchronize(s));
  NT_CUDA(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  cudaError_t e = enqueue();
  cudaGraph_t g = nullptr;
  cudaError_t e2 = cudaStreamEndCapture(s, &g);
  if (e || e2) {
    if (g) cudaGraphDestroy(g);
    return cuda_fail(e ? e : e2, "nt_profile_gemvs: capture");
  }
  const int launches = n + 1;
  cudaGraphExec_t ex = nullptr;
  e = cudaGraphInstantiate(&ex, g, 0);
  cudaGraphDestroy(g);
  if (e) return cuda_fail(e, "nt_profile_gemvs: instantiate");
  nt_status st = NT_OK;
  e = cudaGraphLaunch(ex, s);   // warm-up
  if (!e) e = cudaEventRecord(m->ev_step0, s);
  for (int i = 0; i < n_reps && !e; i++) e = cudaGraphLaunch(ex, s);
  if (!e) e = cudaEventRecord(m->ev_step1, s);
  if (e) st = cuda_fail(e, "nt_profile_gemvs: launch");
  if (!st) st = wait_event(m->ev_step1, "nt_profile_gemvs");
  float ms = 0.f;
  if (!st && (e = cudaEventElapsedTime(&ms, m->ev_step0, m->ev_step1))) st = cuda_fail(e, "nt_profile_gemvs");
  cudaGraphExecDestroy(ex);
  if (st) return st;
  *ms_per_launch = double(ms) / (double(n_reps) * launches);
  *bytes_per_launch = bytes / launches;
  *launches_per_step = launches;
  return NT_OK;
}

nt_status nt_plan_residency(const nt_config* cfg, int64_t budget_bytes, int32_t* n_resident, int64_t* device_bytes,
                            int64_t* layer_bytes) {
  if (!cfg || !n_resident) return fail(NT_E_INVAL, "nt_plan_residency: NULL argument");
  if (budget_bytes < 0) return fail(NT_E_INVAL, "nt_plan_residency: negative budget");
  nt_status st = validate(cfg);
  if (st) return st;
  int64_t layer = 0, fixed = 0;
  model_bytes(*cfg, &layer, &fixed);
  const int L = cfg->n_layers;
  *n_resident = 0;
  if (layer_bytes) *layer_bytes = layer;
  int n;
  if (fixed + int64_t(L) * layer <= budget_bytes) {
    n = L;   // everything resident: no staging buffers
  } else {
    const int64_t room = budget_bytes - fixed - 2 * layer;
    if (room < 0) {
      if (device_bytes) *device_bytes = fixed + 2 * layer;
      return fail(NT_E_NOMEM, "nt_plan_residency: the non-layer allocations and staging buffers exceed the budget");
    }
    n = int(room / layer);
    if (n >= L) n = L - 1;
  }
  *n_resident = n;
  if (device_bytes) *device_bytes = fixed + int64_t(n) * layer + (n < L ? 2 * layer : 0);
  return NT_OK;
}

nt_status nt_auto_residency(nt_model* m, int64_t margin_bytes, int32_t* n_resident_out) {
  if (!m) return fail(NT_E_INVAL, "nt_auto_residency: model is NULL");
  if (margin_bytes < 0) return fail(NT_E_INVAL, "nt_auto_residency: negative margin");
  NT_CUDA(cudaStreamSynchronize(m->stream));
  size_t free_b = 0, total_b = 0;
  NT_CUDA(cudaMemGetInfo(&free_b, &total_b));
  const int64_t budget = int64_t(free_b) + int64_t(m->dev_bytes) - margin_bytes;
  int32_t n = 0;
  nt_status st = nt_plan_residency(&m->c, budget > 0 ? budget : 0, &n, nullptr, nullptr);
  if (st) return st;
  if ((st = nt_stream_layers(m, n, 2))) return st;
  if (n_resident_out) *n_resident_out = n;
  return NT_OK;
}

// ---- isolated attention ----------------------------------------------------

nt_status nt_attention_workspace_bytes(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx,
                                       size_t* bytes) {
  if (!bytes) return fail(NT_E_INVAL, "nt_attention_workspace_bytes: NULL argument");
  AttnWorkspace w;
  const nt_status st = attn_workspace(n_heads, n_kv_heads, head_dim, max_ctx, &w);
  if (st) return st;
  *bytes = w.bytes;
  return NT_OK;
}

nt_status nt_attention(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx, int32_t n_ctx,
                       const float* dev_q, const void* dev_k, const void* dev_v, float* dev_out, void* dev_workspace,
                       size_t workspace_bytes, void* stream) {
  AttnWorkspace w;
  const nt_status st = attn_workspace(n_heads, n_kv_heads, head_dim, max_ctx, &w);
  if (st) return st;
  if (n_ctx < 1 || n_ctx > max_ctx) return fail(NT_E_INVAL, "nt_attention: n_ctx outside [1, max_ctx]");
  if (!dev_q || !dev_k || !dev_v || !dev_out || !dev_workspace) return fail(NT_E_INVAL, "nt_attention: NULL pointer");
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(dev_q) || !a16(dev_k) || !a16(dev_v) || !a16(dev_out) || !a16(dev_workspace))
    return fail(NT_E_INVAL, "nt_attention: pointers must be 16-byte aligned");
  if (workspace_bytes < w.bytes) return fail(NT_E_INVAL, "nt_attention: workspace too small");
  const int64_t qb = int64_t(n_heads) * head_dim * 4, cb = int64_t(n_kv_heads) * max_ctx * head_dim * 2;
  auto overlap = [](const void* a, int64_t na, const void* b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + uintptr_t(nb) && y < x + uintptr_t(na);
  };
  if (overlap(dev_out, qb, dev_q, qb) || overlap(dev_out, qb, dev_k, cb) || overlap(dev_out, qb, dev_v, cb) ||
      overlap(dev_out, qb, dev_workspace, int64_t(w.bytes)) || overlap(dev_workspace, int64_t(w.bytes), dev_q, qb) ||
      overlap(dev_workspace, int64_t(w.bytes), dev_k, cb) || overlap(dev_workspace, int64_t(w.bytes), dev_v, cb))
    return fail(NT_E_INVAL, "nt_attention: the output or the workspace overlaps another buffer");
  uint8_t* base = static_cast<uint8_t*>(dev_workspace);
  AttnArgs a;
  a.q = dev_q;
  a.kc = static_cast<const __half*>(dev_k);
  a.vc = static_cast<const __half*>(dev_v);
  a.max_ctx = max_ctx;
  a.chunk = w.chunk;
  a.scale = 1.0f / sqrtf(float(head_dim));
  a.tickets = reinterpret_cast<unsigned*>(base + w.off_tickets);
  a.part_ml = reinterpret_cast<float2*>(base + w.off_ml);
  a.part_o = reinterpret_cast<float*>(base + w.off_o);
  a.n_chunks = w.n_chunks;
  a.out = dev_out;
  int32_t* d_pos = reinterpret_cast<int32_t*>(base + w.off_pos);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  k_attn_setup<<<1, 128, 0, s>>>(a.tickets, n_kv_heads, d_pos, n_ctx - 1);
  NT_CUDA(cudaGetLastError());
  const dim3 grid(unsigned(n_kv_heads), unsigned(w.n_chunks));
  NT_CUDA(launch_attn(head_dim, n_heads / n_kv_heads, grid, s, a, d_pos, false));
  return NT_OK;
}

nt_status nt_model_tensor(const nt_model* m, int32_t layer, int32_t role, const nt_qtensor** out) {
  if (!m || !out) return fail(NT_E_INVAL, "nt_model_tensor: NULL argument");
  if (role == NT_ROLE_EMBD) { *out = &m->embd; return NT_OK; }
  if (role == NT_ROLE_OUTPUT) { *out = &m->output; return NT_OK; }
  if (layer < 0 || layer >= m->c.n_layers || role < 0 || role > 6) return fail(NT_E_INVAL, "nt_model_tensor: index");
  *out = &m->layers[size_t(layer)].view[role];
  return NT_OK;
}

}  // extern "C"
