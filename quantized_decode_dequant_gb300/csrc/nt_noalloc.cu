// nt_noalloc.cu -- y = W x with greedy selection of the largest y, without any
// allocation: the per-CTA top-2 summaries the selection needs live in a
// file-scope device array instead of caller- or library-allocated memory.
//
// Some callers cannot allocate device memory on this path: embedders whose
// whole device memory is reserved up front by their own allocator, and
// latency-critical loops where cudaMalloc/cudaFree would add their implicit
// device synchronisation.  They pass only inputs and outputs; the scratch is
// this array, which every GPU that loads the library holds until exit.
#include <mutex>

#include "nt_gemv.cuh"

namespace nt {

// Maximum number of CTAs whose summaries the array holds.  The GEMV launch is
// capped to it: launch_gemv never starts more CTAs than GemvArgs::max_grid
// (itself at most kMaxGemvGrid) on any of its paths.
constexpr int kNoAllocMaxCtas = 1024;
static_assert(kNoAllocMaxCtas <= kMaxGemvGrid, "max_grid must reach the GEMV launch unchanged");

// 1024 x 16 B = 16 KiB per device.  Shared by every call: each call's GEMV
// overwrites the first grid-size entries before the selection reads them, so
// nothing has to start at zero; calls that overlap on the GPU race on it.
static __device__ __align__(256) float4 g_noalloc_top2[kNoAllocMaxCtas];

constexpr int kNoAllocMaxDevices = 64;
static std::mutex g_noalloc_mu;
static float4* g_noalloc_addr[kNoAllocMaxDevices];   // device address of the array, per device

// The array's device address for the current device.  In host code the array's
// name is only a host-side stand-in, so it is resolved once per device with
// that device current, and kept for the life of the process: a cudaDeviceReset
// (which unloads the module) makes the kept address stale.
static nt_status noalloc_scratch(float4** out) {
  int dev = 0;
  NT_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(NT_E_UNSUPPORTED, "nt_gemv_argmax_noalloc: device id >= 64");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_top2);
    if (e != cudaSuccess) return cuda_fail(e, "nt_gemv_argmax_noalloc: cudaGetSymbolAddress");
    g_noalloc_addr[dev] = static_cast<float4*>(p);
  }
  *out = g_noalloc_addr[dev];
  return NT_OK;
}

// Largest entry over the n per-CTA summaries (ties to the lowest row; NaN
// entries are never selected), and the gap to the second largest.
__global__ void k_noalloc_select(const float4* __restrict__ top2, int n, int32_t* out_index, float* out_margin) {
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
    *out_index = bi == 0x7fffffff ? -1 : bi;
    *out_margin = b - s;
  }
}

}  // namespace nt

using namespace nt;

extern "C" nt_status nt_gemv_argmax_noalloc(const nt_qtensor* t, const float* dev_x, float* dev_y,
                                            int32_t* dev_index, float* dev_margin, void* stream) {
  if (!t || !dev_x || !dev_y || !dev_index || !dev_margin)
    return fail(NT_E_INVAL, "nt_gemv_argmax_noalloc: NULL argument");
  if (t->on_host) return fail(NT_E_STATE, "nt_gemv_argmax_noalloc: tensor lives in host memory (streamed layer)");
  if ((reinterpret_cast<uintptr_t>(dev_x) | reinterpret_cast<uintptr_t>(dev_y)) & 15)
    return fail(NT_E_INVAL, "nt_gemv_argmax_noalloc: x and y must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(dev_index) | reinterpret_cast<uintptr_t>(dev_margin)) & 3)
    return fail(NT_E_INVAL, "nt_gemv_argmax_noalloc: index and margin must be 4-byte aligned");
  if (t->m.rows > 0x7ffffffeLL) return fail(NT_E_INVAL, "nt_gemv_argmax_noalloc: more than 2^31 - 2 rows");
  if (t->m.cols > 28672) return fail(NT_E_UNSUPPORTED, "nt_gemv_argmax_noalloc: more than 28672 columns");
  const char* xb = reinterpret_cast<const char*>(dev_x);
  const char* yb = reinterpret_cast<const char*>(dev_y);
  if (xb < yb + t->m.rows * 4 && yb < xb + t->m.cols * 4)
    return fail(NT_E_INVAL, "nt_gemv_argmax_noalloc: x and y overlap");
  float4* scratch = nullptr;
  nt_status st = noalloc_scratch(&scratch);
  if (st) return st;
  GemvArgs a;
  a.max_grid = kNoAllocMaxCtas;
  a.seg[0] = t->m;
  a.nseg = 1;
  a.x = dev_x;
  a.epi.y = dev_y;
  a.epi.top2 = scratch;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int grid = 0;
  cudaError_t e = launch_gemv(a, EPI_LOGITS, s, false, &grid);
  if (e != cudaSuccess) return cuda_fail(e, "nt_gemv_argmax_noalloc: GEMV");
  k_noalloc_select<<<1, 256, 0, s>>>(scratch, grid, dev_index, dev_margin);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "nt_gemv_argmax_noalloc: selection");
  return NT_OK;
}
