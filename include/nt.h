/*
 * nt.h -- C ABI of the batch-1 quantized Llama decode step for NVIDIA GB300 (sm_103a).
 *
 * What it computes.  The decode step of the layer-streaming Llama engine that
 * the "ntransformer" pages describe (de.news.hada.io, "Überblick über
 * NTransformer" and "Hauptfunktionen": GGUF-style Q4_0 / Q8_0 / Q4_K / Q6_K
 * weights; Llama with RoPE, GQA, SwiGLU, RMSNorm and a KV cache; section
 * "Architektur und Codestruktur": GEMV, RMSNorm, RoPE, SwiGLU and softmax
 * kernels; "3-stufiges adaptives Caching" and "SLEP-Streaming": VRAM-resident
 * layers plus pinned-RAM layers copied host-to-device with double buffering;
 * blog.hotdry.top, "gpu-nvme-direct的实现架构": two staging buffers whose copy
 * and compute overlap on CUDA streams).  The pages plan but never show a
 * public C API ("Phase 5 ... öffentliche C-API (geplant)"), so the entry
 * points below are this library's own.
 *
 * Conventions for every function:
 *  - Returns nt_status; NT_OK on success.  On failure the output parameters
 *    are left untouched and nt_last_error() returns a message (thread-local).
 *    No C++ exception crosses this boundary.
 *  - "dev" pointers are CUDA device pointers owned by the caller; "host"
 *    pointers are ordinary host memory owned by the caller.  Objects created
 *    by *_create are owned by the library until the matching *_destroy.
 *  - "stream" is a cudaStream_t passed as void*; NULL means the legacy
 *    default stream.  Functions that take a stream are asynchronous on it;
 *    the others synchronise before they return.
 *  - One model is used by one host thread at a time.
 */
#ifndef NT_H
#define NT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NT_OK = 0,
  NT_E_INVAL = 1,        /* invalid argument: shape, token, position, pointer, size */
  NT_E_NOMEM = 2,        /* device or pinned-host allocation failed                 */
  NT_E_CUDA = 3,         /* a CUDA runtime call failed (message has the CUDA error)  */
  NT_E_TIMEOUT = 4,      /* the host watchdog gave up waiting for the device         */
  NT_E_UNSUPPORTED = 5,  /* valid request this build does not implement              */
  NT_E_STATE = 6         /* call not valid in the object's current state             */
} nt_status;

/* Weight formats ("Quantisierungsformate Q4_0, Q8_0, Q4_K_M, Q5_K, Q6_K, F16
 * und F32", hada "Überblick").  F16 and F32 weights are not implemented
 * (NT_E_UNSUPPORTED); F16 is used only for the KV cache.
 * Canonical block bytes (little-endian), the export format:
 *   Q8_0  32 weights, 34 B:  f16 d | int8 q[32]                  w = d*q
 *   Q4_0  32 weights, 18 B:  f16 d | u8 qs[16]                   w = d*(q-8)
 *         (element k in byte k/2, low nibble for even k)
 *   Q4_K  256 weights, 144 B: f16 d | f16 dmin | 12 B of sixteen 6-bit fields
 *         (sc_0..7 then m_0..7, least-significant bit first) | u8 qs[128]
 *                                                               w = d*sc_j*q - dmin*m_j
 *   Q6_K  256 weights, 210 B: u8 ql[128] (low 4 bits, as Q4_0) | u8 qh[64]
 *         (high 2 bits of element k in byte k/4 at bits 2*(k%4)) | int8 sc[16] | f16 d
 *                                                               w = d*sc_j*(q-32)
 *   Q5_K  256 weights, 176 B: f16 d | f16 dmin | 12 B of 6-bit fields as Q4_K |
 *         u8 qh[32] (fifth bit of element k in byte k/8 at bit k%8) | u8 qs[128]
 *         (low 4 bits, as Q4_0), q in 0..31              w = d*sc_j*q - dmin*m_j
 * On the device each tensor is held as separate 16-byte-aligned streams
 * (codes, scales) with the same byte count. */
typedef enum { NT_F32 = 0, NT_F16 = 1, NT_Q8_0 = 2, NT_Q4_0 = 3, NT_Q4_K = 4, NT_Q6_K = 5, NT_Q5_K = 6 } nt_qtype;

/* Tensor roles inside a layer, and the two model-level matrices. */
enum {
  NT_ROLE_Q = 0, NT_ROLE_K = 1, NT_ROLE_V = 2, NT_ROLE_O = 3,
  NT_ROLE_GATE = 4, NT_ROLE_UP = 5, NT_ROLE_DOWN = 6,
  NT_ROLE_EMBD = 16,    /* [vocab x hidden], layer argument ignored */
  NT_ROLE_OUTPUT = 17   /* [vocab x hidden], layer argument ignored */
};

typedef struct nt_model nt_model;
typedef struct nt_qtensor nt_qtensor;

/* Model description.  Llama architecture with untied embeddings and unit norm
 * gains.  Weights are drawn from N(0, init_std^2) by the counter-based
 * generator keyed by (seed, tensor uid, element index) and quantized on the
 * device into the per-role formats. */
typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, max_ctx;
  float rms_eps;      /* RMSNorm epsilon, e.g. 1e-5                  */
  float rope_theta;   /* RoPE base, e.g. 500000                      */
  float init_std;     /* weight standard deviation, e.g. 0.02        */
  nt_qtype t_embd, t_q, t_k, t_v, t_o, t_gate, t_up, t_down, t_out;
  uint64_t seed;
} nt_config;

/* Counters of the last steps (nt_get_stats). */
typedef struct {
  int64_t steps;           /* decode steps since create or reset                     */
  int32_t pos;             /* current position (number of cached tokens)            */
  int32_t n_resident;      /* layers resident in device memory                      */
  double last_step_ms;     /* wall time of the last nt_decode_step, device events    */
  double h2d_bytes;        /* bytes copied host-to-device in the last step          */
  double h2d_ms;           /* summed duration of those copies (copy-stream events)  */
  double compute_ms;       /* summed duration of the layer computations             */
  double overlap;          /* (h2d_ms + compute_ms - last_step_ms) / min(...), in [0,1] */
  int64_t weight_bytes;    /* quantized weight bytes read per step                  */
  int64_t kv_bytes_per_pos;/* KV cache bytes read per cached position per step      */
  double verify_weight_bytes; /* layer weight bytes the verification pass of the last
                              nt_speculative_step read (each multi-token launch reads
                              its weights once)                                      */
  double h2d_layer_min_GBs;   /* slowest and fastest single layer copy of the last   */
  double h2d_layer_max_GBs;   /* step, GB/s (0 when no layer was copied)             */
  int32_t h2d_layer_min_idx;  /* the layer whose copy was slowest (-1: none)         */
} nt_stats;

/* Per-kernel-class device times of profiled steps (nt_profile_steps). */
enum { NT_KC_GEMV = 0, NT_KC_ATTN = 1, NT_KC_OTHER = 2, NT_KC_COUNT = 3 };
typedef struct {
  int64_t launches[NT_KC_COUNT];
  double ms[NT_KC_COUNT];          /* summed event-to-event time of the launches */
  double bytes[NT_KC_COUNT];       /* summed algorithmic bytes of the launches   */
  double step_ms;                  /* mean wall time of a profiled step          */
  int64_t kernel_launches;         /* kernels launched over the profiled steps   */
} nt_kernel_times;

/* Message of the last failure on this thread ("" if none).  Never NULL. */
const char* nt_last_error(void);

/* ------------------------------------------------------------------ model -- */

/* Allocates device memory for all weights, the f16 KV cache ([layer][K|V]
 * [kv_head][max_ctx][head_dim]) and the activations, then generates and
 * quantizes every weight on the device.  Position starts at 0.
 * NT_E_INVAL: non-positive sizes, n_heads not a multiple of n_kv_heads,
 * head_dim odd, a column count not a multiple of the role format's block,
 * unsupported format.  NT_E_NOMEM: device allocation failed, or the model's
 * device allocations would pass the byte cap in the environment variable
 * NT_DEVICE_BYTES_LIMIT (decimal bytes; unset: no cap), a host-side stand-in
 * for running out of device memory. */
nt_status nt_model_create(const nt_config* cfg, nt_model** out);
void nt_model_destroy(nt_model* m);

/* Sets the position to 0 (cache contents are kept but no longer attended). */
nt_status nt_kv_reset(nt_model* m);

/* Fills cache positions [0, n_ctx) of every layer with N(0,1) draws rounded to
 * f16 (element (t, kv_head, d) of layer l uses counter index
 * (t*n_kv_heads + kv_head)*head_dim + d), treated as already-rotated keys, and
 * sets the position to n_ctx.  NT_E_INVAL if n_ctx > max_ctx. */
nt_status nt_kv_prefill(nt_model* m, int32_t n_ctx, uint64_t seed);

/* One decode step at the current position p (the pages' per-token loop:
 * embedding, n_layers x [RMSNorm, Q/K/V GEMV, RoPE, KV append, GQA attention,
 * O GEMV + residual, RMSNorm, gate/up GEMV, SwiGLU, down GEMV + residual],
 * final RMSNorm, output GEMV, greedy argmax with ties to the lowest id).
 * token: input id in [0, vocab).  next_token (host, required): the argmax.
 * logits_host (nullable): vocab floats.  top2_margin (nullable): top-1 minus
 * top-2 logit.  Synchronous.  Position becomes p+1.
 * A resident model runs the step as a CUDA graph of per-kernel launches.
 * NT_E_INVAL: token out of range or p == max_ctx.  NT_E_TIMEOUT: the host
 * watchdog (NT_WATCHDOG_MS, default 120 s) expired before the step finished. */
nt_status nt_decode_step(nt_model* m, int32_t token, int32_t* next_token, float* logits_host,
                         float* top2_margin);

/* n_steps greedy steps that feed each argmax back as the next input on the
 * device, starting from token; asynchronous on stream (the model's own
 * stream waits for it).  The produced ids are kept on the device
 * (nt_get_tokens).  Layer-streamed models are not supported here (NT_E_STATE);
 * use nt_decode_step. */
nt_status nt_decode_run(nt_model* m, int32_t token, int32_t n_steps, void* stream);

/* Copies the ids produced at positions [t0, t0+n) into host_out (n int32). */
nt_status nt_get_tokens(nt_model* m, int32_t t0, int32_t n, int32_t* host_out);

/* Reads n f16 cache values of (layer, kv: 0=K 1=V, kv_head) at positions
 * [t0, t0+n), head_dim values each, into host_out (n*head_dim uint16). */
nt_status nt_kv_export(nt_model* m, int32_t layer, int32_t kv, int32_t kv_head, int32_t t0, int32_t n,
                       uint16_t* host_out);

/* Layer streaming ("3-stufiges adaptives Caching": VRAM-resident layers plus
 * pinned-RAM layers copied host-to-device; "SLEP-Streaming ... Double
 * Buffering").  Layers [n_resident, n_layers) move to page-locked host memory
 * and their device copies are freed.  Every later nt_decode_step copies each
 * of them into one of n_staging device buffers on a copy stream while the
 * previous layer computes.  n_staging must be 2.  Results are bitwise
 * identical to the resident model.  Calling it again with n_resident =
 * n_layers brings every layer back to the device. */
nt_status nt_stream_layers(nt_model* m, int32_t n_resident, int32_t n_staging);

/* Tier placement ("Tier A" VRAM-resident layers, the rest streamed from pinned
 * RAM): how many layers of a model with configuration cfg fit in budget_bytes of
 * device memory next to everything else the model keeps there -- the token
 * embedding and output tensors, the K/V cache for max_ctx positions, the
 * activations and partials, and two staging buffers of one layer each when any
 * layer streams.  All layers have the same size, so the resident ones are the
 * first n.  Pure host arithmetic on the configuration (no device work).
 * n_resident (required) receives n in [0, n_layers]; device_bytes (nullable)
 * the device bytes of that placement; layer_bytes (nullable) the bytes of one
 * layer.  NT_E_INVAL: invalid configuration or negative budget.
 * NT_E_NOMEM: not even the non-layer allocations fit (n_resident is set to 0). */
nt_status nt_plan_residency(const nt_config* cfg, int64_t budget_bytes, int32_t* n_resident, int64_t* device_bytes,
                            int64_t* layer_bytes);

/* nt_stream_layers with the placement nt_plan_residency gives for the device
 * memory this model could use now: the driver's free memory plus what the
 * model already holds, minus margin_bytes.  n_resident_out (nullable) receives
 * the placement. */
nt_status nt_auto_residency(nt_model* m, int64_t margin_bytes, int32_t* n_resident_out);

/* ---- layer skip (hada "Leistung und Caching-Struktur": layer skip by cosine similarity;
 * hotdry "性能数据与瓶颈分析": the similarity between layer outputs is
 * computed beforehand and layers at or above the threshold, 0.98 there, are
 * skipped at inference) ----
 *
 * nt_layer_similarity runs one decode step exactly like nt_decode_step (same
 * result, position advanced by one, every layer evaluated whatever the skip
 * mask) and also writes cos_out[l], l < n_layers: the cosine similarity
 * between the residual stream entering layer l and leaving it, accumulated in
 * fp64 from the fp32 activations.  cos_out is host memory owned by the caller;
 * next_token as in nt_decode_step.  Works for resident and streamed models. */
nt_status nt_layer_similarity(nt_model* m, int32_t token, int32_t* next_token, double* cos_out);

/* Sets the layers later steps skip: mask[l] != 0 (n_layers bytes of host
 * memory, copied) skips layer l -- its weights are neither read nor copied from
 * the host tier, its K/V row is not written, and the residual stream passes
 * through unchanged.  mask = NULL evaluates every layer again.  Applies to
 * nt_decode_step, nt_decode_run and nt_profile_steps. */
nt_status nt_set_layer_skip(nt_model* m, const uint8_t* mask);

/* Host arithmetic: mask_out[l] = 1 for every layer with cos[l] >= threshold;
 * when max_skip > 0 and more qualify, only the max_skip most similar ones
 * (ties: lower layer first).  n_skipped (nullable) receives the count.
 * NT_E_INVAL on NULL arrays or n_layers < 0. */
nt_status nt_plan_layer_skip(const double* cos, int32_t n_layers, double threshold, int32_t max_skip,
                             uint8_t* mask_out, int32_t* n_skipped);

/* ---- self-speculative decoding (hada "Hauptfunktionen": the
 * VRAM-resident layers serve as the draft model, no extra model) ----
 *
 * One cycle from the current position p with input token `token`:
 *   draft   k greedy steps (1 <= k <= 8) of the model restricted to layers
 *           [0, n_draft) and the output head: d_1..d_k;
 *   verify  layers [n_draft, n_layers) and the head for token, d_1..d_{k-1} at
 *           positions p..p+k-1, layer by layer, so a host-tier layer is copied
 *           once per cycle rather than once per token; y_i is the full model's
 *           greedy token after position p+i;
 *   accept  j = the longest prefix with y_i == d_{i+1}; the emitted tokens are
 *           d_1..d_j, then y_j when j < k.
 * The emitted tokens are those nt_decode_step would produce from the same state,
 * bit for bit (every token gets the same arithmetic on the same inputs; layers
 * below n_draft are not recomputed, their K/V rows from the draft are the full
 * model's).  The verification runs each layer's GEMVs for several tokens per
 * launch (as nt_gemv_q_batch), so a resident layer's weights are read fewer than
 * k times; nt_stats.verify_weight_bytes reports the bytes read.  For a model
 * with every layer resident the cycle's device work is captured once as a CUDA
 * graph per (n_draft, k, skip mask) and replayed (nt_stream_layers and
 * nt_set_layer_skip discard it).  out_tokens (host, >= k entries) receives them, *n_out their count
 * (j + 1, or k when all are accepted), *n_accepted (nullable) j; the position
 * advances by *n_out.  Layers the skip mask names are skipped in both passes.
 * NT_E_INVAL: bad token, k or n_draft, or p + k > max_ctx. */
nt_status nt_speculative_step(nt_model* m, int32_t token, int32_t n_draft, int32_t k, int32_t* out_tokens,
                              int32_t* n_out, int32_t* n_accepted);

nt_status nt_get_stats(const nt_model* m, nt_stats* out);

/* Runs n_steps decode steps (from token, feeding back argmax) and returns
 * per-class device times: a CUDA event pair around every launch (not
 * graph-captured, no programmatic dependent launch).  For measurement only. */
nt_status nt_profile_steps(nt_model* m, int32_t token, int32_t n_steps, nt_kernel_times* out);

/* Times the step's GEMV launches on their own: one CUDA graph of a step's GEMV
 * launches (per layer QKV, O, gate/up, down, then the output head) as the step
 * issues them (programmatic dependent launches back to back), replayed n_reps
 * times between CUDA events on the model's stream.  Returns the mean device
 * time per GEMV launch, the mean algorithmic bytes per launch and the launches
 * per step.  The GEMVs read and overwrite the model's activations and the K/V
 * row at the current position: prefill or reset the cache afterwards.
 * Resident models only (NT_E_STATE otherwise).  For measurement only. */
nt_status nt_profile_gemvs(nt_model* m, int32_t n_reps, double* ms_per_launch, double* bytes_per_launch,
                           int32_t* launches_per_step);

/* Pointer to a weight tensor of the model (owned by the model).  For a
 * streamed layer the tensor refers to host memory: nt_qtensor_export works,
 * nt_gemv_q and nt_dequant return NT_E_STATE. */
nt_status nt_model_tensor(const nt_model* m, int32_t layer, int32_t role, const nt_qtensor** out);

/* -------------------------------------------------- quantized tensors -- */

/* A rows x cols quantized matrix (row-major, blocks along the columns)
 * generated on the device: element (r, c) is N(0, std^2) from (seed, uid,
 * r*cols + c), quantized by the format's rule.  NT_E_INVAL if cols is not a
 * multiple of the block (32 for Q8_0/Q4_0, 256 for Q4_K/Q6_K). */
nt_status nt_qtensor_create(nt_qtype type, int64_t rows, int64_t cols, uint64_t seed, uint32_t uid, float std,
                            nt_qtensor** out);
void nt_qtensor_destroy(nt_qtensor* t);

/* Format, shape and device bytes (the sum of the streams = rows*cols*bpw). */
nt_status nt_qtensor_info(const nt_qtensor* t, nt_qtype* type, int64_t* rows, int64_t* cols,
                          size_t* device_bytes);

/* Canonical block bytes of rows [row0, row0+nrows) into host_blocks;
 * nbytes must be at least nrows * (cols / block) * block_bytes. */
nt_status nt_qtensor_export(const nt_qtensor* t, int64_t row0, int64_t nrows, void* host_blocks, size_t nbytes);

/* Dequantized fp32 weights of rows [row0, row0+nrows) into dev_out
 * (nrows*cols floats, row-major), bit-exact under the formats' fp32
 * formulas (Q4_K as one fused multiply-add: fma(d*sc, q, -(dmin*m))). */
nt_status nt_dequant(const nt_qtensor* t, int64_t row0, int64_t nrows, float* dev_out, void* stream);

/* y = W x (hada "cuda/: GEMV-...-Kernel"): dev_x fp32[cols], dev_y fp32[rows].
 * Codes are multiplied exactly in integers against x carried as 16-bit fixed
 * point per 32-column block (error at most 2^-16 of the block's largest |x|);
 * per-block results are scaled and accumulated in fp32.  Asynchronous on
 * stream; launched with programmatic dependent launch, so it may start (and
 * read W) before the previous kernel on the stream ends, but reads x and
 * writes y only after it.  dev_x and dev_y must not overlap and must be
 * 16-byte aligned.  Matrices wider than 32768 columns (a multiple of 1024;
 * NT_E_UNSUPPORTED otherwise) run as launches over column windows of at most
 * 32768, each adding its window's products to y in window order. */
nt_status nt_gemv_q(const nt_qtensor* t, const float* dev_x, float* dev_y, void* stream);

/* y_i = W x_i for k vectors (1 <= k <= 8) in as few launches as fit: the
 * verification GEMV of self-speculative decoding (hada "Hauptfunktionen"), where
 * k draft tokens go through the same weights.  Each launch stages the x of up to
 * four tokens beside its weight ring and multiplies every weight tile it copies
 * by each of them, so the weights are read once per launch instead of once per
 * vector; where fewer than two x fit, one launch per vector.  Every y_i is bit for
 * bit what nt_gemv_q(t, dev_x[i], dev_y[i]) writes.  dev_x and dev_y are host
 * arrays of k device pointers (16-byte aligned; no y may overlap an x or another
 * y).  launches (nullable, host) receives the number of launches.  Asynchronous
 * on stream.  NT_E_INVAL: k outside [1, 8], NULL or misaligned vectors, overlaps. */
nt_status nt_gemv_q_batch(const nt_qtensor* t, const float* const* dev_x, float* const* dev_y, int32_t k,
                          int32_t* launches, void* stream);

/* ------------------------------------------------------------ attention -- */

/* GQA decode attention over an f16 cache, the step the decode step runs once
 * per layer (hada "Überblick": Llama with GQA and a KV cache; "Architektur und
 * Codestruktur": the softmax kernel).  For every query head j, with kv head
 * g = j / (n_heads / n_kv_heads):
 *   s_t = (q_j . K[g][t]) / sqrt(head_dim)  for t in [0, n_ctx),
 *   out_j = sum_t softmax(s)_t V[g][t]      (softmax with the maximum subtracted).
 * dev_q: fp32 [n_heads][head_dim], already rotated.  dev_k, dev_v: f16
 * [n_kv_heads][max_ctx][head_dim] (one layer of a model's cache); only
 * positions [0, n_ctx) are read.  dev_out: fp32 [n_heads][head_dim].
 * It runs the kernel the decode step launches, split into the same items as a
 * model with this max_ctx: chunks of C positions, C = max(32, 16 ceil(max_ctx/128))
 * up to max_ctx 2560 and min(320, 16 ceil(max_ctx/256)) beyond, ceil(max_ctx / C)
 * items per kv head, of which the first ceil(n_ctx / per) take
 * per = max(32, ceil(n_ctx / items)) positions each (the last the rest).  The
 * item partials are merged in a fixed order, so results do not depend on
 * timing; where the GPU can hold one thread-block cluster of a kv head's items
 * for every kv head at once the merge reads them across the cluster, otherwise
 * through the workspace, with the same arithmetic and bit-identical results.
 * dev_workspace: nt_attention_workspace_bytes() bytes of device memory or more,
 * owned by the caller; its contents on entry do not matter.  Calls that share a
 * workspace must not overlap on the GPU.  All device pointers 16-byte aligned;
 * dev_out and the workspace overlap no other buffer.
 * Asynchronous on stream: a one-CTA setup kernel, then the attention kernel.
 * NT_E_INVAL: n_ctx outside [1, max_ctx], non-positive sizes, n_heads not a
 * multiple of n_kv_heads, NULL, misaligned or overlapping pointers, a workspace
 * too small.  NT_E_UNSUPPORTED: head_dim other than 64 or 128, or n_heads /
 * n_kv_heads other than 1, 2, 4, 8 or 16. */
nt_status nt_attention_workspace_bytes(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx,
                                       size_t* bytes);
nt_status nt_attention(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx, int32_t n_ctx,
                       const float* dev_q, const void* dev_k, const void* dev_v, float* dev_out, void* dev_workspace,
                       size_t workspace_bytes, void* stream);

/* ------------------------------------------------ allocation-free variant -- */

/* y = W x as nt_gemv_q, then the index of the largest y (ties to the lowest
 * row; NaN values are never selected) into dev_index and the gap between the
 * largest and second-largest y into dev_margin (both device pointers, 4-byte
 * aligned).  dev_index is -1 only when every y is NaN; dev_margin is +inf when
 * a single y is not NaN, and NaN when the two largest are both +inf.  The pages have no counterpart: this entry point exists for
 * callers that cannot allocate device memory on this path, such as embedders
 * whose device memory is all reserved by their own allocator, or latency-bound
 * loops that cannot afford the implicit synchronisation of cudaMalloc/cudaFree.
 * It allocates nothing: the per-CTA partial results of the selection live in a
 * file-scope device array of 1024 x 16 bytes (16 KiB) that every GPU loading
 * this library holds until the process exits.  The first call on a device, with
 * that device current, looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the process; make that
 * first call before any stream capture, and make no call on a device after a
 * cudaDeviceReset of it (the reset unloads the array and the kept address goes
 * stale).
 * Every call shares the array and overwrites what it reads, so nothing needs
 * clearing, but calls that overlap on the GPU (for example on two streams at
 * once) race on it: serialise them.  Asynchronous on stream.
 * The GEMV launch is capped at 1024 CTAs, one summary slot each.
 * Errors: nt_gemv_q's argument rules; NT_E_INVAL for more than 2^31 - 2 rows;
 * NT_E_UNSUPPORTED for more than 28672 columns. */
nt_status nt_gemv_argmax_noalloc(const nt_qtensor* t, const float* dev_x, float* dev_y, int32_t* dev_index,
                                 float* dev_margin, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NT_H */
