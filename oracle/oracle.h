/*
 * oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-purpose CPU restatement of the batch-1 quantized Llama
 * decode step ("ntransformer", ai-stack / hotdry / hada.io pages), written in C
 * with fp64 arithmetic wherever the method leaves the precision open.  It exists
 * so that the CUDA library can be checked against something written from the
 * definitions alone.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it; the product path never does.  It shares no code, header,
 * table or constant generator with the CUDA library.
 *
 * Citations refer to:
 *   [hada] de.news.hada.io "ntransformer - NVMe-zu-GPU-Inferenz-Engine ...",
 *          sections "Überblick", "Hauptfunktionen", "Architektur und Codestruktur".
 *   [hotdry] blog.hotdry.top "Llama 3.1 70B单卡推理的PCIe P2P传输", section
 *          "gpu-nvme-direct的实现架构" (double buffering) and "性能数据与瓶颈分析".
 * The block formulas (w = d*q, d*(q-8), d*sc*q - dmin*m, d*sc*(q-32)) are the
 * ones the workload definitions fix for Q8_0 / Q4_0 / Q4_K / Q6_K; the quantizer
 * rules, the byte packing, the generator and the RoPE pairing are readings the
 * pages leave open (each stated beside its function).
 *
 * Parity status: every function is pinned by a test in tests/test_oracle_*.py
 * (hand-worked blocks, closed forms, invariants, brute force on tiny inputs),
 * except the composed decode step, which is pinned only through its parts and
 * through the degenerate zero-layer case.
 */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Format codes used by the oracle (its own numbering). */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_Q8_0 = 2, ORC_Q4_0 = 3, ORC_Q4_K = 4, ORC_Q6_K = 5, ORC_Q5_K = 6 };

/* Elements per block and bytes per block of each quantized format. */
int orc_block_elems(int qtype);
int orc_block_bytes(int qtype);

/* ---- counter-based generator (SplitMix64 finaliser + Irwin-Hall sum) ---- */
uint64_t orc_mix64(uint64_t z);
float    orc_normal(uint64_t seed, uint32_t uid, uint64_t i);      /* z, approx N(0,1) */
void     orc_gen_normal(uint64_t seed, uint32_t uid, uint64_t i0, int64_t n, float std, float* out);
int32_t  orc_token(uint64_t seed, uint32_t uid, uint64_t i, int32_t vocab);

/* ---- IEEE binary16 ---- */
uint16_t orc_f16_from_double(double x);      /* round to nearest, ties to even */
double   orc_f16_to_double(uint16_t h);

/* ---- block formats (canonical AoS bytes, little-endian) ---- */
int  orc_quantize_row(int qtype, const float* w, int64_t n, uint8_t* blocks);
int  orc_dequant_row(int qtype, const uint8_t* blocks, int64_t n, float* w);
/* generate rows [row0,row0+nrows) of a rows x cols tensor from (seed, uid, std) and quantize */
int  orc_qtensor_rows(int qtype, int64_t rows, int64_t cols, uint64_t seed, uint32_t uid, float std,
                      int64_t row0, int64_t nrows, uint8_t* out_blocks, int nthreads);

/* y[r] = sum_c (double)w[r][c] * (double)x[c], rows of canonical blocks */
int  orc_gemv(int qtype, const uint8_t* blocks, int64_t rows, int64_t cols, const float* x, double* y,
              int nthreads);
int  orc_gemv_d(int qtype, const uint8_t* blocks, int64_t rows, int64_t cols, const double* x, double* y,
                int nthreads);

/* ---- small ops, fp64 ---- */
void   orc_rmsnorm(const double* x, int64_t n, double eps, double* out);
void   orc_rope(double* v, int n_heads, int head_dim, int64_t pos, double theta);
void   orc_softmax(const double* s, int64_t n, double* p);
double orc_silu(double z);
/* one query head against cached f16 keys/values k[t*head_dim+d], t < n_ctx */
void   orc_attend(const double* q, const uint16_t* k, const uint16_t* v, int64_t n_ctx, int head_dim,
                  double* out);
int64_t orc_argmax(const double* x, int64_t n, double* top2_margin);

/* ---- the decode step ---- */
typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, max_ctx;
  double  rms_eps, rope_theta;
  float   init_std;
  int32_t t_embd, t_q, t_k, t_v, t_o, t_gate, t_up, t_down, t_out;
  uint64_t seed;
  int32_t lazy;       /* 1: generate each layer when it is used and free it after */
  int32_t nthreads;   /* worker threads for row-parallel generation and GEMV */
} orc_config;

typedef struct orc_model orc_model;

/* uid scheme for generated tensors */
#define ORC_UID_LAYER(l, role) ((uint32_t)((l) * 16 + (role)))
#define ORC_UID_EMBD   0x100000u
#define ORC_UID_OUTPUT 0x100001u
#define ORC_UID_KV(l, kv) ((uint32_t)(0x200000u + 2u * (uint32_t)(l) + (uint32_t)(kv)))
#define ORC_UID_TOKENS 0x300000u

enum { ORC_ROLE_Q = 0, ORC_ROLE_K, ORC_ROLE_V, ORC_ROLE_O, ORC_ROLE_GATE, ORC_ROLE_UP, ORC_ROLE_DOWN };

orc_model* orc_model_create(const orc_config* cfg);
void       orc_model_destroy(orc_model* m);
int        orc_kv_reset(orc_model* m);
int        orc_set_pos(orc_model* m, int32_t pos);
int        orc_kv_prefill(orc_model* m, int32_t n_ctx, uint64_t seed);
int32_t    orc_pos(const orc_model* m);
void       orc_set_threads(orc_model* m, int32_t nthreads);
/* logits (vocab doubles, nullable), next token, top-2 margin (nullable) */
int        orc_decode_step(orc_model* m, int32_t token, double* logits, int32_t* next, double* margin);
/* Layer skip: mask[l] != 0 skips layer l (no arithmetic, no K/V row); NULL clears. */
int        orc_set_layer_skip(orc_model* m, const uint8_t* mask);
/* last step: cosine similarity between the residual entering and leaving each layer (1 when skipped) */
void       orc_layer_cos(const orc_model* m, double* out);
/* last step: residual stream after the last layer (before the output norm) */
void       orc_hidden(const orc_model* m, double* out);
double     orc_cosine(const double* a, const double* b, int64_t n);
/* read one cached f16 value (for tests) */
uint16_t   orc_kv_get(const orc_model* m, int layer, int kv, int kv_head, int t, int d);

#ifdef __cplusplus
}
#endif
#endif
