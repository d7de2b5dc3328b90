/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Plain C, no vector intrinsics, no fused arithmetic except where a formula
 * names one (the Q4_K dequant).  Build with -ffp-contract=off so the compiler
 * does not fuse multiplies and adds on its own.  Threads, where used, split
 * independent rows; every row is computed exactly as in the single-threaded case.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* formats                                                                   */
/* ------------------------------------------------------------------------ */

int orc_block_elems(int qtype) {
  switch (qtype) {
    case ORC_F32: case ORC_F16: return 1;
    case ORC_Q8_0: case ORC_Q4_0: return 32;
    case ORC_Q4_K: case ORC_Q5_K: case ORC_Q6_K: return 256;
  }
  return 0;
}

int orc_block_bytes(int qtype) {
  switch (qtype) {
    case ORC_F32: return 4;
    case ORC_F16: return 2;
    case ORC_Q8_0: return 34;   /* f16 d | int8 q[32]                         */
    case ORC_Q4_0: return 18;   /* f16 d | u8 qs[16]                          */
    case ORC_Q4_K: return 144;  /* f16 d | f16 dmin | 12 B scales | u8 qs[128] */
    case ORC_Q6_K: return 210;  /* u8 ql[128] | u8 qh[64] | int8 sc[16] | f16 d */
    case ORC_Q5_K: return 176;  /* f16 d | f16 dmin | 12 B scales | u8 qh[32] | u8 qs[128] */
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* generator: SplitMix64 output function (Steele, Lea, Flood, "Fast Splittable */
/* Pseudorandom Number Generators", OOPSLA 2014) applied to a counter, and an  */
/* Irwin-Hall sum of twelve 16-bit uniforms as the normal draw.               */
/* ------------------------------------------------------------------------ */

static const uint64_t ORC_GAMMA = 0x9E3779B97F4A7C15ull;

uint64_t orc_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* r_j = mix64(seed + gamma * (uid * 2^40 + 3 i + j + 1)), j = 0..2; the 192 bits
 * give twelve 16-bit lanes u_k and z = (sum u_k - 393210) / 65536, which equals
 * sum_k (u_k + 0.5) / 65536 - 6 (mean 0, variance 12 * (1/12) = 1).            */
float orc_normal(uint64_t seed, uint32_t uid, uint64_t i) {
  uint64_t base = ((uint64_t)uid << 40) + 3u * i;
  int64_t s = 0;
  for (int j = 0; j < 3; j++) {
    uint64_t r = orc_mix64(seed + ORC_GAMMA * (base + (uint64_t)j + 1u));
    for (int k = 0; k < 4; k++) s += (int64_t)((r >> (16 * k)) & 0xFFFFu);
  }
  return (float)(s - 393210) / 65536.0f;
}

void orc_gen_normal(uint64_t seed, uint32_t uid, uint64_t i0, int64_t n, float std, float* out) {
  for (int64_t k = 0; k < n; k++) out[k] = orc_normal(seed, uid, i0 + (uint64_t)k) * std;
}

int32_t orc_token(uint64_t seed, uint32_t uid, uint64_t i, int32_t vocab) {
  uint64_t r = orc_mix64(seed + ORC_GAMMA * (((uint64_t)uid << 40) + 3u * i + 1u));
  return (int32_t)(r % (uint64_t)vocab);
}

/* ------------------------------------------------------------------------ */
/* binary16 (IEEE 754-2008): 1 sign, 5 exponent (bias 15), 10 fraction bits   */
/* ------------------------------------------------------------------------ */

uint16_t orc_f16_from_double(double x) {
  if (isnan(x)) return 0x7E00;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);                         /* a = f * 2^e, f in [0.5, 1) */
  int E = e - 1;                        /* floor(log2 a) */
  if (E < -14) E = -14;                 /* subnormal range: spacing 2^-24 */
  if (E > 16) E = 16;
  double spacing = ldexp(1.0, E - 10);
  double m = nearbyint(a / spacing);    /* exact quotient, rounded to nearest even */
  double v = m * spacing;
  if (v >= 65536.0) return sign | 0x7C00;   /* beyond the largest finite (65504) */
  if (v < ldexp(1.0, -14)) return sign | (uint16_t)(v / ldexp(1.0, -24));
  frexp(v, &e);
  E = e - 1;
  uint16_t frac = (uint16_t)(v / ldexp(1.0, E - 10) - 1024.0);
  return sign | (uint16_t)((E + 15) << 10) | frac;
}

double orc_f16_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)f, -24);
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp(1024.0 + f, e - 25);
  return s ? -v : v;
}

static float h2f(uint16_t h) { return (float)orc_f16_to_double(h); }
static uint16_t f2h(float x) { return orc_f16_from_double((double)x); }
static void put16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }
static uint16_t get16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }
/* roundf: nearest, halfway cases away from zero */
static int rnd(float v) { return (int)roundf(v); }

/* 4-bit codes: element k in byte k/2, low nibble for even k */
static void put_nib(uint8_t* qs, int k, int q) {
  if (k & 1) qs[k >> 1] = (uint8_t)((qs[k >> 1] & 0x0F) | (q << 4));
  else qs[k >> 1] = (uint8_t)((qs[k >> 1] & 0xF0) | (q & 0x0F));
}
static int get_nib(const uint8_t* qs, int k) { return (qs[k >> 1] >> ((k & 1) * 4)) & 0x0F; }

/* Q4_K scale/min fields: sixteen 6-bit fields (sc_0..7 then m_0..7) packed
 * least-significant-bit first into 12 bytes: field f occupies bits [6f, 6f+6). */
static void put6(uint8_t* s, int f, int v) {
  for (int b = 0; b < 6; b++) {
    int bit = 6 * f + b;
    if ((v >> b) & 1) s[bit >> 3] |= (uint8_t)(1u << (bit & 7));
    else s[bit >> 3] &= (uint8_t)~(1u << (bit & 7));
  }
}
static int get6(const uint8_t* s, int f) {
  int v = 0;
  for (int b = 0; b < 6; b++) {
    int bit = 6 * f + b;
    v |= ((s[bit >> 3] >> (bit & 7)) & 1) << b;
  }
  return v;
}

/* Q6_K codes: low 4 bits as the 4-bit layout in ql[128]; high 2 bits of
 * element k in qh[k/4] at bits 2*(k%4). */
static void put_q6(uint8_t* ql, uint8_t* qh, int k, int q) {
  put_nib(ql, k, q & 0x0F);
  int sh = 2 * (k & 3);
  qh[k >> 2] = (uint8_t)((qh[k >> 2] & ~(3u << sh)) | (((q >> 4) & 3) << sh));
}
static int get_q6(const uint8_t* ql, const uint8_t* qh, int k) {
  return get_nib(ql, k) | (((qh[k >> 2] >> (2 * (k & 3))) & 3) << 4);
}

/* Q5_K codes: low 4 bits as the 4-bit layout in qs[128]; the fifth bit of
 * element k in qh[k/8] at bit k%8. */
static void put_q5(uint8_t* qs, uint8_t* qh, int k, int q) {
  put_nib(qs, k, q & 0x0F);
  qh[k >> 3] = (uint8_t)((qh[k >> 3] & ~(1u << (k & 7))) | (((q >> 4) & 1) << (k & 7)));
}
static int get_q5(const uint8_t* qs, const uint8_t* qh, int k) {
  return get_nib(qs, k) | (((qh[k >> 3] >> (k & 7)) & 1) << 4);
}

/* Q8_0: d32 = absmax/127, d = f16(d32), q = clamp(round(w/d32), -127, 127). */
static void quant_q8_0(const float* w, uint8_t* blk) {
  float amax = 0.0f;
  for (int k = 0; k < 32; k++) amax = fmaxf(amax, fabsf(w[k]));
  float d32 = amax / 127.0f;
  put16(blk, f2h(d32));
  for (int k = 0; k < 32; k++) {
    int q = (d32 == 0.0f) ? 0 : clampi(rnd(w[k] / d32), -127, 127);
    blk[2 + k] = (uint8_t)(int8_t)q;
  }
}

/* Q4_0 (symmetric reading): d32 = absmax/7, d = f16(d32), q = clamp(round(w/d32)+8, 0, 15). */
static void quant_q4_0(const float* w, uint8_t* blk) {
  float amax = 0.0f;
  for (int k = 0; k < 32; k++) amax = fmaxf(amax, fabsf(w[k]));
  float d32 = amax / 7.0f;
  put16(blk, f2h(d32));
  memset(blk + 2, 0, 16);
  for (int k = 0; k < 32; k++) {
    int q = (d32 == 0.0f) ? 8 : clampi(rnd(w[k] / d32) + 8, 0, 15);
    put_nib(blk + 2, k, q);
  }
}

/* Q4_K: per 32-element sub-block j: lo = min(0, min w), hi = max w,
 * s_j = (hi - lo)/15, m*_j = -lo; d = f16(max s / 63), dmin = f16(max m* / 63);
 * sc_j = clamp(round(s_j/d), 0, 63), m_j = clamp(round(m*_j/dmin), 0, 63);
 * q = clamp(round((w + dmin*m_j) / (d*sc_j)), 0, 15), 0 where d*sc_j = 0. */
static void quant_q4_k(const float* w, uint8_t* blk) {
  float s[8], ms[8], smax = 0.0f, mmax = 0.0f;
  for (int j = 0; j < 8; j++) {
    float lo = 0.0f, hi = w[32 * j];
    for (int k = 0; k < 32; k++) {
      lo = fminf(lo, w[32 * j + k]);
      hi = fmaxf(hi, w[32 * j + k]);
    }
    s[j] = (hi - lo) / 15.0f;
    ms[j] = -lo;
    smax = fmaxf(smax, s[j]);
    mmax = fmaxf(mmax, ms[j]);
  }
  uint16_t dh = f2h(smax / 63.0f), mh = f2h(mmax / 63.0f);
  float d = h2f(dh), dmin = h2f(mh);
  put16(blk, dh);
  put16(blk + 2, mh);
  memset(blk + 4, 0, 12 + 128);
  int sc[8], mm[8];
  for (int j = 0; j < 8; j++) {
    sc[j] = (d == 0.0f) ? 0 : clampi(rnd(s[j] / d), 0, 63);
    mm[j] = (dmin == 0.0f) ? 0 : clampi(rnd(ms[j] / dmin), 0, 63);
    put6(blk + 4, j, sc[j]);
    put6(blk + 4, 8 + j, mm[j]);
  }
  for (int j = 0; j < 8; j++) {
    float a = d * (float)sc[j];
    float b = dmin * (float)mm[j];
    for (int k = 0; k < 32; k++) {
      int q = (a == 0.0f) ? 0 : clampi(rnd((w[32 * j + k] + b) / a), 0, 15);
      put_nib(blk + 16, 32 * j + k, q);
    }
  }
}

/* Q5_K: the Q4_K rule with 32 levels: per 32-element sub-block j: lo = min(0, min w),
 * hi = max w, s_j = (hi - lo)/31, m*_j = -lo; d = f16(max s / 63),
 * dmin = f16(max m* / 63); sc_j = clamp(round(s_j/d), 0, 63),
 * m_j = clamp(round(m*_j/dmin), 0, 63); q = clamp(round((w + dmin*m_j) / (d*sc_j)), 0, 31),
 * 0 where d*sc_j = 0. */
static void quant_q5_k(const float* w, uint8_t* blk) {
  float s[8], ms[8], smax = 0.0f, mmax = 0.0f;
  for (int j = 0; j < 8; j++) {
    float lo = 0.0f, hi = w[32 * j];
    for (int k = 0; k < 32; k++) {
      lo = fminf(lo, w[32 * j + k]);
      hi = fmaxf(hi, w[32 * j + k]);
    }
    s[j] = (hi - lo) / 31.0f;
    ms[j] = -lo;
    smax = fmaxf(smax, s[j]);
    mmax = fmaxf(mmax, ms[j]);
  }
  uint16_t dh = f2h(smax / 63.0f), mh = f2h(mmax / 63.0f);
  float d = h2f(dh), dmin = h2f(mh);
  put16(blk, dh);
  put16(blk + 2, mh);
  memset(blk + 4, 0, 12 + 32 + 128);
  int sc[8], mm[8];
  for (int j = 0; j < 8; j++) {
    sc[j] = (d == 0.0f) ? 0 : clampi(rnd(s[j] / d), 0, 63);
    mm[j] = (dmin == 0.0f) ? 0 : clampi(rnd(ms[j] / dmin), 0, 63);
    put6(blk + 4, j, sc[j]);
    put6(blk + 4, 8 + j, mm[j]);
  }
  for (int j = 0; j < 8; j++) {
    float a = d * (float)sc[j];
    float b = dmin * (float)mm[j];
    for (int k = 0; k < 32; k++) {
      int q = (a == 0.0f) ? 0 : clampi(rnd((w[32 * j + k] + b) / a), 0, 31);
      put_q5(blk + 48, blk + 16, 32 * j + k, q);
    }
  }
}

/* Q6_K: per 16-element sub-block j: s_j = absmax/31; d = f16(max s / 127);
 * sc_j = clamp(round(s_j/d), 0, 127); q = clamp(round(w/(d*sc_j)) + 32, 0, 63),
 * 32 where d*sc_j = 0. */
static void quant_q6_k(const float* w, uint8_t* blk) {
  float s[16], smax = 0.0f;
  for (int j = 0; j < 16; j++) {
    float amax = 0.0f;
    for (int k = 0; k < 16; k++) amax = fmaxf(amax, fabsf(w[16 * j + k]));
    s[j] = amax / 31.0f;
    smax = fmaxf(smax, s[j]);
  }
  uint16_t dh = f2h(smax / 127.0f);
  float d = h2f(dh);
  uint8_t* ql = blk;
  uint8_t* qh = blk + 128;
  int8_t* scs = (int8_t*)(blk + 192);
  memset(blk, 0, 208);
  put16(blk + 208, dh);
  for (int j = 0; j < 16; j++) {
    int sc = (d == 0.0f) ? 0 : clampi(rnd(s[j] / d), 0, 127);
    scs[j] = (int8_t)sc;
    float a = d * (float)sc;
    for (int k = 0; k < 16; k++) {
      int q = (a == 0.0f) ? 32 : clampi(rnd(w[16 * j + k] / a) + 32, 0, 63);
      put_q6(ql, qh, 16 * j + k, q);
    }
  }
}

int orc_quantize_row(int qtype, const float* w, int64_t n, uint8_t* blocks) {
  int qk = orc_block_elems(qtype), bb = orc_block_bytes(qtype);
  if (qk == 0 || n % qk) return -1;
  for (int64_t b = 0; b < n / qk; b++) {
    const float* wb = w + b * qk;
    uint8_t* ob = blocks + b * bb;
    switch (qtype) {
      case ORC_F32: memcpy(ob, wb, 4); break;
      case ORC_F16: put16(ob, f2h(*wb)); break;
      case ORC_Q8_0: quant_q8_0(wb, ob); break;
      case ORC_Q4_0: quant_q4_0(wb, ob); break;
      case ORC_Q4_K: quant_q4_k(wb, ob); break;
      case ORC_Q6_K: quant_q6_k(wb, ob); break;
      case ORC_Q5_K: quant_q5_k(wb, ob); break;
    }
  }
  return 0;
}

/* Dequantization, the stated fp32 formulas, one rounding per operation:
 *   Q8_0  w = d * q
 *   Q4_0  w = d * (q - 8)
 *   Q4_K  w = fma(d*sc, q, -(dmin*m))     (a single fused multiply-add)
 *   Q5_K  w = fma(d*sc, q, -(dmin*m))     (as Q4_K, q in 0..31)
 *   Q6_K  w = (d*sc) * (q - 32)                                              */
int orc_dequant_row(int qtype, const uint8_t* blocks, int64_t n, float* w) {
  int qk = orc_block_elems(qtype), bb = orc_block_bytes(qtype);
  if (qk == 0 || n % qk) return -1;
  for (int64_t b = 0; b < n / qk; b++) {
    const uint8_t* blk = blocks + b * bb;
    float* wb = w + b * qk;
    switch (qtype) {
      case ORC_F32: memcpy(wb, blk, 4); break;
      case ORC_F16: wb[0] = h2f(get16(blk)); break;
      case ORC_Q8_0: {
        float d = h2f(get16(blk));
        for (int k = 0; k < 32; k++) wb[k] = d * (float)(int8_t)blk[2 + k];
      } break;
      case ORC_Q4_0: {
        float d = h2f(get16(blk));
        for (int k = 0; k < 32; k++) wb[k] = d * (float)(get_nib(blk + 2, k) - 8);
      } break;
      case ORC_Q4_K: {
        float d = h2f(get16(blk)), dmin = h2f(get16(blk + 2));
        for (int j = 0; j < 8; j++) {
          float a = d * (float)get6(blk + 4, j);
          float bm = dmin * (float)get6(blk + 4, 8 + j);
          for (int k = 0; k < 32; k++)
            wb[32 * j + k] = fmaf(a, (float)get_nib(blk + 16, 32 * j + k), -bm);
        }
      } break;
      case ORC_Q5_K: {
        float d = h2f(get16(blk)), dmin = h2f(get16(blk + 2));
        for (int j = 0; j < 8; j++) {
          float a = d * (float)get6(blk + 4, j);
          float bm = dmin * (float)get6(blk + 4, 8 + j);
          for (int k = 0; k < 32; k++)
            wb[32 * j + k] = fmaf(a, (float)get_q5(blk + 48, blk + 16, 32 * j + k), -bm);
        }
      } break;
      case ORC_Q6_K: {
        float d = h2f(get16(blk + 208));
        const int8_t* scs = (const int8_t*)(blk + 192);
        for (int j = 0; j < 16; j++) {
          float a = d * (float)scs[j];
          for (int k = 0; k < 16; k++)
            wb[16 * j + k] = a * (float)(get_q6(blk, blk + 128, 16 * j + k) - 32);
        }
      } break;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* row-parallel helpers (threads only split independent rows)                */
/* ------------------------------------------------------------------------ */

typedef struct {
  int kind;  /* 0 = generate+quantize, 1 = gemv (float x), 2 = gemv (double x) */
  int qtype;
  int64_t rows, cols, r_begin, r_end;
  uint64_t seed;
  uint32_t uid;
  float std;
  int64_t row0;
  uint8_t* blocks;
  const uint8_t* cblocks;
  const float* xf;
  const double* xd;
  double* y;
  int err;
} orc_job;

static int64_t row_bytes(int qtype, int64_t cols) {
  return cols / orc_block_elems(qtype) * orc_block_bytes(qtype);
}

static void* orc_worker(void* arg) {
  orc_job* j = (orc_job*)arg;
  float* buf = (float*)malloc(sizeof(float) * (size_t)j->cols);
  if (!buf) { j->err = -2; return NULL; }
  int64_t rb = row_bytes(j->qtype, j->cols);
  for (int64_t r = j->r_begin; r < j->r_end; r++) {
    if (j->kind == 0) {
      int64_t gr = j->row0 + r;  /* global row */
      orc_gen_normal(j->seed, j->uid, (uint64_t)(gr * j->cols), j->cols, j->std, buf);
      if (orc_quantize_row(j->qtype, buf, j->cols, j->blocks + r * rb)) j->err = -1;
    } else {
      if (orc_dequant_row(j->qtype, j->cblocks + r * rb, j->cols, buf)) { j->err = -1; continue; }
      double acc = 0.0;
      if (j->kind == 1)
        for (int64_t c = 0; c < j->cols; c++) acc += (double)buf[c] * (double)j->xf[c];
      else
        for (int64_t c = 0; c < j->cols; c++) acc += (double)buf[c] * j->xd[c];
      j->y[r] = acc;
    }
  }
  free(buf);
  return NULL;
}

static int run_rows(orc_job proto, int64_t nrows, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nrows < nthreads) nthreads = nrows > 0 ? (int)nrows : 1;
  orc_job jobs[256];
  pthread_t th[256];
  int live[256];
  int64_t per = (nrows + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; t++) {
    jobs[t] = proto;
    jobs[t].r_begin = t * per;
    jobs[t].r_end = (t + 1) * per < nrows ? (t + 1) * per : nrows;
    jobs[t].err = 0;
    live[t] = 0;
    if (jobs[t].r_begin >= jobs[t].r_end) continue;
    if (nthreads > 1 && pthread_create(&th[t], NULL, orc_worker, &jobs[t]) == 0) live[t] = 1;
    else orc_worker(&jobs[t]);
  }
  int err = 0;
  for (int t = 0; t < nthreads; t++) {
    if (live[t]) pthread_join(th[t], NULL);
    if (jobs[t].err) err = jobs[t].err;
  }
  return err;
}

int orc_qtensor_rows(int qtype, int64_t rows, int64_t cols, uint64_t seed, uint32_t uid, float std,
                     int64_t row0, int64_t nrows, uint8_t* out_blocks, int nthreads) {
  int qk = orc_block_elems(qtype);
  if (qk == 0 || cols % qk || row0 < 0 || nrows < 0 || row0 + nrows > rows) return -1;
  orc_job p;
  memset(&p, 0, sizeof p);
  p.kind = 0; p.qtype = qtype; p.rows = rows; p.cols = cols; p.seed = seed; p.uid = uid;
  p.std = std; p.row0 = row0; p.blocks = out_blocks;
  return run_rows(p, nrows, nthreads);
}

int orc_gemv(int qtype, const uint8_t* blocks, int64_t rows, int64_t cols, const float* x, double* y,
             int nthreads) {
  int qk = orc_block_elems(qtype);
  if (qk == 0 || cols % qk) return -1;
  orc_job p;
  memset(&p, 0, sizeof p);
  p.kind = 1; p.qtype = qtype; p.rows = rows; p.cols = cols; p.cblocks = blocks; p.xf = x; p.y = y;
  return run_rows(p, rows, nthreads);
}

int orc_gemv_d(int qtype, const uint8_t* blocks, int64_t rows, int64_t cols, const double* x, double* y,
               int nthreads) {
  int qk = orc_block_elems(qtype);
  if (qk == 0 || cols % qk) return -1;
  orc_job p;
  memset(&p, 0, sizeof p);
  p.kind = 2; p.qtype = qtype; p.rows = rows; p.cols = cols; p.cblocks = blocks; p.xd = x; p.y = y;
  return run_rows(p, rows, nthreads);
}

/* ------------------------------------------------------------------------ */
/* small ops (architecture list in [hada] "Hauptfunktionen": RoPE, GQA,       */
/* SwiGLU, RMSNorm, KV cache; kernel list in "Architektur und Codestruktur") */
/* ------------------------------------------------------------------------ */

/* RMSNorm with unit gains: x / sqrt(mean(x^2) + eps) */
void orc_rmsnorm(const double* x, int64_t n, double eps, double* out) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; i++) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int64_t i = 0; i < n; i++) out[i] = x[i] * inv;
}

/* RoPE, adjacent-pair reading: pair (2i, 2i+1) of every head is rotated by
 * the angle pos * theta^(-2i/head_dim). */
void orc_rope(double* v, int n_heads, int head_dim, int64_t pos, double theta) {
  for (int h = 0; h < n_heads; h++) {
    double* hv = v + (int64_t)h * head_dim;
    for (int i = 0; i < head_dim / 2; i++) {
      double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)head_dim);
      double c = cos(ang), s = sin(ang);
      double a = hv[2 * i], b = hv[2 * i + 1];
      hv[2 * i] = a * c - b * s;
      hv[2 * i + 1] = a * s + b * c;
    }
  }
}

/* softmax with the maximum subtracted first */
void orc_softmax(const double* s, int64_t n, double* p) {
  double mx = -INFINITY;
  for (int64_t i = 0; i < n; i++) mx = s[i] > mx ? s[i] : mx;
  double sum = 0.0;
  for (int64_t i = 0; i < n; i++) { p[i] = exp(s[i] - mx); sum += p[i]; }
  for (int64_t i = 0; i < n; i++) p[i] /= sum;
}

/* silu(z) = z / (1 + e^-z) */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* scores s_t = q.k_t / sqrt(head_dim), p = softmax(s), out = sum_t p_t v_t */
void orc_attend(const double* q, const uint16_t* k, const uint16_t* v, int64_t n_ctx, int head_dim,
                double* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_ctx > 0 ? n_ctx : 1));
  double* p = (double*)malloc(sizeof(double) * (size_t)(n_ctx > 0 ? n_ctx : 1));
  double scale = 1.0 / sqrt((double)head_dim);
  for (int64_t t = 0; t < n_ctx; t++) {
    double acc = 0.0;
    for (int d = 0; d < head_dim; d++) acc += q[d] * orc_f16_to_double(k[t * head_dim + d]);
    s[t] = acc * scale;
  }
  orc_softmax(s, n_ctx, p);
  for (int d = 0; d < head_dim; d++) {
    double acc = 0.0;
    for (int64_t t = 0; t < n_ctx; t++) acc += p[t] * orc_f16_to_double(v[t * head_dim + d]);
    out[d] = acc;
  }
  free(s);
  free(p);
}

/* greedy choice: largest value, lowest index on ties; margin = top1 - top2 */
int64_t orc_argmax(const double* x, int64_t n, double* top2_margin) {
  int64_t best = 0;
  for (int64_t i = 1; i < n; i++) if (x[i] > x[best]) best = i;
  if (top2_margin) {
    double second = -INFINITY;
    for (int64_t i = 0; i < n; i++) if (i != best && x[i] > second) second = x[i];
    *top2_margin = x[best] - second;
  }
  return best;
}

/* ------------------------------------------------------------------------ */
/* model                                                                      */
/* ------------------------------------------------------------------------ */

struct orc_model {
  orc_config c;
  uint8_t* embd;         /* vocab x hidden, canonical blocks (always generated: only one row is read,
                            but the tiny case keeps it whole; large cases generate the needed row)   */
  uint8_t* output;       /* vocab x hidden (NULL when lazy)                                          */
  uint8_t** layer;       /* [n_layers][7] tensors (NULL entries when lazy)                           */
  uint16_t* kv;          /* [n_layers][2][n_kv_heads][max_ctx][head_dim] binary16                    */
  int32_t pos;
  uint8_t* skip;         /* [n_layers]: 1 = layer skipped (NULL: none)                               */
  double* layer_cos;     /* [n_layers]: cosine between the residual entering and leaving each layer  */
  double* hidden;        /* [hidden]: residual stream after the last layer, last step                */
};

static void role_shape(const orc_config* c, int role, int64_t* rows, int64_t* cols, int* qt) {
  int64_t h = c->hidden, qd = (int64_t)c->n_heads * c->head_dim, kd = (int64_t)c->n_kv_heads * c->head_dim;
  int64_t f = c->ffn_dim;
  switch (role) {
    case ORC_ROLE_Q: *rows = qd; *cols = h; *qt = c->t_q; break;
    case ORC_ROLE_K: *rows = kd; *cols = h; *qt = c->t_k; break;
    case ORC_ROLE_V: *rows = kd; *cols = h; *qt = c->t_v; break;
    case ORC_ROLE_O: *rows = h; *cols = qd; *qt = c->t_o; break;
    case ORC_ROLE_GATE: *rows = f; *cols = h; *qt = c->t_gate; break;
    case ORC_ROLE_UP: *rows = f; *cols = h; *qt = c->t_up; break;
    default: *rows = h; *cols = f; *qt = c->t_down; break;
  }
}

static uint8_t* gen_tensor(const orc_config* c, int qt, int64_t rows, int64_t cols, uint32_t uid) {
  uint8_t* b = (uint8_t*)malloc((size_t)(rows * row_bytes(qt, cols)));
  if (!b) return NULL;
  if (orc_qtensor_rows(qt, rows, cols, c->seed, uid, c->init_std, 0, rows, b, c->nthreads)) {
    free(b);
    return NULL;
  }
  return b;
}

static uint8_t* gen_layer_tensor(const orc_config* c, int l, int role) {
  int64_t rows, cols;
  int qt;
  role_shape(c, role, &rows, &cols, &qt);
  return gen_tensor(c, qt, rows, cols, ORC_UID_LAYER(l, role));
}

orc_model* orc_model_create(const orc_config* cfg) {
  orc_model* m = (orc_model*)calloc(1, sizeof(orc_model));
  if (!m) return NULL;
  m->c = *cfg;
  const orc_config* c = &m->c;
  m->layer = (uint8_t**)calloc((size_t)c->n_layers * 7, sizeof(uint8_t*));
  size_t kvn = (size_t)c->n_layers * 2 * c->n_kv_heads * (size_t)c->max_ctx * c->head_dim;
  m->kv = (uint16_t*)calloc(kvn > 0 ? kvn : 1, sizeof(uint16_t));
  m->layer_cos = (double*)calloc((size_t)(c->n_layers > 0 ? c->n_layers : 1), sizeof(double));
  m->hidden = (double*)calloc((size_t)c->hidden, sizeof(double));
  if (!m->layer || !m->kv || !m->layer_cos || !m->hidden) { orc_model_destroy(m); return NULL; }
  if (!c->lazy) {
    m->embd = gen_tensor(c, c->t_embd, c->vocab, c->hidden, ORC_UID_EMBD);
    m->output = gen_tensor(c, c->t_out, c->vocab, c->hidden, ORC_UID_OUTPUT);
    if (!m->embd || !m->output) { orc_model_destroy(m); return NULL; }
    for (int l = 0; l < c->n_layers; l++)
      for (int r = 0; r < 7; r++) {
        m->layer[l * 7 + r] = gen_layer_tensor(c, l, r);
        if (!m->layer[l * 7 + r]) { orc_model_destroy(m); return NULL; }
      }
  }
  return m;
}

void orc_model_destroy(orc_model* m) {
  if (!m) return;
  if (m->layer)
    for (int i = 0; i < m->c.n_layers * 7; i++) free(m->layer[i]);
  free(m->layer);
  free(m->embd);
  free(m->output);
  free(m->kv);
  free(m->skip);
  free(m->layer_cos);
  free(m->hidden);
  free(m);
}

/* Layer skip ([hada] "Leistung und Caching-Struktur": layers skipped by cosine similarity;
 * [hotdry] "性能数据与瓶颈分析": similarity between layer outputs is computed
 * beforehand and layers above the threshold are skipped at inference).  Reading:
 * a skipped layer is not evaluated at all -- the residual stream passes through
 * unchanged and no K/V row is written for it. */
int orc_set_layer_skip(orc_model* m, const uint8_t* mask) {
  if (!mask) {
    free(m->skip);
    m->skip = NULL;
    return 0;
  }
  if (!m->skip) m->skip = (uint8_t*)malloc((size_t)(m->c.n_layers > 0 ? m->c.n_layers : 1));
  if (!m->skip) return -2;
  for (int l = 0; l < m->c.n_layers; l++) m->skip[l] = mask[l] ? 1 : 0;
  return 0;
}

void orc_layer_cos(const orc_model* m, double* out) {
  memcpy(out, m->layer_cos, sizeof(double) * (size_t)m->c.n_layers);
}

void orc_hidden(const orc_model* m, double* out) { memcpy(out, m->hidden, sizeof(double) * (size_t)m->c.hidden); }

/* cos(a, b) = sum a_i b_i / (sqrt(sum a_i^2) sqrt(sum b_i^2)); 0 when either is the zero vector. */
double orc_cosine(const double* a, const double* b, int64_t n) {
  double ab = 0, aa = 0, bb = 0;
  for (int64_t i = 0; i < n; i++) {
    ab += a[i] * b[i];
    aa += a[i] * a[i];
    bb += b[i] * b[i];
  }
  if (aa == 0 || bb == 0) return 0;
  return ab / (sqrt(aa) * sqrt(bb));
}

int32_t orc_pos(const orc_model* m) { return m->pos; }

void orc_set_threads(orc_model* m, int32_t nthreads) { m->c.nthreads = nthreads < 1 ? 1 : nthreads; }

int orc_kv_reset(orc_model* m) {
  m->pos = 0;
  return 0;
}

/* Moves the position (rows at and past it are overwritten as decoding reaches them). */
int orc_set_pos(orc_model* m, int32_t pos) {
  if (pos < 0 || pos > m->c.max_ctx) return -1;
  m->pos = pos;
  return 0;
}

static size_t kv_index(const orc_config* c, int l, int kv, int kvh, int64_t t, int d) {
  return ((((size_t)l * 2 + kv) * c->n_kv_heads + kvh) * (size_t)c->max_ctx + (size_t)t) * c->head_dim + d;
}

uint16_t orc_kv_get(const orc_model* m, int layer, int kv, int kv_head, int t, int d) {
  return m->kv[kv_index(&m->c, layer, kv, kv_head, t, d)];
}

/* prefill: N(0,1) draws rounded to binary16, element (t, kv_head, d) of layer l
 * takes counter index (t * n_kv_heads + kv_head) * head_dim + d; stored as
 * already-rotated keys (no RoPE applied). */
int orc_kv_prefill(orc_model* m, int32_t n_ctx, uint64_t seed) {
  const orc_config* c = &m->c;
  if (n_ctx < 0 || n_ctx > c->max_ctx) return -1;
  for (int l = 0; l < c->n_layers; l++)
    for (int kv = 0; kv < 2; kv++)
      for (int64_t t = 0; t < n_ctx; t++)
        for (int g = 0; g < c->n_kv_heads; g++)
          for (int d = 0; d < c->head_dim; d++) {
            uint64_t i = ((uint64_t)t * c->n_kv_heads + g) * c->head_dim + d;
            float z = orc_normal(seed, ORC_UID_KV(l, kv), i) * 1.0f;
            m->kv[kv_index(c, l, kv, g, t, d)] = orc_f16_from_double((double)z);
          }
  m->pos = n_ctx;
  return 0;
}

static int gemv_role(orc_model* m, int l, int role, const double* x, double* y) {
  int64_t rows, cols;
  int qt;
  role_shape(&m->c, role, &rows, &cols, &qt);
  uint8_t* w = m->layer[l * 7 + role];
  int owned = 0;
  if (!w) { w = gen_layer_tensor(&m->c, l, role); owned = 1; }
  if (!w) return -2;
  int rc = orc_gemv_d(qt, w, rows, cols, x, y, m->c.nthreads);
  if (owned) free(w);
  return rc;
}

/* One decode step: embedding -> n_layers x (RMSNorm, Q/K/V, RoPE, KV store,
 * GQA attention, O + residual, RMSNorm, gate/up, SwiGLU, down + residual) ->
 * RMSNorm -> output projection -> greedy argmax.  All activations in double;
 * weights are the fp32 dequantized values; K/V are rounded to binary16 when
 * stored and the current position is stored before it is attended to. */
int orc_decode_step(orc_model* m, int32_t token, double* logits, int32_t* next, double* margin) {
  const orc_config* c = &m->c;
  if (token < 0 || token >= c->vocab || m->pos >= c->max_ctx) return -1;
  int64_t h = c->hidden, hd = c->head_dim, nq = c->n_heads, nkv = c->n_kv_heads, f = c->ffn_dim;
  int64_t qd = nq * hd, kd = nkv * hd;
  int64_t pos = m->pos;
  double *x = (double*)malloc(sizeof(double) * h), *xn = (double*)malloc(sizeof(double) * h);
  double *q = (double*)malloc(sizeof(double) * qd), *k = (double*)malloc(sizeof(double) * kd);
  double *v = (double*)malloc(sizeof(double) * kd), *o = (double*)malloc(sizeof(double) * qd);
  double *t = (double*)malloc(sizeof(double) * (h > f ? h : f));
  double *g = (double*)malloc(sizeof(double) * f), *u = (double*)malloc(sizeof(double) * f);
  double *lg = (double*)malloc(sizeof(double) * c->vocab);
  double *x_in = (double*)malloc(sizeof(double) * h);
  float* row = (float*)malloc(sizeof(float) * h);
  uint16_t *kc = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(pos + 1) * hd);
  uint16_t *vc = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(pos + 1) * hd);
  uint8_t* er = (uint8_t*)malloc((size_t)row_bytes(c->t_embd, h));
  int rc = 0;
  if (!x || !xn || !q || !k || !v || !o || !t || !g || !u || !lg || !x_in || !row || !kc || !vc || !er) { rc = -2; goto done; }

  /* embedding row */
  if (m->embd) memcpy(er, m->embd + (int64_t)token * row_bytes(c->t_embd, h), (size_t)row_bytes(c->t_embd, h));
  else if (orc_qtensor_rows(c->t_embd, c->vocab, h, c->seed, ORC_UID_EMBD, c->init_std, token, 1, er, 1)) { rc = -2; goto done; }
  orc_dequant_row(c->t_embd, er, h, row);
  for (int64_t i = 0; i < h; i++) x[i] = (double)row[i];

  for (int l = 0; l < c->n_layers; l++) {
    if (m->skip && m->skip[l]) {
      m->layer_cos[l] = 1.0;
      continue;
    }
    memcpy(x_in, x, sizeof(double) * h);
    orc_rmsnorm(x, h, c->rms_eps, xn);
    if ((rc = gemv_role(m, l, ORC_ROLE_Q, xn, q))) goto done;
    if ((rc = gemv_role(m, l, ORC_ROLE_K, xn, k))) goto done;
    if ((rc = gemv_role(m, l, ORC_ROLE_V, xn, v))) goto done;
    orc_rope(q, (int)nq, (int)hd, pos, c->rope_theta);
    orc_rope(k, (int)nkv, (int)hd, pos, c->rope_theta);
    for (int gh = 0; gh < nkv; gh++)
      for (int d = 0; d < hd; d++) {
        m->kv[kv_index(c, l, 0, gh, pos, d)] = orc_f16_from_double(k[gh * hd + d]);
        m->kv[kv_index(c, l, 1, gh, pos, d)] = orc_f16_from_double(v[gh * hd + d]);
      }
    int64_t group = nq / nkv;
    for (int j = 0; j < nq; j++) {
      int gh = (int)(j / group);
      for (int64_t tt = 0; tt <= pos; tt++)
        for (int d = 0; d < hd; d++) {
          kc[tt * hd + d] = m->kv[kv_index(c, l, 0, gh, tt, d)];
          vc[tt * hd + d] = m->kv[kv_index(c, l, 1, gh, tt, d)];
        }
      orc_attend(q + j * hd, kc, vc, pos + 1, (int)hd, o + j * hd);
    }
    if ((rc = gemv_role(m, l, ORC_ROLE_O, o, t))) goto done;
    for (int64_t i = 0; i < h; i++) x[i] += t[i];
    orc_rmsnorm(x, h, c->rms_eps, xn);
    if ((rc = gemv_role(m, l, ORC_ROLE_GATE, xn, g))) goto done;
    if ((rc = gemv_role(m, l, ORC_ROLE_UP, xn, u))) goto done;
    for (int64_t i = 0; i < f; i++) u[i] = orc_silu(g[i]) * u[i];
    if ((rc = gemv_role(m, l, ORC_ROLE_DOWN, u, t))) goto done;
    for (int64_t i = 0; i < h; i++) x[i] += t[i];
    m->layer_cos[l] = orc_cosine(x_in, x, h);
  }
  memcpy(m->hidden, x, sizeof(double) * h);
  orc_rmsnorm(x, h, c->rms_eps, xn);
  {
    uint8_t* w = m->output;
    int owned = 0;
    if (!w) { w = gen_tensor(c, c->t_out, c->vocab, h, ORC_UID_OUTPUT); owned = 1; }
    if (!w) { rc = -2; goto done; }
    rc = orc_gemv_d(c->t_out, w, c->vocab, h, xn, lg, c->nthreads);
    if (owned) free(w);
    if (rc) goto done;
  }
  {
    double mg;
    int64_t nx = orc_argmax(lg, c->vocab, &mg);
    if (next) *next = (int32_t)nx;
    if (margin) *margin = mg;
    if (logits) memcpy(logits, lg, sizeof(double) * c->vocab);
  }
  m->pos = (int32_t)(pos + 1);
done:
  free(x); free(x_in); free(xn); free(q); free(k); free(v); free(o); free(t); free(g); free(u); free(lg);
  free(row); free(kc); free(vc); free(er);
  return rc;
}
