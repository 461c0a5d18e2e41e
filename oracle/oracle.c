/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the mixed-batch
 * attention step over a block-quantised KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg (and its
 * `--impl reference` arm) load it.  It shares no code, header, table or helper
 * with the CUDA library; it does its own fp16 conversion and its own rounding.
 *
 * Sources (page titles and sections of the reference pages):
 *  - "自研RDNA高併發推論引擎 以AI Max+ 395為範例" (lcz.me topic 2938), §2 modes
 *    table: q8 = blocked 8-bit, one f16 scale per 32 elements, 34 bytes per
 *    block; the 4-bit K/V modes pack a 32-element block into 18 bytes.  §2
 *    occupancy table: bytes per KV position 2048 / 1088 / 832 / 576.
 *  - same page, §1 "統一 mixed-batch 介面": chunk rows and decode rows share
 *    one ForwardBatch and one attention kernel.
 *  - The block formulas are the GGUF Q8_0 / Q4_0 conventions of the model
 *    files the same page says the engine reads: Q8_0 d = amax/127, q = round(x/d);
 *    Q4_0 d = (signed max)/-8, q = min(15, trunc(x/d + 8.5)), x^ = (q-8)*d.
 *
 * Readings where the pages leave a step open:
 *  - blocks run along head_dim, per (token, kv head);
 *  - q is computed as x * id with id = 1/d in fp32 (d in fp32); only the stored
 *    scale is rounded to fp16 (round-to-nearest-even);
 *  - "round" is round-half-away-from-zero (C roundf);
 *  - the Q4_0 product x*id and the sum +8.5 are each rounded to fp32 (no fused
 *    multiply-add; this file must be compiled with -ffp-contract=off);
 *  - Q4_0 signed max: the element of largest magnitude, lowest index on ties;
 *  - d == 0 gives id = 0 (all q = 0 for Q8_0, all q = 8 for Q4_0);
 *  - Q4_0 nibbles: byte k holds element k (low nibble) and element k+16 (high);
 *  - attention: s_j = (q . k^_j) / sqrt(D), softmax over keys 0..p (causal),
 *    kv head of q head h is h / (Hq/Hkv); all in fp64 over the dequantised KV.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_FMT_F16 0
#define ORC_FMT_Q8_0 1
#define ORC_FMT_Q4_0 2
#define ORC_QK 32 /* elements per block */

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the format definitions.          */
/* ------------------------------------------------------------------------ */

/* Round a binary32 value to binary16, round-to-nearest, ties-to-even. */
static uint16_t orc_f32_to_f16(float f) {
  uint32_t x;
  memcpy(&x, &f, sizeof x);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t mag = x & 0x7FFFFFFFu;
  if (mag >= 0x7F800000u) { /* inf or nan */
    return (uint16_t)(sign | 0x7C00u | (mag > 0x7F800000u ? 0x0200u : 0u));
  }
  if (mag >= 0x477FF000u) { /* >= 65520: rounds to infinity */
    return (uint16_t)(sign | 0x7C00u);
  }
  uint32_t e32 = mag >> 23;
  uint32_t man = mag & 0x7FFFFFu;
  if (e32 < 113u) {
    /* Below 2^-14: the result is a binary16 subnormal (unit 2^-24) or zero.
     * value = sig * 2^(e - 150) with e = max(e32, 1); in units of 2^-24 that
     * is sig >> (126 - e), rounded to nearest even. */
    uint32_t sig = (e32 == 0u) ? man : (man | 0x800000u);
    uint32_t e = (e32 == 0u) ? 1u : e32;
    uint32_t sh = 126u - e; /* >= 14 */
    if (sh > 31u) return (uint16_t)sign;
    uint32_t q = sig >> sh;
    uint32_t rem = sig & ((1u << sh) - 1u);
    uint32_t half = 1u << (sh - 1u);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q); /* q == 0x400 encodes the smallest normal */
  }
  /* Normal binary16 range: rebias the exponent, keep 10 mantissa bits. */
  uint32_t q = ((e32 - 112u) << 10) | (man >> 13);
  uint32_t rem = man & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q += 1u;
  return (uint16_t)(sign | q);
}

static float orc_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  float v;
  if (e == 0) {
    v = ldexpf((float)m, -24);
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexpf((float)(1024 + m), e - 25);
  }
  return sign ? -v : v;
}

void orc_f32_to_f16_array(const float* x, uint16_t* h, int64_t n) {
  for (int64_t i = 0; i < n; ++i) h[i] = orc_f32_to_f16(x[i]);
}

void orc_f16_to_f32_array(const uint16_t* h, float* x, int64_t n) {
  for (int64_t i = 0; i < n; ++i) x[i] = orc_f16_to_f32(h[i]);
}

/* ------------------------------------------------------------------------ */
/* Block codecs.  A canonical block is the byte string the pages size:      */
/*   Q8_0: fp16 d (little endian) + 32 int8 q            = 34 bytes          */
/*   Q4_0: fp16 d (little endian) + 16 bytes of nibbles  = 18 bytes          */
/*   F16 : 32 fp16 values                                = 64 bytes          */
/* ------------------------------------------------------------------------ */

int orc_block_bytes(int fmt) {
  switch (fmt) {
    case ORC_FMT_F16: return 2 * ORC_QK;
    case ORC_FMT_Q8_0: return 2 + ORC_QK;
    case ORC_FMT_Q4_0: return 2 + ORC_QK / 2;
    default: return -1;
  }
}

static void put_u16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xFFu);
  p[1] = (uint8_t)(v >> 8);
}

static uint16_t get_u16(const uint8_t* p) {
  return (uint16_t)(p[0] | ((uint16_t)p[1] << 8));
}

/* Q8_0: d = amax / 127, q_j = round(x_j / d) with round-half-away. */
static void q8_0_quantize(const float* x, uint8_t* blk) {
  float amax = 0.0f;
  for (int j = 0; j < ORC_QK; ++j) {
    float a = fabsf(x[j]);
    if (a > amax) amax = a;
  }
  float d = amax / 127.0f;
  float id = (d != 0.0f) ? 1.0f / d : 0.0f;
  put_u16(blk, orc_f32_to_f16(d));
  for (int j = 0; j < ORC_QK; ++j) {
    float v = x[j] * id;
    int q = (int)roundf(v);
    blk[2 + j] = (uint8_t)(int8_t)q;
  }
}

/* Q4_0: m = signed value of largest magnitude (first on ties), d = m / -8,
 * q_j = min(15, trunc(x_j / d + 8.5)); element k and k+16 share byte k. */
static void q4_0_quantize(const float* x, uint8_t* blk) {
  float amax = 0.0f, m = 0.0f;
  for (int j = 0; j < ORC_QK; ++j) {
    float a = fabsf(x[j]);
    if (a > amax) {
      amax = a;
      m = x[j];
    }
  }
  float d = m / -8.0f;
  float id = (d != 0.0f) ? 1.0f / d : 0.0f;
  put_u16(blk, orc_f32_to_f16(d));
  for (int k = 0; k < ORC_QK / 2; ++k) {
    float p0 = x[k] * id;
    float p1 = x[k + ORC_QK / 2] * id;
    float s0 = p0 + 8.5f;
    float s1 = p1 + 8.5f;
    int q0 = (int)truncf(s0);
    int q1 = (int)truncf(s1);
    if (q0 > 15) q0 = 15;
    if (q1 > 15) q1 = 15;
    blk[2 + k] = (uint8_t)((unsigned)q0 | ((unsigned)q1 << 4));
  }
}

static void f16_store(const float* x, uint8_t* blk) {
  for (int j = 0; j < ORC_QK; ++j) put_u16(blk + 2 * j, orc_f32_to_f16(x[j]));
}

/* Quantise n_blocks consecutive 32-element blocks of fp16 input. */
int orc_quantize(int fmt, const uint16_t* x_f16, int64_t n_blocks, uint8_t* out) {
  int bb = orc_block_bytes(fmt);
  if (bb < 0) return -1;
  for (int64_t b = 0; b < n_blocks; ++b) {
    float x[ORC_QK];
    for (int j = 0; j < ORC_QK; ++j) x[j] = orc_f16_to_f32(x_f16[b * ORC_QK + j]);
    uint8_t* blk = out + b * bb;
    if (fmt == ORC_FMT_Q8_0) q8_0_quantize(x, blk);
    else if (fmt == ORC_FMT_Q4_0) q4_0_quantize(x, blk);
    else f16_store(x, blk);
  }
  return 0;
}

/* Dequantise one block into 32 doubles (exact: d_h * q has <= 18 bits). */
static void dequant_block(int fmt, const uint8_t* blk, double* y) {
  if (fmt == ORC_FMT_F16) {
    for (int j = 0; j < ORC_QK; ++j) y[j] = (double)orc_f16_to_f32(get_u16(blk + 2 * j));
  } else if (fmt == ORC_FMT_Q8_0) {
    double d = (double)orc_f16_to_f32(get_u16(blk));
    for (int j = 0; j < ORC_QK; ++j) y[j] = d * (double)(int8_t)blk[2 + j];
  } else {
    double d = (double)orc_f16_to_f32(get_u16(blk));
    for (int k = 0; k < ORC_QK / 2; ++k) {
      int lo = blk[2 + k] & 0x0F;
      int hi = blk[2 + k] >> 4;
      y[k] = d * (double)(lo - 8);
      y[k + ORC_QK / 2] = d * (double)(hi - 8);
    }
  }
}

int orc_dequantize(int fmt, const uint8_t* blocks, int64_t n_blocks, double* out) {
  int bb = orc_block_bytes(fmt);
  if (bb < 0) return -1;
  for (int64_t b = 0; b < n_blocks; ++b) dequant_block(fmt, blocks + b * bb, out + b * ORC_QK);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Attention over the dequantised cache, fp64.                               */
/*                                                                            */
/* Row r has seq_len[r] keys (its whole history, in logical token order) and */
/* n_q[r] = seq_len[r] - q_offset[r] queries at positions q_offset[r] + i.   */
/* A decode row is the case n_q = 1.  Queries are packed row after row:      */
/* q_f16[(q_start[r] + i) * Hq * D + h * D + d].  The row's K (V) blocks are */
/* k_blocks + k_off[r] bytes, laid out [seq_len][Hkv][D/32] canonical blocks.*/
/*                                                                            */
/* sel lists packed query-token indices to evaluate (n_sel of them); out is  */
/* [n_sel][Hq][D].  Queries not listed are skipped (sampled parity at size). */
/* ------------------------------------------------------------------------ */

static int find_row(int n_rows, const int32_t* q_start, const int32_t* n_q, int32_t t) {
  for (int r = 0; r < n_rows; ++r)
    if (t >= q_start[r] && t < q_start[r] + n_q[r]) return r;
  return -1;
}

/* window > 0: sliding-window attention -- the query at position p sees only */
/* the `window` most recent keys, p - window + 1 .. p (the page's per-model   */
/* table, Gemma 4 row: its SWA layers read the same Q8 cache).  window <= 0:  */
/* every key 0 .. p.                                                          */
int orc_attention_window(int fmt_k, int fmt_v, int D, int Hq, int Hkv, int n_rows,
                         const int32_t* seq_len, const int32_t* q_offset,
                         const uint16_t* q_f16, const uint8_t* k_blocks, const int64_t* k_off,
                         const uint8_t* v_blocks, const int64_t* v_off, int n_sel,
                         const int32_t* sel, double* out, int n_threads, int window) {
  if (D % ORC_QK != 0 || Hkv <= 0 || Hq % Hkv != 0) return -1;
  int bbk = orc_block_bytes(fmt_k), bbv = orc_block_bytes(fmt_v);
  if (bbk < 0 || bbv < 0) return -1;
  int32_t* q_start = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_rows + 1));
  int32_t* n_q = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_rows + 1));
  int32_t acc = 0;
  for (int r = 0; r < n_rows; ++r) {
    q_start[r] = acc;
    n_q[r] = seq_len[r] - q_offset[r];
    acc += n_q[r];
  }
  const int G = Hq / Hkv;
  const int nb = D / ORC_QK;
  const double scale = 1.0 / sqrt((double)D);
  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t job = 0; job < (int64_t)n_sel * Hq; ++job) {
    int si = (int)(job / Hq);
    int h = (int)(job % Hq);
    int32_t t = sel[si];
    int r = find_row(n_rows, q_start, n_q, t);
    if (r < 0) {
      status = -2;
      continue;
    }
    int g = h / G;
    int p = q_offset[r] + (t - q_start[r]); /* position of this query */
    int nkeys = p + 1;                     /* causal: keys 0..p */
    int first = (window > 0 && p + 1 > window) ? p + 1 - window : 0; /* sliding window */
    double q[512], kh[512], vh[512];
    for (int d = 0; d < D; ++d) q[d] = (double)orc_f16_to_f32(q_f16[((int64_t)t * Hq + h) * D + d]);
    double* s = (double*)malloc(sizeof(double) * (size_t)nkeys);
    double smax = -INFINITY;
    for (int j = first; j < nkeys; ++j) {
      const uint8_t* kb = k_blocks + k_off[r] + (((int64_t)j * Hkv + g) * nb) * bbk;
      for (int b = 0; b < nb; ++b) dequant_block(fmt_k, kb + b * bbk, kh + b * ORC_QK);
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += q[d] * kh[d];
      s[j] = dot * scale;
      if (s[j] > smax) smax = s[j];
    }
    double denom = 0.0;
    double o[512];
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int j = first; j < nkeys; ++j) {
      double w = exp(s[j] - smax);
      denom += w;
      const uint8_t* vb = v_blocks + v_off[r] + (((int64_t)j * Hkv + g) * nb) * bbv;
      for (int b = 0; b < nb; ++b) dequant_block(fmt_v, vb + b * bbv, vh + b * ORC_QK);
      for (int d = 0; d < D; ++d) o[d] += w * vh[d];
    }
    double* dst = out + ((int64_t)si * Hq + h) * D;
    for (int d = 0; d < D; ++d) dst[d] = o[d] / denom;
    free(s);
  }
  free(q_start);
  free(n_q);
  return status;
}

int orc_attention(int fmt_k, int fmt_v, int D, int Hq, int Hkv, int n_rows,
                  const int32_t* seq_len, const int32_t* q_offset,
                  const uint16_t* q_f16, const uint8_t* k_blocks, const int64_t* k_off,
                  const uint8_t* v_blocks, const int64_t* v_off, int n_sel,
                  const int32_t* sel, double* out, int n_threads) {
  return orc_attention_window(fmt_k, fmt_v, D, Hq, Hkv, n_rows, seq_len, q_offset, q_f16, k_blocks, k_off,
                              v_blocks, v_off, n_sel, sel, out, n_threads, 0);
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
