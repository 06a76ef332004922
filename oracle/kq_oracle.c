/*
 * kq_oracle.c -- TEST INFRASTRUCTURE ONLY.  The plain, slow, obviously
 * correct CPU reference that the GPU library is checked against.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header or table with the library.
 *
 * Everything is single-threaded and computed in fp64 (IEEE double, no FMA
 * contraction: build with -ffp-contract=off).
 *
 * What is computed (sources):
 *  - The formats: GGUF K-quant super-blocks Q4_K / Q5_K / Q6_K, which the
 *    daily.dev summary "Fast on-device agentic AI with Muse Glimmer on
 *    ExecuTorch" names as the CUDA GEMV input (answer on exporting GGUF
 *    checkpoints).  The field geometry is the public GGUF one: Q4_K = 8
 *    sub-blocks of 32 with 6-bit scale and min and fp16 d/dmin; Q5_K adds a
 *    fifth bit; Q6_K = 16 sub-blocks of 16 with int8 scales and fp16 d.
 *    The byte placement is written out in the header comment of kq.h and
 *    repeated, in this file's own words, at each decoder below.
 *  - The group-128 merged layout: the same page says adjacent sub-blocks with
 *    identical scale/min are merged into groups of up to 128 when lossless;
 *    the SGLang day-0 post names a Q4_K_M checkpoint with 128-weight groups.
 *    Reading taken: one (sc, m) per 128 weights, planar storage.
 *  - The product: y[t][n] = sum_k w^[n][k] x[t][k], in k order, in fp64,
 *    with bf16 x widened exactly, and A[t][n] = sum_k |w^[n][k] x[t][k]|,
 *    which sets the tolerance |y - y_ref| <= 1e-3 A + 1e-5.
 *  - The quantiser (test data only; the pages do not define one): q rounded
 *    to nearest-even, d and dmin rounded UP to fp16 so the grid of every
 *    sub-block covers its weights, giving |w - w^| <= step/2.
 *
 * Parity pins live in tests/test_oracle_*.py.  GGUF bit-placement
 * compatibility with real checkpoint files is parity unpinned (no GGUF file
 * is available to compare with).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define KQO_Q4_K 0
#define KQO_Q5_K 1
#define KQO_Q6_K 2
#define KQO_Q4_G128 3

#define KQO_OK 0
#define KQO_BAD_ARG 1
#define KQO_BAD_SHAPE 2
#define KQO_NOT_MERGEABLE 4
#define KQO_RANGE 5

/* ---------------- scalar conversions (IEEE definitions) ---------------- */

/* binary16 -> double: sign, 5-bit biased exponent (bias 15), 10-bit
 * fraction; exponent 0 is subnormal (fraction * 2^-24). */
double kqo_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int f = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);
  } else if (e == 31) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + f), e - 25);
  }
  return sign ? -v : v;
}

/* bfloat16 -> double: the upper 16 bits of an IEEE binary32. */
double kqo_bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Smallest binary16 value >= v, for finite v >= 0, returned as a double;
 * *bits receives its encoding.  Returns 0 if the value would exceed the
 * largest finite binary16 (65504). */
int kqo_half_round_up(double v, double* val, uint16_t* bits) {
  if (!(v >= 0.0)) return 0;
  if (v == 0.0) { *val = 0.0; *bits = 0; return 1; }
  double r;
  if (v < ldexp(1.0, -14)) {
    /* subnormal grid: multiples of 2^-24 */
    r = ldexp(ceil(ldexp(v, 24)), -24);
  } else {
    int E;
    (void)frexp(v, &E);              /* v = f * 2^E, f in [0.5, 1) */
    int e = E - 1;                   /* v in [2^e, 2^(e+1))        */
    r = ldexp(ceil(ldexp(v, 10 - e)), e - 10);  /* 11-bit significand */
  }
  if (r > 65504.0) return 0;
  /* encode r */
  if (r < ldexp(1.0, -14)) {
    *bits = (uint16_t)ldexp(r, 24);
  } else {
    int E;
    double f = frexp(r, &E);         /* r = f * 2^E */
    int e = E - 1;
    uint16_t frac = (uint16_t)(ldexp(f, 11) - 1024.0);
    *bits = (uint16_t)(((e + 15) << 10) | frac);
  }
  *val = r;
  return 1;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 255); p[1] = (uint8_t)(v >> 8); }

/* ---------------------------- sizes ------------------------------------ */

int kqo_block_bytes(int fmt) {
  switch (fmt) {
    case KQO_Q4_K: return 144;
    case KQO_Q5_K: return 176;
    case KQO_Q6_K: return 210;
    case KQO_Q4_G128: return 136;
    default: return 0;
  }
}

/* ------------------------------ decoders -------------------------------- */

/* The 12-byte scale field of Q4_K/Q5_K holds eight 6-bit scales and eight
 * 6-bit mins.  Sub-blocks 0..3 keep theirs in the low six bits of bytes
 * 0..3 (scale) and 4..7 (min).  Sub-blocks 4..7 keep the low four bits of
 * the scale in the low nibble of byte 8+(j-4), the low four bits of the min
 * in its high nibble, and the top two bits of each in the top two bits of
 * bytes j-4 (scale) and j (min). */
static void kqo_scale_min(const uint8_t* s12, int j, int* sc, int* m) {
  if (j < 4) {
    *sc = s12[j] & 63;
    *m = s12[j + 4] & 63;
  } else {
    int lo = s12[j + 4];
    *sc = (lo & 15) | ((s12[j - 4] >> 6) << 4);
    *m = (lo >> 4) | ((s12[j] >> 6) << 4);
  }
}

/* Q4_K: qs[128] covers four 64-weight chunks.  In chunk c, byte r (0..31)
 * carries weight 64c+r in its low nibble (sub-block 2c) and weight 64c+32+r
 * in its high nibble (sub-block 2c+1). */
static void kqo_dequant_q4k(const uint8_t* b, double* out) {
  double d = kqo_half_to_double(rd16(b));
  double dmin = kqo_half_to_double(rd16(b + 2));
  const uint8_t* s12 = b + 4;
  const uint8_t* qs = b + 16;
  for (int i = 0; i < 256; i++) {
    int c = i / 64, r = i % 64;
    int q, j;
    if (r < 32) { q = qs[32 * c + r] & 15; j = 2 * c; }
    else        { q = qs[32 * c + r - 32] >> 4; j = 2 * c + 1; }
    int sc, m;
    kqo_scale_min(s12, j, &sc, &m);
    out[i] = d * sc * q - dmin * m;
  }
}

/* Q5_K: as Q4_K for the low four bits (qs at byte 48); the fifth bit of
 * weight 64c+r comes from qh[r % 32], bit 2c for r < 32 and bit 2c+1 for
 * r >= 32. */
static void kqo_dequant_q5k(const uint8_t* b, double* out) {
  double d = kqo_half_to_double(rd16(b));
  double dmin = kqo_half_to_double(rd16(b + 2));
  const uint8_t* s12 = b + 4;
  const uint8_t* qh = b + 16;
  const uint8_t* qs = b + 48;
  for (int i = 0; i < 256; i++) {
    int c = i / 64, r = i % 64, l = r % 32;
    int hi = r >= 32;
    int nib = hi ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 15);
    int bit = (qh[l] >> (2 * c + hi)) & 1;
    int q = nib | (bit << 4);
    int sc, m;
    kqo_scale_min(s12, 2 * c + hi, &sc, &m);
    out[i] = d * sc * q - dmin * m;
  }
}

/* Q6_K: two halves of 128 weights.  In half h, weight 128h + 32t + l
 * (t = 0..3, l = 0..31) takes its low four bits from ql[64h + l + 32*(t&1)]
 * (low nibble for t = 0,1, high nibble for t = 2,3) and its top two bits from
 * bits 2t, 2t+1 of qh[32h + l].  Sub-block i/16 has an int8 scale. */
static void kqo_dequant_q6k(const uint8_t* b, double* out) {
  const uint8_t* ql = b;
  const uint8_t* qh = b + 128;
  const int8_t* sc = (const int8_t*)(b + 192);
  double d = kqo_half_to_double(rd16(b + 208));
  for (int i = 0; i < 256; i++) {
    int h = i / 128, t = (i % 128) / 32, l = i % 32;
    uint8_t lb = ql[64 * h + l + 32 * (t & 1)];
    int nib = (t < 2) ? (lb & 15) : (lb >> 4);
    int hb = (qh[32 * h + l] >> (2 * t)) & 3;
    int q = nib | (hb << 4);
    out[i] = d * sc[i / 16] * (q - 32);
  }
}

/* Q4_G128: q as Q4_K's qs (128 bytes), params in
 * the 8-byte record {d fp16, dmin fp16, sc0, sc1, m0, m1}; weight i uses
 * group i/128. */
static void kqo_dequant_g128(const uint8_t* qs, const uint8_t* p, double* out) {
  double d = kqo_half_to_double(rd16(p));
  double dmin = kqo_half_to_double(rd16(p + 2));
  for (int i = 0; i < 256; i++) {
    int c = i / 64, r = i % 64;
    int q = (r < 32) ? (qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4);
    int g = i / 128;
    out[i] = d * p[4 + g] * q - dmin * p[6 + g];
  }
}

/* Pointers to super-block (n, b) of an N x K matrix in format fmt. */
static void kqo_locate(int fmt, const uint8_t* W, int64_t N, int64_t K,
                       int64_t n, int64_t b, const uint8_t** blk,
                       const uint8_t** par) {
  int64_t nsb = K / 256;
  int64_t idx = n * nsb + b;
  if (fmt == KQO_Q4_G128) {
    *blk = W + idx * 128;
    *par = W + N * nsb * 128 + idx * 8;
  } else {
    *blk = W + idx * kqo_block_bytes(fmt);
    *par = 0;
  }
}

static void kqo_dequant_sb(int fmt, const uint8_t* blk, const uint8_t* par,
                           double* out) {
  switch (fmt) {
    case KQO_Q4_K: kqo_dequant_q4k(blk, out); break;
    case KQO_Q5_K: kqo_dequant_q5k(blk, out); break;
    case KQO_Q6_K: kqo_dequant_q6k(blk, out); break;
    default: kqo_dequant_g128(blk, par, out); break;
  }
}

static int kqo_check(int fmt, int64_t N, int64_t K) {
  if (kqo_block_bytes(fmt) == 0) return KQO_BAD_ARG;
  if (N <= 0 || K <= 0 || K % 256 != 0) return KQO_BAD_SHAPE;
  return KQO_OK;
}

/* out[n][k] = w^[n][k] in fp64, row-major N x K. */
int kqo_dequantize(int fmt, const uint8_t* W, int64_t N, int64_t K,
                   double* out) {
  int st = kqo_check(fmt, N, K);
  if (st) return st;
  int64_t nsb = K / 256;
  for (int64_t n = 0; n < N; n++)
    for (int64_t b = 0; b < nsb; b++) {
      const uint8_t *blk, *par;
      kqo_locate(fmt, W, N, K, n, b, &blk, &par);
      kqo_dequant_sb(fmt, blk, par, out + n * K + b * 256);
    }
  return KQO_OK;
}

/* For each listed row n = rows[r] (r < nrows) and each token t < n_tok:
 *   y[t*nrows + r] = sum_k w^[n][k] * x[t][k]      (k ascending, fp64)
 *   A[t*nrows + r] = sum_k |w^[n][k] * x[t][k]|
 * x is bf16 [n_tok][K].  W is the whole N x K matrix.  A may be NULL. */
int kqo_gemv_rows(int fmt, const uint8_t* W, int64_t N, int64_t K,
                  const int64_t* rows, int64_t nrows, const uint16_t* x,
                  int n_tok, double* y, double* A) {
  int st = kqo_check(fmt, N, K);
  if (st) return st;
  if (n_tok < 1) return KQO_BAD_ARG;
  int64_t nsb = K / 256;
  double w[256];
  for (int64_t r = 0; r < nrows; r++) {
    int64_t n = rows[r];
    if (n < 0 || n >= N) return KQO_BAD_ARG;
    for (int t = 0; t < n_tok; t++) {
      y[t * nrows + r] = 0.0;
      if (A) A[t * nrows + r] = 0.0;
    }
    for (int64_t b = 0; b < nsb; b++) {
      const uint8_t *blk, *par;
      kqo_locate(fmt, W, N, K, n, b, &blk, &par);
      kqo_dequant_sb(fmt, blk, par, w);
      for (int t = 0; t < n_tok; t++) {
        const uint16_t* xt = x + (int64_t)t * K + b * 256;
        double acc = y[t * nrows + r];
        double aa = A ? A[t * nrows + r] : 0.0;
        for (int i = 0; i < 256; i++) {
          double p = w[i] * kqo_bf16_to_double(xt[i]);
          acc += p;
          aa += fabs(p);
        }
        y[t * nrows + r] = acc;
        if (A) A[t * nrows + r] = aa;
      }
    }
  }
  return KQO_OK;
}

/* All rows: y[t][n], A[t][n]. */
int kqo_gemv(int fmt, const uint8_t* W, int64_t N, int64_t K,
             const uint16_t* x, int n_tok, double* y, double* A) {
  int st = kqo_check(fmt, N, K);
  if (st) return st;
  /* rows 0..N-1 in order: the row list is the identity. */
  int64_t nsb = K / 256;
  double w[256];
  for (int64_t n = 0; n < N; n++) {
    for (int t = 0; t < n_tok; t++) {
      y[t * N + n] = 0.0;
      if (A) A[t * N + n] = 0.0;
    }
    for (int64_t b = 0; b < nsb; b++) {
      const uint8_t *blk, *par;
      kqo_locate(fmt, W, N, K, n, b, &blk, &par);
      kqo_dequant_sb(fmt, blk, par, w);
      for (int t = 0; t < n_tok; t++) {
        const uint16_t* xt = x + (int64_t)t * K + b * 256;
        for (int i = 0; i < 256; i++) {
          double p = w[i] * kqo_bf16_to_double(xt[i]);
          y[t * N + n] += p;
          if (A) A[t * N + n] += fabs(p);
        }
      }
    }
  }
  return KQO_OK;
}

/* ------------------------------ quantiser ------------------------------- */

/* Asymmetric quantiser with L+1 levels over sub-blocks of `gs` weights of
 * one 256-weight super-block (gs = 32 for Q4_K/Q5_K, 128 for the group-128
 * statistics).  Outputs per-weight q, per-group sc/m, and the fp16 d/dmin. */
static int kqo_quant_asym(const float* w, int gs, int L, int* q, int* sc,
                          int* m, uint16_t* d_bits, uint16_t* dmin_bits) {
  int ng = 256 / gs;
  double mn[8], mx[8], r[8];
  double max_mn = 0.0;
  for (int g = 0; g < ng; g++) {
    double lo = w[g * gs], hi = w[g * gs];
    for (int i = 1; i < gs; i++) {
      double v = w[g * gs + i];
      if (v < lo) lo = v;
      if (v > hi) hi = v;
    }
    mn[g] = (-lo > 0.0) ? -lo : 0.0;
    mx[g] = hi;
    if (mn[g] > max_mn) max_mn = mn[g];
  }
  double dmin;
  if (!kqo_half_round_up(max_mn / 63.0, &dmin, dmin_bits)) return KQO_RANGE;
  double max_r = 0.0;
  for (int g = 0; g < ng; g++) {
    int mg = 0;
    if (dmin > 0.0) {
      double t = ceil(mn[g] / dmin);
      mg = (t > 63.0) ? 63 : (int)t;
    }
    m[g] = mg;
    r[g] = (mx[g] + dmin * mg) / L;
    if (r[g] > max_r) max_r = r[g];
  }
  double d;
  if (!kqo_half_round_up(max_r / 63.0, &d, d_bits)) return KQO_RANGE;
  for (int g = 0; g < ng; g++) {
    int s = 0;
    if (d > 0.0) {
      double t = ceil(r[g] / d);
      s = (t > 63.0) ? 63 : (t < 0.0 ? 0 : (int)t);
    }
    sc[g] = s;
    double step = d * s;
    for (int i = 0; i < gs; i++) {
      int qi = 0;
      if (step > 0.0) {
        double t = nearbyint(((double)w[g * gs + i] + dmin * m[g]) / step);
        qi = (t < 0.0) ? 0 : (t > L ? L : (int)t);
      }
      q[g * gs + i] = qi;
    }
  }
  return KQO_OK;
}

/* Pack eight 6-bit (sc, m) pairs into the 12-byte field (inverse of
 * kqo_scale_min). */
static void kqo_pack_scales(const int* sc, const int* m, uint8_t* s12) {
  memset(s12, 0, 12);
  for (int j = 0; j < 4; j++) {
    s12[j] = (uint8_t)(sc[j] & 63);
    s12[j + 4] = (uint8_t)(m[j] & 63);
  }
  for (int j = 4; j < 8; j++) {
    s12[j + 4] = (uint8_t)((sc[j] & 15) | ((m[j] & 15) << 4));
    s12[j - 4] |= (uint8_t)((sc[j] >> 4) << 6);
    s12[j] |= (uint8_t)((m[j] >> 4) << 6);
  }
}

/* Pack 256 nibbles into Q4_K's 128-byte qs. */
static void kqo_pack_nibbles(const int* q, uint8_t* qs) {
  for (int c = 0; c < 4; c++)
    for (int r = 0; r < 32; r++)
      qs[32 * c + r] = (uint8_t)((q[64 * c + r] & 15) | ((q[64 * c + 32 + r] & 15) << 4));
}

static int kqo_quant_sb_q4k(const float* w, int group, uint8_t* out) {
  int q[256], sc[8], m[8], scj[8], mj[8];
  uint16_t db, dmb;
  int gs = group;
  int st = kqo_quant_asym(w, gs, 15, q, sc, m, &db, &dmb);
  if (st) return st;
  for (int j = 0; j < 8; j++) { scj[j] = sc[j * 32 / gs]; mj[j] = m[j * 32 / gs]; }
  wr16(out, db);
  wr16(out + 2, dmb);
  kqo_pack_scales(scj, mj, out + 4);
  kqo_pack_nibbles(q, out + 16);
  return KQO_OK;
}

static int kqo_quant_sb_q5k(const float* w, uint8_t* out) {
  int q[256], sc[8], m[8];
  uint16_t db, dmb;
  int st = kqo_quant_asym(w, 32, 31, q, sc, m, &db, &dmb);
  if (st) return st;
  wr16(out, db);
  wr16(out + 2, dmb);
  kqo_pack_scales(sc, m, out + 4);
  uint8_t* qh = out + 16;
  uint8_t* qs = out + 48;
  memset(qh, 0, 32);
  for (int c = 0; c < 4; c++)
    for (int r = 0; r < 32; r++) {
      int a = q[64 * c + r], b = q[64 * c + 32 + r];
      qs[32 * c + r] = (uint8_t)((a & 15) | ((b & 15) << 4));
      qh[r] |= (uint8_t)(((a >> 4) & 1) << (2 * c));
      qh[r] |= (uint8_t)(((b >> 4) & 1) << (2 * c + 1));
    }
  return KQO_OK;
}

/* Symmetric Q6_K: per 16-weight sub-block, s = amax/31; d = fp16 round-up
 * of max s / 127; sc = ceil(s/d); q = rne(w/(d sc)) + 32 clamped to 0..63. */
static int kqo_quant_sb_q6k(const float* w, uint8_t* out) {
  double s[16], max_s = 0.0;
  for (int j = 0; j < 16; j++) {
    double a = 0.0;
    for (int i = 0; i < 16; i++) {
      double v = fabs((double)w[16 * j + i]);
      if (v > a) a = v;
    }
    s[j] = a / 31.0;
    if (s[j] > max_s) max_s = s[j];
  }
  double d;
  uint16_t db;
  if (!kqo_half_round_up(max_s / 127.0, &d, &db)) return KQO_RANGE;
  int sc[16], q[256];
  for (int j = 0; j < 16; j++) {
    int v = 0;
    if (d > 0.0) {
      double t = ceil(s[j] / d);
      v = (t > 127.0) ? 127 : (int)t;
    }
    sc[j] = v;
    double step = d * v;
    for (int i = 0; i < 16; i++) {
      int qi = 0;
      if (step > 0.0) {
        double t = nearbyint((double)w[16 * j + i] / step) + 32.0;
        qi = (t < 0.0) ? 0 : (t > 63.0 ? 63 : (int)t);
      }
      q[16 * j + i] = qi;
    }
  }
  uint8_t* ql = out;
  uint8_t* qh = out + 128;
  memset(ql, 0, 128);
  memset(qh, 0, 64);
  for (int i = 0; i < 256; i++) {
    int h = i / 128, t = (i % 128) / 32, l = i % 32;
    int lo = q[i] & 15, hb = q[i] >> 4;
    uint8_t* lp = &ql[64 * h + l + 32 * (t & 1)];
    *lp |= (uint8_t)((t < 2) ? lo : (lo << 4));
    qh[32 * h + l] |= (uint8_t)(hb << (2 * t));
  }
  for (int j = 0; j < 16; j++) out[192 + j] = (uint8_t)(int8_t)sc[j];
  wr16(out + 208, db);
  return KQO_OK;
}

/* Quantise an N x K fp32 matrix into format fmt. */
int kqo_quantize(int fmt, const float* W, int64_t N, int64_t K, uint8_t* out) {
  int st = kqo_check(fmt, N, K);
  if (st) return st;
  int64_t nsb = K / 256;
  for (int64_t n = 0; n < N; n++)
    for (int64_t b = 0; b < nsb; b++) {
      const float* w = W + n * K + b * 256;
      int64_t idx = n * nsb + b;
      if (fmt == KQO_Q4_K) st = kqo_quant_sb_q4k(w, 32, out + idx * 144);
      else if (fmt == KQO_Q5_K) st = kqo_quant_sb_q5k(w, out + idx * 176);
      else if (fmt == KQO_Q6_K) st = kqo_quant_sb_q6k(w, out + idx * 210);
      else {
        int q[256], sc[2], m[2];
        uint16_t db, dmb;
        st = kqo_quant_asym(w, 128, 15, q, sc, m, &db, &dmb);
        if (!st) {
          kqo_pack_nibbles(q, out + idx * 128);
          uint8_t* p = out + N * nsb * 128 + idx * 8;
          wr16(p, db);
          wr16(p + 2, dmb);
          p[4] = (uint8_t)sc[0]; p[5] = (uint8_t)sc[1];
          p[6] = (uint8_t)m[0];  p[7] = (uint8_t)m[1];
        }
      }
      if (st) return st;
    }
  return KQO_OK;
}

/* Q4_K blocks whose (sc, m) statistics are taken over 128-weight groups, so
 * sub-blocks 0..3 and 4..7 each share one pair (mergeable data). */
int kqo_quantize_q4k_group128(const float* W, int64_t N, int64_t K,
                              uint8_t* out) {
  int st = kqo_check(KQO_Q4_K, N, K);
  if (st) return st;
  int64_t nsb = K / 256;
  for (int64_t n = 0; n < N; n++)
    for (int64_t b = 0; b < nsb; b++) {
      st = kqo_quant_sb_q4k(W + n * K + b * 256, 128, out + (n * nsb + b) * 144);
      if (st) return st;
    }
  return KQO_OK;
}

/* Lossless merge Q4_K -> G128: requires sub-blocks 0..3 to share (sc, m)
 * and 4..7 to share (sc, m) in every super-block. */
int kqo_merge_g128(const uint8_t* q4k, int64_t N, int64_t K, uint8_t* out) {
  int st = kqo_check(KQO_Q4_K, N, K);
  if (st) return st;
  int64_t nsb = K / 256, total = N * nsb;
  for (int64_t idx = 0; idx < total; idx++) {
    const uint8_t* b = q4k + idx * 144;
    int sc[8], m[8];
    for (int j = 0; j < 8; j++) kqo_scale_min(b + 4, j, &sc[j], &m[j]);
    for (int g = 0; g < 2; g++)
      for (int j = 4 * g + 1; j < 4 * g + 4; j++)
        if (sc[j] != sc[4 * g] || m[j] != m[4 * g]) return KQO_NOT_MERGEABLE;
    memcpy(out + idx * 128, b + 16, 128);
    uint8_t* p = out + total * 128 + idx * 8;
    p[0] = b[0]; p[1] = b[1]; p[2] = b[2]; p[3] = b[3];
    p[4] = (uint8_t)sc[0]; p[5] = (uint8_t)sc[4];
    p[6] = (uint8_t)m[0];  p[7] = (uint8_t)m[4];
  }
  return KQO_OK;
}

/* ------------------------- SwiGLU activation ---------------------------- */
/*
 * The decoder's feed-forward block is SwiGLU (the Core AI card for
 * Muse-Glimmer-30B, section "The architecture, and what the port had to do
 * about it"): the input of the down projection is silu(gate) * up, element
 * by element, with gate and up the outputs of the two projections that read
 * the same hidden state.  The pages name the block but do not write the
 * function out; the reading taken is the standard one, silu(v) = v * s(v)
 * with s the logistic function s(v) = 1 / (1 + e^-v).  The result feeds the
 * next GEMV as bf16 (the activation type of the whole path), rounded to
 * nearest, ties to even.
 */

/* silu(v) = v / (1 + e^-v), plain fp64.  For v -> -inf, e^-v -> +inf and
 * the quotient -> -0. */
double kqo_silu(double v) { return v / (1.0 + exp(-v)); }

/* double -> bf16 bits, round to nearest, ties to even, directly from the
 * double (no intermediate rounding).  bf16 = 1 sign, 8 exponent (bias 127),
 * 7 fraction bits; the quantum of a value in [2^e, 2^(e+1)) is 2^(e-7),
 * and never below 2^-133 (the subnormal quantum).  Magnitudes that round
 * to 2^128 or more become infinity. */
uint16_t kqo_bf16_from_double(double v) {
  if (v != v) return 0x7FC0;                      /* NaN */
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);                                   /* a = m 2^e, m in [0.5, 1) */
  int qexp = (e - 1) - 7;                         /* quantum exponent */
  if (qexp < -133) qexp = -133;
  double r = nearbyint(ldexp(a, -qexp));          /* default mode: to nearest, ties to even */
  r = ldexp(r, qexp);
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  float f = (float)r;                             /* exact: 8 significant bits */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* h_exact[i] = silu(g[i]) * u[i] (fp64) and h_bf16[i] its bf16 rounding,
 * for i < n. */
void kqo_swiglu(const double* g, const double* u, int64_t n, double* h_exact,
                uint16_t* h_bf16) {
  for (int64_t i = 0; i < n; i++) {
    h_exact[i] = kqo_silu(g[i]) * u[i];
    h_bf16[i] = kqo_bf16_from_double(h_exact[i]);
  }
}

/* out[n] = sum_k |w^[n][k]| * e[k] (k ascending, fp64), for an error
 * vector e >= 0 over the K inputs: how far y[n] may move when every input
 * k may move by e[k]. */
int kqo_gemv_absw(int fmt, const uint8_t* W, int64_t N, int64_t K, const double* e,
                  double* out) {
  int st = kqo_check(fmt, N, K);
  if (st) return st;
  int64_t nsb = K / 256;
  double w[256];
  for (int64_t n = 0; n < N; n++) {
    double acc = 0.0;
    for (int64_t b = 0; b < nsb; b++) {
      const uint8_t *blk, *par;
      kqo_locate(fmt, W, N, K, n, b, &blk, &par);
      kqo_dequant_sb(fmt, blk, par, w);
      for (int i = 0; i < 256; i++) acc += fabs(w[i]) * e[b * 256 + i];
    }
    out[n] = acc;
  }
  return KQO_OK;
}

/* ------------------- int8 activations (dp4a GEMV) ---------------------- */
/*
 * The CUDA backend of the pages runs the packed K-quant weights as integer
 * GEMV kernels with dp4a (the daily.dev summary, answer on exporting GGUF
 * checkpoints): the activations are quantised to int8 as well, and each
 * sub-block's dot product is an integer sum.  The pages give no block size
 * or rounding; the reading taken is per 32 activations of a token (the
 * Q4_K / Q5_K sub-block), symmetric:
 *     dx = amax / 127,  xq = round_to_nearest_even(x / dx),  x~ = dx * xq
 * with amax the largest |x| of the block, both operations in fp32
 * (binary32 division, round to nearest), and xq = 0, dx = 0 for an all-zero
 * block.  The GEMV of this path is then exactly
 *     y[t][n] = sum_k w^[n][k] * x~[t][k]
 * which this file computes in fp64 like kqo_gemv, and A = sum |w^ x~|.
 */
int kqo_quantize_x_q8(const uint16_t* x, int n_tok, int64_t K, int8_t* xq, float* dx) {
  if (n_tok < 1 || K <= 0 || K % 32 != 0) return KQO_BAD_SHAPE;
  for (int t = 0; t < n_tok; t++)
    for (int64_t b = 0; b < K / 32; b++) {
      const uint16_t* xb = x + (int64_t)t * K + 32 * b;
      float amax = 0.0f;
      for (int i = 0; i < 32; i++) {
        float v = (float)kqo_bf16_to_double(xb[i]);   /* exact: bf16 -> fp32 */
        float a = fabsf(v);
        if (a > amax) amax = a;
      }
      float d = amax / 127.0f;                         /* binary32, to nearest */
      dx[(int64_t)t * (K / 32) + b] = d;
      for (int i = 0; i < 32; i++) {
        float v = (float)kqo_bf16_to_double(xb[i]);
        long q = 0;
        if (d > 0.0f) {
          float r = v / d;                             /* binary32, to nearest */
          q = lrintf(r);                               /* to nearest, ties to even */
          if (q > 127) q = 127;
          if (q < -127) q = -127;
        }
        xq[(int64_t)t * K + 32 * b + i] = (int8_t)q;
      }
    }
  return KQO_OK;
}

/* y[t][n] = sum_k w^[n][k] * dx[t][k/32] * xq[t][k] (fp64, k ascending),
 * A[t][n] = sum_k |.|; xq, dx from kqo_quantize_x_q8. */
int kqo_gemv_q8(int fmt, const uint8_t* W, int64_t N, int64_t K, const int8_t* xq,
                const float* dx, int n_tok, double* y, double* A) {
  int st = kqo_check(fmt, N, K);
  if (st) return st;
  int64_t nsb = K / 256;
  double w[256];
  for (int64_t n = 0; n < N; n++) {
    for (int t = 0; t < n_tok; t++) {
      y[t * N + n] = 0.0;
      if (A) A[t * N + n] = 0.0;
    }
    for (int64_t b = 0; b < nsb; b++) {
      const uint8_t *blk, *par;
      kqo_locate(fmt, W, N, K, n, b, &blk, &par);
      kqo_dequant_sb(fmt, blk, par, w);
      for (int t = 0; t < n_tok; t++) {
        for (int i = 0; i < 256; i++) {
          int64_t k = b * 256 + i;
          double xv = (double)dx[(int64_t)t * (K / 32) + k / 32] * (double)xq[(int64_t)t * K + k];
          double p = w[i] * xv;
          y[t * N + n] += p;
          if (A) A[t * N + n] += fabs(p);
        }
      }
    }
  }
  return KQO_OK;
}
