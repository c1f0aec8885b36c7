/*
 * qoq_oracle.c -- plain, slow CPU oracle for the QoQ W4A8 g128 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of the
 * package entry file and the CPU-baseline leg of the benchmark may load this
 * library.  The CUDA product path never links, calls or imports it, and this
 * file shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (sources are the four web pages on W4A8 serving):
 *  - QServe talk write-up (greptalks.ai, MLSys'25), section "Progressive Group
 *    Quantization for W4A8 GEMM": fp16 weights are quantized per output channel
 *    to 8 bits, held in a protective range (-119..119), then per group to 4 bits;
 *    the 4-bit codes are dequantized back to 8 bits before the integer GEMM and
 *    the per-channel scale is applied in the epilogue.
 *  - Lecture 15 notes (cs2680), section 15.6: level 1 per channel, int8 range,
 *    fp16 scales; level 2 per group g = 128, int8 -> int4, integer scales.
 *  - QFactory notes (papercache.org), section 2 "dequantization" and Fig. 3:
 *    asymmetric dequantization is w = (w_quant - zero) * scale.
 *  - QServe talk write-up, "Precision Data Flow": activations are 8-bit,
 *    quantized per token (symmetric; the pages fix only the bit width).
 *
 * Readings taken where the pages are silent (each one is listed, with its
 * reason, in the design document):
 *  R1 level-1 scale s1 = fp16(amax_k |W[n,k]| / 119), the divide in IEEE fp32,
 *     then rounded to fp16 (nearest-even); codes Q8 = clamp(rint(W/s1), +-119),
 *     the divide again IEEE fp32 and rint ties-to-even.
 *  R2 level-2 group range includes zero: lo = min(0, min Q8), hi = max(0, max Q8);
 *     s2 = max(1, ceil((hi - lo) / 15)); z = rne(-lo / s2);
 *     q4 = clamp(rne(Q8 / s2) + z, 0, 15); all in exact integer arithmetic,
 *     rne = round half to even.
 *  R3 activation scale s_x = fp16(amax_k |X[m,k]| / 127) (fp32 divide, then fp16),
 *     Xq = clamp(rint(X / s_x), -127, 127).
 *  R4 an all-zero row (or a scale that underflows to fp16 zero) gets scale 0 and
 *     codes 0; its level-2 groups get s2 = 1, z = 0.
 *  R6, R7 (the norm fused with the activation quantizer): see
 *     qoq_oracle_norm_quant_act.
 *  R5 acc[m,n] = sum_k Xq[m,k] * ((q4[n,k] - z[n,k/g]) * s2[n,k/g]) in int64;
 *     Y[m,n] = fp16_rn(acc * s_x[m] * s1[n]) with the product taken in double
 *     (exact: 31 + 11 + 11 significant bits fit in 53), rounded once.
 *
 * fp16 <-> binary64 conversions below are written from the IEEE 754 binary16
 * definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread -ffp-contract=off (no fast-math).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QOQ_ORACLE_OK 0
#define QOQ_ORACLE_EARG 1
#define QOQ_ORACLE_ERANGE 2

/* ------------------------------------------------------------------------ */
/* binary16 helpers                                                          */
/* ------------------------------------------------------------------------ */

/* Exact value of a binary16 bit pattern. */
double qoq_oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24); /* subnormal: frac * 2^-24 */
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
  }
  return sign ? -v : v;
}

/* Round a binary64 value to the nearest binary16, ties to even. */
uint16_t qoq_oracle_double_to_half(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7e00;
  if (isinf(a)) return sign | 0x7c00;
  if (a == 0.0) return sign;
  /* a = m * 2^e with m in [0.5, 1): the leading bit has weight 2^(e-1). */
  int e;
  (void)frexp(a, &e);
  int lead = e - 1;
  if (lead < -14) lead = -14; /* subnormal range shares the quantum 2^-24 */
  double quantum = ldexp(1.0, lead - 10);
  double r = nearbyint(a / quantum); /* exact scaling by a power of two; RNE */
  double v = r * quantum;            /* the rounded magnitude, exact */
  if (v > 65504.0) return sign | 0x7c00; /* overflow to inf (ties at 65520 go up) */
  if (v < ldexp(1.0, -14)) {
    /* subnormal (or rounded up to the smallest normal, handled below) */
    return sign | (uint16_t)(v / ldexp(1.0, -24));
  }
  int e2;
  double m2 = frexp(v, &e2); /* v = m2 * 2^e2, m2 in [0.5,1) */
  int expo = e2 - 1 + 15;
  int frac = (int)((m2 * 2.0 - 1.0) * 1024.0);
  return sign | (uint16_t)(expo << 10) | (uint16_t)frac;
}

/* ------------------------------------------------------------------------ */
/* exact integer helpers                                                     */
/* ------------------------------------------------------------------------ */

/* floor(a / b) for b > 0 */
static int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && (a < 0)) q -= 1;
  return q;
}

/* a / b rounded to nearest, ties to even, b > 0, exact. */
static int64_t rne_div(int64_t a, int64_t b) {
  int64_t q = floor_div(a, b);
  int64_t r = a - q * b; /* 0 <= r < b */
  if (2 * r > b) return q + 1;
  if (2 * r == b) return (q & 1) ? q + 1 : q;
  return q;
}

static int64_t clamp64(int64_t v, int64_t lo, int64_t hi) {
  return v < lo ? lo : (v > hi ? hi : v);
}

/* Dequantization of one code: (w_quant - zero) * scale (QFactory notes,
 * section 2 and the Fig. 3 example; QServe: "subtraction after
 * multiplication" is a kernel reordering of the same value). */
int64_t qoq_oracle_dequant_code(int64_t q, int64_t zero, int64_t scale) {
  return (q - zero) * scale;
}

/* Same formula on real-valued parameters, for the QFactory Fig. 3 example. */
double qoq_oracle_dequant_real(double q, double zero, double scale) {
  return (q - zero) * scale;
}

/* ------------------------------------------------------------------------ */
/* symmetric per-row 8-bit quantization (shared recipe of R1 and R3)         */
/* ------------------------------------------------------------------------ */

/* Quantize one fp16 row symmetrically to [-qmax, qmax] with an fp16 scale.
 * scale = fp16(amax / qmax) with an IEEE fp32 divide; codes = rint(x / scale)
 * with an IEEE fp32 divide and ties to even, then clamped. */
static void symmetric_row(int K, const uint16_t* row, int qmax, uint16_t* scale_out,
                          int8_t* codes) {
  float amax = 0.0f;
  for (int k = 0; k < K; ++k) {
    float v = (float)fabs(qoq_oracle_half_to_double(row[k]));
    if (v > amax) amax = v;
  }
  uint16_t s = 0;
  if (amax > 0.0f) {
    volatile float q = amax / (float)qmax; /* IEEE binary32 divide */
    s = qoq_oracle_double_to_half((double)q);
  }
  *scale_out = s;
  float sf = (float)qoq_oracle_half_to_double(s);
  for (int k = 0; k < K; ++k) {
    if (sf == 0.0f) {
      codes[k] = 0;
      continue;
    }
    volatile float t = (float)qoq_oracle_half_to_double(row[k]) / sf; /* binary32 */
    float r = rintf(t);                                               /* ties to even */
    if (r > (float)qmax) r = (float)qmax;
    if (r < (float)-qmax) r = (float)-qmax;
    codes[k] = (int8_t)r;
  }
}

/* ------------------------------------------------------------------------ */
/* weights: progressive group quantization                                   */
/* ------------------------------------------------------------------------ */

/* Level 1 then level 2 for W [N][K] (row n = output channel).
 * Outputs: s1 [N] fp16 bits, Q8 [N][K] (level-1 codes, may be NULL),
 * q4 [N][K] (one code per byte, 0..15), s2 [N][K/g], z [N][K/g].
 * Returns QOQ_ORACLE_EARG on bad sizes. */
int qoq_oracle_weight_quant(int N, int K, int g, const uint16_t* W, uint16_t* s1, int8_t* Q8,
                            uint8_t* q4, uint8_t* s2, uint8_t* z) {
  if (N <= 0 || K <= 0 || g <= 0 || K % g != 0 || !W || !s1 || !q4 || !s2 || !z)
    return QOQ_ORACLE_EARG;
  int G = K / g;
  int8_t* row_q8 = (int8_t*)malloc((size_t)K);
  if (!row_q8) return QOQ_ORACLE_EARG;
  for (int n = 0; n < N; ++n) {
    const uint16_t* wrow = W + (size_t)n * K;
    /* level 1: per output channel, protective range [-119, 119] */
    symmetric_row(K, wrow, 119, &s1[n], row_q8);
    if (Q8) memcpy(Q8 + (size_t)n * K, row_q8, (size_t)K);
    /* level 2: per group of g along K, asymmetric unsigned 4-bit */
    for (int j = 0; j < G; ++j) {
      const int8_t* grp = row_q8 + (size_t)j * g;
      int64_t lo = 0, hi = 0; /* the range always includes zero (R2) */
      for (int t = 0; t < g; ++t) {
        if (grp[t] < lo) lo = grp[t];
        if (grp[t] > hi) hi = grp[t];
      }
      int64_t scale = (hi - lo + 14) / 15; /* ceil((hi - lo) / 15) */
      if (scale < 1) scale = 1;
      int64_t zero = rne_div(-lo, scale);
      s2[(size_t)n * G + j] = (uint8_t)scale;
      z[(size_t)n * G + j] = (uint8_t)zero;
      for (int t = 0; t < g; ++t) {
        int64_t q = clamp64(rne_div(grp[t], scale) + zero, 0, 15);
        q4[(size_t)n * K + (size_t)j * g + t] = (uint8_t)q;
      }
    }
  }
  free(row_q8);
  return QOQ_ORACLE_OK;
}

/* Reconstructed 8-bit weight w8 = (q4 - z) * s2 for every element (int16 out). */
int qoq_oracle_dequant_weights(int N, int K, int g, const uint8_t* q4, const uint8_t* s2,
                               const uint8_t* z, int16_t* w8) {
  if (N <= 0 || K <= 0 || g <= 0 || K % g != 0 || !q4 || !s2 || !z || !w8) return QOQ_ORACLE_EARG;
  int G = K / g;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      size_t gi = (size_t)n * G + k / g;
      w8[(size_t)n * K + k] = (int16_t)qoq_oracle_dequant_code(q4[(size_t)n * K + k], z[gi], s2[gi]);
    }
  return QOQ_ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* activations: per-token symmetric int8                                     */
/* ------------------------------------------------------------------------ */

int qoq_oracle_act_quant(int M, int K, const uint16_t* X, int8_t* Xq, uint16_t* sx) {
  if (M <= 0 || K <= 0 || !X || !Xq || !sx) return QOQ_ORACLE_EARG;
  for (int m = 0; m < M; ++m)
    symmetric_row(K, X + (size_t)m * K, 127, &sx[m], Xq + (size_t)m * K);
  return QOQ_ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* W4Ax activations: 4-bit blocks with 8-bit outlier blocks                  */
/* ------------------------------------------------------------------------ */

/* COMET explainer (bookshelf), FMPQ: activations are quantized in blocks of
 * 128 channels (the tensor-core tile's granularity); the outlier channels,
 * clustered into a few blocks by a channel permutation, stay at 8 bits and
 * every other block goes to 4 bits.  Readings taken (the pages fix neither
 * the scale nor the rounding): the permutation puts the outlier blocks first,
 * so the n8 leading blocks are 8-bit; each (token m, block b) has its own
 * symmetric scale, the recipe of the per-token quantizer with qmax = 127
 * (8-bit) or 7 (4-bit):
 *   s[m,b] = fp16(amax_b / qmax) (IEEE fp32 divide), code = clamp(rint(x / s), +-qmax).
 * Out: codes [M][K] int8 (one code per byte), sxb [M][K/128] fp16 bits. */
int qoq_oracle_act_quant_w4ax(int M, int K, int n8, const uint16_t* X, int8_t* codes, uint16_t* sxb) {
  if (M <= 0 || K <= 0 || K % 128 != 0 || n8 < 0 || n8 > K / 128 || !X || !codes || !sxb)
    return QOQ_ORACLE_EARG;
  const int G = K / 128;
  for (int m = 0; m < M; ++m)
    for (int b = 0; b < G; ++b)
      symmetric_row(128, X + (size_t)m * K + (size_t)b * 128, b < n8 ? 127 : 7, &sxb[(size_t)m * G + b],
                    codes + (size_t)m * K + (size_t)b * 128);
  return QOQ_ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* GEMM: integer accumulation, per-channel scales in the epilogue            */
/* ------------------------------------------------------------------------ */

static int64_t dot_entry(int K, int g, const int8_t* xrow, const uint8_t* q4row,
                         const uint8_t* s2row, const uint8_t* zrow) {
  int64_t acc = 0;
  for (int k = 0; k < K; ++k) {
    int64_t w = qoq_oracle_dequant_code(q4row[k], zrow[k / g], s2row[k / g]);
    acc += (int64_t)xrow[k] * w;
  }
  return acc;
}

static uint16_t epilogue(int64_t acc, uint16_t sx, uint16_t s1) {
  double y = (double)acc * qoq_oracle_half_to_double(sx) * qoq_oracle_half_to_double(s1);
  return qoq_oracle_double_to_half(y);
}

/* Full product: acc [M][N] int64 (may be NULL), Y [M][N] fp16 bits (may be NULL).
 * Returns QOQ_ORACLE_ERANGE if some |acc| >= 2^31 (cannot happen for K <= 131072). */
int qoq_oracle_gemm(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx,
                    const uint8_t* q4, const uint8_t* s2, const uint8_t* z, const uint16_t* s1,
                    int64_t* acc, uint16_t* Y) {
  if (M <= 0 || N <= 0 || K <= 0 || g <= 0 || K % g != 0 || !Xq || !sx || !q4 || !s2 || !z || !s1)
    return QOQ_ORACLE_EARG;
  int G = K / g;
  int rc = QOQ_ORACLE_OK;
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      int64_t a = dot_entry(K, g, Xq + (size_t)m * K, q4 + (size_t)n * K, s2 + (size_t)n * G,
                            z + (size_t)n * G);
      if (a >= ((int64_t)1 << 31) || a < -((int64_t)1 << 31)) rc = QOQ_ORACLE_ERANGE;
      if (acc) acc[(size_t)m * N + n] = a;
      if (Y) Y[(size_t)m * N + n] = epilogue(a, sx[m], s1[n]);
    }
  return rc;
}

/* W4Ax product (COMET explainer, the W4Ax kernel: mixed 4-bit and 8-bit
 * activation blocks times 4-bit weights, each block's partial sums scaled by
 * the block's activation scale on the general-purpose cores).  With the
 * dequantized weights w8 = (q4 - z) s2 of the progressive group format:
 *   acc_b[m,n] = sum over the 128 channels k of block b of codes[m,k] w8[n,k]  (int64),
 *   Y[m,n] = fp16_rn(s1[n] * sum_b sxb[m,b] * acc_b[m,n])
 * the sum over blocks taken in double, in block order, then rounded once to
 * fp16 (each term s * acc_b is exact in double).  acc_sum (nullable) gets
 * sum_b acc_b, acc_blocks (nullable) every acc_b as [M][N][K/128]. */
int qoq_oracle_gemm_w4ax(int M, int N, int K, int g, const int8_t* codes, const uint16_t* sxb,
                         const uint8_t* q4, const uint8_t* s2, const uint8_t* z, const uint16_t* s1,
                         int64_t* acc_blocks, int64_t* acc_sum, uint16_t* Y) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 != 0 || g <= 0 || K % g != 0 || !codes || !sxb || !q4 || !s2 ||
      !z || !s1)
    return QOQ_ORACLE_EARG;
  const int G = K / g, B = K / 128;
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      double y = 0.0;
      int64_t total = 0;
      for (int b = 0; b < B; ++b) {
        int64_t a = 0;
        for (int k = b * 128; k < (b + 1) * 128; ++k) {
          const size_t gi = (size_t)n * G + k / g;
          a += (int64_t)codes[(size_t)m * K + k] * qoq_oracle_dequant_code(q4[(size_t)n * K + k], z[gi], s2[gi]);
        }
        if (acc_blocks) acc_blocks[((size_t)m * N + n) * B + b] = a;
        total += a;
        y += qoq_oracle_half_to_double(sxb[(size_t)m * B + b]) * (double)a;
      }
      if (acc_sum) acc_sum[(size_t)m * N + n] = total;
      if (Y) Y[(size_t)m * N + n] = qoq_oracle_double_to_half(qoq_oracle_half_to_double(s1[n]) * y);
    }
  return QOQ_ORACLE_OK;
}

/* Zero-point folding (QFactory notes, papercache.org, section 4.3 "mapping
 * function transformation", Table 2: a matmul whose operand carries an
 * offset is rewritten as the plain product plus a product with the all-ones
 * matrix J, whose rows are the reduction's sums).  The weights of group j of
 * row n are w8 = s2 q4 - zs with zs = z s2, so
 *   acc[m,n] = sum_k Xq[m,k] (q4[n,k] s2[n,k/g])  -  sum_j zs[n,j] RS[m,j],
 *   RS[m,j]  = sum over the g channels k of group j of Xq[m,k]  (Xq times J),
 * all in int64, then the same epilogue as qoq_oracle_gemm.  The steps are
 * taken in that order: row sums, the scale-only product, the correction.
 * rowsum (nullable) receives RS [M][K/g].  Equal to qoq_oracle_gemm's acc by
 * distributivity; the tests check that and a hand-worked example. */
int qoq_oracle_gemm_zero_folded(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx,
                                const uint8_t* q4, const uint8_t* s2, const uint8_t* z, const uint16_t* s1,
                                int64_t* rowsum, int64_t* acc, uint16_t* Y) {
  if (M <= 0 || N <= 0 || K <= 0 || g <= 0 || K % g != 0 || !Xq || !sx || !q4 || !s2 || !z || !s1)
    return QOQ_ORACLE_EARG;
  const int G = K / g;
  int64_t* RS = (int64_t*)malloc((size_t)M * G * sizeof(int64_t));
  if (!RS) return QOQ_ORACLE_EARG;
  for (int m = 0; m < M; ++m)
    for (int j = 0; j < G; ++j) {
      int64_t t = 0;
      for (int k = j * g; k < (j + 1) * g; ++k) t += Xq[(size_t)m * K + k];
      RS[(size_t)m * G + j] = t;
    }
  int rc = QOQ_ORACLE_OK;
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      const int8_t* xrow = Xq + (size_t)m * K;
      const uint8_t* qrow = q4 + (size_t)n * K;
      int64_t scaled = 0;
      for (int k = 0; k < K; ++k) scaled += (int64_t)xrow[k] * ((int64_t)qrow[k] * s2[(size_t)n * G + k / g]);
      int64_t corr = 0;
      for (int j = 0; j < G; ++j)
        corr += ((int64_t)z[(size_t)n * G + j] * s2[(size_t)n * G + j]) * RS[(size_t)m * G + j];
      const int64_t a = scaled - corr;
      if (a >= ((int64_t)1 << 31) || a < -((int64_t)1 << 31)) rc = QOQ_ORACLE_ERANGE;
      if (acc) acc[(size_t)m * N + n] = a;
      if (Y) Y[(size_t)m * N + n] = epilogue(a, sx[m], s1[n]);
    }
  if (rowsum) memcpy(rowsum, RS, (size_t)M * G * sizeof(int64_t));
  free(RS);
  return rc;
}

/* The same product on several host threads, for full-size checks.  The
 * output channels are cut into `threads` contiguous ranges, one per POSIX
 * thread.  Per output channel n the thread first dequantizes the weight row,
 * w8[k] = (q4[n,k] - z[n,k/g]) * s2[n,k/g] (the dequantization step, once per
 * row instead of once per token), then sums Xq[m,k] * w8[k] over k in int64
 * for every token m and applies the same epilogue.  Integer sums do not
 * depend on their order, so every acc and Y equals qoq_oracle_gemm's.
 * Returns QOQ_ORACLE_EARG for bad sizes or a failed thread start or buffer. */
typedef struct {
  int M, N, K, g, n0, n1, rc;
  const int8_t* Xq;
  const uint16_t* sx;
  const uint8_t *q4, *s2, *z;
  const uint16_t* s1;
  int64_t* acc;
  uint16_t* Y;
} gemm_range;

static void* gemm_range_run(void* arg) {
  gemm_range* r = (gemm_range*)arg;
  const int K = r->K, G = K / r->g;
  int16_t* w8 = (int16_t*)malloc((size_t)K * sizeof(int16_t)); /* |w8| <= 240 */
  if (!w8) {
    r->rc = QOQ_ORACLE_EARG;
    return NULL;
  }
  r->rc = QOQ_ORACLE_OK;
  for (int n = r->n0; n < r->n1; ++n) {
    const uint8_t* q4row = r->q4 + (size_t)n * K;
    for (int k = 0; k < K; ++k)
      w8[k] = (int16_t)qoq_oracle_dequant_code(q4row[k], r->z[(size_t)n * G + k / r->g], r->s2[(size_t)n * G + k / r->g]);
    for (int m = 0; m < r->M; ++m) {
      const int8_t* xrow = r->Xq + (size_t)m * K;
      int64_t a = 0;
      for (int k = 0; k < K; ++k) a += (int64_t)xrow[k] * w8[k];
      if (a >= ((int64_t)1 << 31) || a < -((int64_t)1 << 31)) r->rc = QOQ_ORACLE_ERANGE;
      if (r->acc) r->acc[(size_t)m * r->N + n] = a;
      if (r->Y) r->Y[(size_t)m * r->N + n] = epilogue(a, r->sx[m], r->s1[n]);
    }
  }
  free(w8);
  return NULL;
}

int qoq_oracle_gemm_threads(int M, int N, int K, int g, const int8_t* Xq, const uint16_t* sx,
                            const uint8_t* q4, const uint8_t* s2, const uint8_t* z, const uint16_t* s1,
                            int64_t* acc, uint16_t* Y, int threads) {
  if (M <= 0 || N <= 0 || K <= 0 || g <= 0 || K % g != 0 || !Xq || !sx || !q4 || !s2 || !z || !s1 ||
      threads <= 0)
    return QOQ_ORACLE_EARG;
  if (threads > N) threads = N;
  gemm_range* rs = (gemm_range*)calloc((size_t)threads, sizeof(gemm_range));
  pthread_t* ts = (pthread_t*)calloc((size_t)threads, sizeof(pthread_t));
  int* started = (int*)calloc((size_t)threads, sizeof(int));
  int rc = QOQ_ORACLE_OK;
  if (!rs || !ts || !started) rc = QOQ_ORACLE_EARG;
  for (int t = 0; rc == QOQ_ORACLE_OK && t < threads; ++t) {
    gemm_range r = {M, N, K, g, (int)((int64_t)N * t / threads), (int)((int64_t)N * (t + 1) / threads),
                    QOQ_ORACLE_OK, Xq, sx, q4, s2, z, s1, acc, Y};
    rs[t] = r;
    if (pthread_create(&ts[t], NULL, gemm_range_run, &rs[t]) != 0)
      rc = QOQ_ORACLE_EARG;
    else
      started[t] = 1;
  }
  for (int t = 0; t < threads && started; ++t)
    if (started[t]) {
      pthread_join(ts[t], NULL);
      if (rs[t].rc == QOQ_ORACLE_EARG) rc = QOQ_ORACLE_EARG;
      else if (rs[t].rc == QOQ_ORACLE_ERANGE && rc == QOQ_ORACLE_OK) rc = QOQ_ORACLE_ERANGE;
    }
  free(rs);
  free(ts);
  free(started);
  return rc;
}

/* Selected entries only: for i < count, entry (m_idx[i], n_idx[i]).
 * Xq is [M][K] and the weight arrays are [N][K] / [N][K/g] as above. */
int qoq_oracle_gemm_entries(int count, const int32_t* m_idx, const int32_t* n_idx, int K, int g,
                            const int8_t* Xq, const uint16_t* sx, const uint8_t* q4,
                            const uint8_t* s2, const uint8_t* z, const uint16_t* s1, int64_t* acc,
                            uint16_t* Y) {
  if (count < 0 || K <= 0 || g <= 0 || K % g != 0 || !m_idx || !n_idx || !Xq || !sx || !q4 || !s2 ||
      !z || !s1)
    return QOQ_ORACLE_EARG;
  int G = K / g;
  for (int i = 0; i < count; ++i) {
    int m = m_idx[i], n = n_idx[i];
    int64_t a = dot_entry(K, g, Xq + (size_t)m * K, q4 + (size_t)n * K, s2 + (size_t)n * G,
                          z + (size_t)n * G);
    if (acc) acc[i] = a;
    if (Y) Y[i] = epilogue(a, sx[m], s1[n]);
  }
  return QOQ_ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* norm fused with the activation quantizer                                  */
/* ------------------------------------------------------------------------ */

/* QServe talk write-up, "Precision Data Flow and Activation Quantization
 * Fusion": a linear layer's input quantization is fused into the preceding
 * layer, such as LayerNorm, whose output is quantized to 8 bits directly.
 * The pages give no norm arithmetic; the readings taken:
 *  R6 the row statistics are exact: S1 = sum_k x_k and S2 = sum_k x_k^2 as
 *     integers in units of 2^-24 and 2^-48 (every fp16 x is an integer
 *     multiple of 2^-24), so they do not depend on summation order;
 *  R7 the rest in fp32, each operation rounded to nearest (fl32(S): the
 *     exact sum rounded once to fp32):
 *     RMSNorm (kind 0): ms = fl32(S2) / K, r = 1 / sqrt(ms + eps),
 *     y_k = fp16_rn(fl32(fl32(x_k * r) * gamma_k));
 *     LayerNorm (kind 1): mu = fl32(S1) / K, var = fl32(K S2 - S1^2) / K^2,
 *     r = 1 / sqrt(var + eps),
 *     y_k = fp16_rn(fl32(fl32(fl32(fl32(x_k - mu) * r) * gamma_k) + beta_k));
 *     eps > 0;
 *  then y is quantized per token exactly as qoq_oracle_act_quant does (R3).
 * Optional outputs: the fp16 row y (Y) and r and mu per row (rmu, 2 floats). */
int qoq_oracle_norm_quant_act(int M, int K, int kind, float eps, const uint16_t* X,
                              const uint16_t* gamma, const uint16_t* beta, uint16_t* Y, int8_t* Xq,
                              uint16_t* sx, float* rmu, int64_t* stats) {
  if (M <= 0 || K <= 0 || (kind != 0 && kind != 1) || !(eps > 0.0f) || !X || !gamma ||
      (kind == 1 && !beta) || !Xq || !sx)
    return QOQ_ORACLE_EARG;
  uint16_t* yrow = (uint16_t*)malloc((size_t)K * sizeof(uint16_t));
  if (!yrow) return QOQ_ORACLE_EARG;
  for (int m = 0; m < M; ++m) {
    const uint16_t* xrow = X + (size_t)m * K;
    int64_t s1 = 0;          /* units of 2^-24 */
    unsigned __int128 s2 = 0; /* units of 2^-48 */
    for (int k = 0; k < K; ++k) {
      int64_t a = (int64_t)(qoq_oracle_half_to_double(xrow[k]) * 16777216.0); /* exact */
      uint64_t mag = (uint64_t)(a < 0 ? -a : a);
      s1 += a;
      s2 += (unsigned __int128)mag * mag;
    }
    if (stats) {
      stats[4 * m + 0] = s1;
      stats[4 * m + 1] = (int64_t)(uint64_t)s2;
      stats[4 * m + 2] = (int64_t)(uint64_t)(s2 >> 64);
      stats[4 * m + 3] = 0;
    }
    volatile float spread; /* mean square (kind 0) or variance (kind 1) */
    volatile float mu = 0.0f;
    if (kind == 0) {
      volatile float s2f = (float)s2 * 0x1p-48f; /* one rounding, then an exact scaling */
      spread = s2f / (float)K;
    } else {
      unsigned __int128 a1 = (unsigned __int128)(uint64_t)(s1 < 0 ? -s1 : s1);
      unsigned __int128 v = (unsigned __int128)K * s2 - a1 * a1; /* >= 0, exact */
      volatile float vf = (float)v * 0x1p-48f;
      spread = vf / ((float)K * (float)K); /* K^2 is exact in fp32 for K = 128 j, j <= 1024 */
      volatile float s1f = (float)s1 * 0x1p-24f;
      mu = s1f / (float)K;
    }
    volatile float den = spread + eps;
    volatile float sq = sqrtf(den);
    const float r = 1.0f / sq;
    if (rmu) {
      rmu[2 * m] = r;
      rmu[2 * m + 1] = mu;
    }
    for (int k = 0; k < K; ++k) {
      float x = (float)qoq_oracle_half_to_double(xrow[k]);
      volatile float t = kind == 1 ? x - mu : x;
      volatile float u = t * r;
      volatile float w = u * (float)qoq_oracle_half_to_double(gamma[k]);
      if (kind == 1) w = w + (float)qoq_oracle_half_to_double(beta[k]);
      yrow[k] = qoq_oracle_double_to_half((double)w);
    }
    if (Y) memcpy(Y + (size_t)m * K, yrow, (size_t)K * sizeof(uint16_t));
    symmetric_row(K, yrow, 127, &sx[m], Xq + (size_t)m * K);
  }
  free(yrow);
  return QOQ_ORACLE_OK;
}
