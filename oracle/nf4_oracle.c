/*
 * nf4_oracle.c -- plain, slow, single-threaded CPU reference for NF4 with
 * double quantization.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load this file; the product path
 * (the CUDA library and its Python binding) never does.
 *
 * It shares no code with the CUDA library.  Every routine is written from the
 * definitions on the source pages, cited by page title and section:
 *
 *   [NF4-OPT]  "NF4反量化算子优化" (roundaboutt.github.io), sections
 *              "NF4 table", "双量化" (first / second level), "反量化",
 *              and the "naive" kernel listing that prints the table.
 *   [NF4-RPT]  "NF4 双重量化反量化 CUDA Kernel 实现报告" (Learning-CUDA report),
 *              sections 1.1 (table), 1.2 (double quantization),
 *              1.3 (dequantization formula), 2.2 (nibble order).
 *   [QTAX]     "RTX 4060 上的 LLM 量化实测：4-bit decode 比 FP16 慢在哪里",
 *              section "Fused kernel：把反量化搬到片上" (fused dequant-GEMV
 *              with fp32 accumulation; fp16 output plus the layer's bias).
 *
 * Build with contraction off (gcc -O2 -ffp-contract=off): every float
 * operation below is one IEEE-754 binary32 or binary64 operation, rounded to
 * nearest-even, in the order written.
 *
 * Readings taken where the pages are silent (each is also a test pin):
 *   - scale = fp32(fp32(code2[q] * absmax2[g]) + offset); no FMA.
 *   - NF4 codes are the 8-digit decimals printed in [NF4-OPT], rounded to fp32.
 *   - nearest-index decisions use binary64 distances, ties to the lower index.
 *   - offset = binary32 of the binary64 mean of all first-level absmax values,
 *     summed group by group (each group's blocks in order, then the group
 *     partial sums in order).
 *   - code2[i] = binary16 RNE of the binary64 value (i - 127.5) / 127.5.
 *   - a partial last block / group uses only the elements / blocks present.
 * Inputs are assumed finite.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* NF4 code book: the sixteen values printed in [NF4-OPT] "NF4 table" (the
 * naive kernel's lookup), each the binary32 nearest its 8-digit decimal.     */
static const float NF4_CODE[16] = {
    -1.00000000f, -0.69619280f, -0.52507305f, -0.39491749f,
    -0.28444138f, -0.18477343f, -0.09105004f, 0.00000000f,
    0.07958030f,  0.16093020f,  0.24611230f,  0.33791524f,
    0.44070983f,  0.56261700f,  0.72295684f,  1.00000000f};

void oracle_nf4_code(float out[16]) {
  for (int j = 0; j < 16; ++j) out[j] = NF4_CODE[j];
}

/* ------------------------------------------------------------------------ */
/* IEEE-754 rounding to a narrower binary format, from the definition.
 *
 * The exact value is (-1)^neg * m * 2^e with m a nonzero integer.  The target
 * format has p significand bits (hidden bit included), minimum normal
 * exponent emin and maximum exponent emax.  Representable magnitudes are
 * q * 2^(E - p + 1) with q < 2^p, where E = max(floor(log2 |v|), emin).
 * Result: the bit pattern with exponent field width ebits.                   */
static uint32_t round_to_format(int neg, uint64_t m, int e, int p, int emin,
                                int emax, int ebits) {
  const uint32_t sign = neg ? (1u << (p - 1 + ebits)) : 0u;
  const uint32_t exp_all_ones = (1u << ebits) - 1u;
  if (m == 0) return sign;
  /* floor(log2 |v|) = (bit length of m) - 1 + e */
  int bl = 0;
  for (uint64_t t = m; t; t >>= 1) ++bl;
  int E = bl - 1 + e;
  if (E < emin) E = emin;              /* subnormal range: fixed quantum */
  const int quantum = E - p + 1;       /* value of one unit in the last place */
  int shift = quantum - e;             /* q = m / 2^shift, rounded */
  uint64_t q;
  if (shift <= 0) {
    q = m << (-shift);                 /* exact (cannot overflow for our uses) */
  } else if (shift >= 64) {
    q = 0;                             /* far below half an ulp: rounds to 0 */
  } else {
    const uint64_t kept = m >> shift;
    const uint64_t rem = m & ((1ull << shift) - 1ull);
    const uint64_t half = 1ull << (shift - 1);
    q = kept;
    if (rem > half || (rem == half && (kept & 1ull))) q += 1ull;  /* RNE */
  }
  if (q >> p) {                        /* carried into a new binade */
    q >>= 1;
    E += 1;
  }
  if (E > emax) return sign | (exp_all_ones << (p - 1));  /* overflow -> inf */
  if (q < (1ull << (p - 1)))           /* subnormal (or zero) */
    return sign | (uint32_t)q;
  const uint32_t biased = (uint32_t)(E - emin + 1);
  return sign | (biased << (p - 1)) | (uint32_t)(q - (1ull << (p - 1)));
}

/* Split a finite binary32 into sign, integer significand and exponent. */
static void split_f32(float f, int* neg, uint64_t* m, int* e) {
  uint32_t u;
  memcpy(&u, &f, 4);
  *neg = (int)(u >> 31);
  const uint32_t bexp = (u >> 23) & 0xffu, frac = u & 0x7fffffu;
  if (bexp == 0) {
    *m = frac;
    *e = -149;
  } else {
    *m = frac | 0x800000u;
    *e = (int)bexp - 150;
  }
}

static void split_f64(double d, int* neg, uint64_t* m, int* e) {
  uint64_t u;
  memcpy(&u, &d, 8);
  *neg = (int)(u >> 63);
  const uint64_t bexp = (u >> 52) & 0x7ffu, frac = u & 0xfffffffffffffull;
  if (bexp == 0) {
    *m = frac;
    *e = -1074;
  } else {
    *m = frac | (1ull << 52);
    *e = (int)bexp - 1075;
  }
}

/* binary32 -> bfloat16 (1-8-7), round to nearest even. NaN -> quiet NaN. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u)
    return (uint16_t)((u >> 16) | ((u & 0x7fffffu) ? 0x40u : 0u));
  int neg, e;
  uint64_t m;
  split_f32(f, &neg, &m, &e);
  return (uint16_t)round_to_format(neg, m, e, 8, -126, 127, 8);
}

/* binary32 -> binary16 (1-5-10), round to nearest even (subnormals kept). */
uint16_t oracle_f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u)
    return (uint16_t)(((u >> 16) & 0x8000u) | 0x7c00u | ((u & 0x7fffffu) ? 0x200u : 0u));
  int neg, e;
  uint64_t m;
  split_f32(f, &neg, &m, &e);
  return (uint16_t)round_to_format(neg, m, e, 11, -14, 15, 5);
}

/* binary64 -> binary16 directly (one rounding, not via binary32). */
uint16_t oracle_f64_to_f16(double d) {
  uint64_t u;
  memcpy(&u, &d, 8);
  if ((u & 0x7ff0000000000000ull) == 0x7ff0000000000000ull)
    return (uint16_t)(((u >> 48) & 0x8000u) | 0x7c00u |
                      ((u & 0xfffffffffffffull) ? 0x200u : 0u));
  int neg, e;
  uint64_t m;
  split_f64(d, &neg, &m, &e);
  return (uint16_t)round_to_format(neg, m, e, 11, -14, 15, 5);
}

/* binary64 -> bfloat16 directly (one rounding). */
uint16_t oracle_f64_to_bf16(double d) {
  uint64_t u;
  memcpy(&u, &d, 8);
  if ((u & 0x7ff0000000000000ull) == 0x7ff0000000000000ull)
    return (uint16_t)(((u >> 48) & 0x8000u) | 0x7f80u |
                      ((u & 0xfffffffffffffull) ? 0x40u : 0u));
  int neg, e;
  uint64_t m;
  split_f64(d, &neg, &m, &e);
  return (uint16_t)round_to_format(neg, m, e, 8, -126, 127, 8);
}

/* binary64 -> binary32 bit pattern (one rounding, subnormals kept). */
uint32_t oracle_f64_to_f32_bits(double d) {
  uint64_t u;
  memcpy(&u, &d, 8);
  if ((u & 0x7ff0000000000000ull) == 0x7ff0000000000000ull)
    return (uint32_t)(((u >> 32) & 0x80000000u) | 0x7f800000u |
                      ((u & 0xfffffffffffffull) ? 0x400000u : 0u));
  int neg, e;
  uint64_t m;
  split_f64(d, &neg, &m, &e);
  return round_to_format(neg, m, e, 24, -126, 127, 8);
}

/* binary16 -> binary32 (exact). */
float oracle_f16_to_f32(uint16_t h) {
  const int neg = h >> 15, bexp = (h >> 10) & 0x1f, frac = h & 0x3ff;
  double v;
  if (bexp == 0x1f) {
    v = frac ? NAN : INFINITY;
  } else if (bexp == 0) {
    v = ldexp((double)frac, -24);
  } else {
    v = ldexp((double)(frac | 0x400), bexp - 25);
  }
  return (float)(neg ? -v : v);
}

/* bfloat16 -> binary32 (exact: the bf16 pattern is the top half). */
float oracle_bf16_to_f32(uint16_t h) {
  const uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ------------------------------------------------------------------------ */
/* Second-level code table: 256 binary16 values (i - 127.5) / 127.5.
 * [NF4-RPT] 1.2 fixes the shape (fp16[256]); the linear content is the
 * reading taken for this library's synthetic workloads.                     */
void oracle_code2_linear(uint16_t code2[256]) {
  for (int i = 0; i < 256; ++i) code2[i] = oracle_f64_to_f16(((double)i - 127.5) / 127.5);
}

/* A non-linear second-level table ("NF4反量化算子优化", section "第二层量化",
 * stores the scales in an 8-bit floating-point format; this is one such
 * map): logarithmically spaced magnitudes, sixteen entries per octave.
 * Entry 128 + k (k = 0..127) is binary16(2^((k - 127) / 16)) and entry
 * 127 - k its negation, so the table is increasing, antisymmetric and ends
 * at -1 and +1. The exponent is an exact binary64 quotient; exp2 of it is
 * rounded once to binary16. */
void oracle_code2_dynamic(uint16_t code2[256]) {
  for (int k = 0; k < 128; ++k) {
    const uint16_t h = oracle_f64_to_f16(exp2(((double)k - 127.0) / 16.0));
    code2[128 + k] = h;
    code2[127 - k] = (uint16_t)(h | 0x8000u);
  }
}

/* ------------------------------------------------------------------------ */
/* First-level quantization, [NF4-OPT] "第一层量化" and [NF4-RPT] 1.1:
 * flatten, cut into blocks of `bs` consecutive elements, absmax per block.  */
void oracle_block_absmax(const float* w, int64_t n, int64_t bs, float* absmax) {
  const int64_t nb = (n + bs - 1) / bs;
  for (int64_t b = 0; b < nb; ++b) {
    float m = 0.0f;
    const int64_t end = (b + 1) * bs < n ? (b + 1) * bs : n;
    for (int64_t k = b * bs; k < end; ++k) {
      const float a = fabsf(w[k]);
      if (a > m) m = a;
    }
    absmax[b] = m;
  }
}

/* Index of the nearest NF4 code to v: binary64 distances, ties -> lower. */
int oracle_nf4_nearest(float v) {
  int best = 0;
  double bestd = fabs((double)v - (double)NF4_CODE[0]);
  for (int j = 1; j < 16; ++j) {
    const double d = fabs((double)v - (double)NF4_CODE[j]);
    if (d < bestd) {
      bestd = d;
      best = j;
    }
  }
  return best;
}

/* Normalise each element by its block's absmax (one binary32 division; 0 if
 * the block is all zero), map to the nearest code, pack two indices per byte
 * with the even element in the high nibble ([NF4-RPT] 2.2, [NF4-OPT]
 * "第一层量化").  For odd n the last byte's low nibble is 0.                 */
void oracle_nf4_encode(const float* w, int64_t n, int64_t bs, const float* absmax,
                       uint8_t* packed) {
  const int64_t nbytes = (n + 1) / 2;
  for (int64_t i = 0; i < nbytes; ++i) packed[i] = 0;
  for (int64_t k = 0; k < n; ++k) {
    const float a = absmax[k / bs];
    const float v = (a == 0.0f) ? 0.0f : w[k] / a;
    const int idx = oracle_nf4_nearest(v);
    if ((k & 1) == 0)
      packed[k / 2] = (uint8_t)(packed[k / 2] | (idx << 4));
    else
      packed[k / 2] = (uint8_t)(packed[k / 2] | idx);
  }
}

/* Index of the nearest code2 entry to r: binary64 distances, ties -> lower. */
int oracle_code2_nearest(float r, const uint16_t code2[256]) {
  int best = 0;
  double bestd = fabs((double)r - (double)oracle_f16_to_f32(code2[0]));
  for (int i = 1; i < 256; ++i) {
    const double d = fabs((double)r - (double)oracle_f16_to_f32(code2[i]));
    if (d < bestd) {
      bestd = d;
      best = i;
    }
  }
  return best;
}

/* Double quantization of the first-level scales, [NF4-RPT] 1.2 and
 * [NF4-OPT] "第二层量化":
 *   offset      = mean of all absmax (binary64 sum group by group, /nb,
 *                 rounded to binary32);
 *   absmax2[g]  = binary16 of the largest |absmax[b] - offset| in group g
 *                 (groups of s2 consecutive blocks, the last may be partial);
 *   absmax_q[b] = nearest code2 index of (absmax[b] - offset) / absmax2[g]
 *                 (binary32 subtraction and division; 0 if absmax2 is 0).    */
void oracle_double_quant(const float* absmax, int64_t nb, int64_t s2,
                         const uint16_t code2[256], uint8_t* absmax_q,
                         uint16_t* absmax2, float* offset_out) {
  const int64_t ng = (nb + s2 - 1) / s2;
  double total = 0.0;
  for (int64_t g = 0; g < ng; ++g) {
    double part = 0.0;
    const int64_t end = (g + 1) * s2 < nb ? (g + 1) * s2 : nb;
    for (int64_t b = g * s2; b < end; ++b) part += (double)absmax[b];
    total += part;
  }
  const float offset = (nb > 0) ? (float)(total / (double)nb) : 0.0f;
  *offset_out = offset;
  for (int64_t g = 0; g < ng; ++g) {
    const int64_t end = (g + 1) * s2 < nb ? (g + 1) * s2 : nb;
    float m = 0.0f;
    for (int64_t b = g * s2; b < end; ++b) {
      const float d = fabsf(absmax[b] - offset);
      if (d > m) m = d;
    }
    absmax2[g] = oracle_f32_to_f16(m);
    const float a2 = oracle_f16_to_f32(absmax2[g]);
    for (int64_t b = g * s2; b < end; ++b) {
      const float r = (a2 == 0.0f) ? 0.0f : (absmax[b] - offset) / a2;
      absmax_q[b] = (uint8_t)oracle_code2_nearest(r, code2);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Dequantization, [NF4-RPT] 1.3:
 *   block b = k / bs, group g = b / s2,
 *   absmax_real = code2[absmax_q[b]] * absmax2[g] + offset   (two binary32
 *                 operations, multiply then add, no fusion),
 *   value       = NF4[idx(k)] * absmax_real                 (binary32),
 * with idx(k) the high nibble of byte k/2 for even k, the low nibble for odd
 * k ([NF4-RPT] 2.2).                                                         */
float oracle_block_scale(const uint8_t* absmax_q, const uint16_t* absmax2,
                         const uint16_t* code2, float offset, int64_t b, int64_t s2) {
  const float c = oracle_f16_to_f32(code2[absmax_q[b]]);
  const float a2 = oracle_f16_to_f32(absmax2[b / s2]);
  const float s1 = c * a2;
  return s1 + offset;
}

static int nibble_at(const uint8_t* packed, int64_t k) {
  const uint8_t byte = packed[k / 2];
  return (k & 1) ? (byte & 0x0f) : (byte >> 4);
}

/* binary32 values before the final 16-bit rounding (the GEMV's weights). */
void oracle_dequant_f32(const uint8_t* packed, const uint8_t* absmax_q,
                        const uint16_t* absmax2, const uint16_t* code2, float offset,
                        int64_t n, int64_t bs, int64_t s2, float* out) {
  for (int64_t k = 0; k < n; ++k) {
    const float s = oracle_block_scale(absmax_q, absmax2, code2, offset, k / bs, s2);
    out[k] = NF4_CODE[nibble_at(packed, k)] * s;
  }
}

/* The 16-bit output: dtype 0 = bfloat16, 1 = binary16, both RNE. */
void oracle_dequant(const uint8_t* packed, const uint8_t* absmax_q,
                    const uint16_t* absmax2, const uint16_t* code2, float offset,
                    int64_t n, int64_t bs, int64_t s2, int dtype, uint16_t* out) {
  for (int64_t k = 0; k < n; ++k) {
    const float s = oracle_block_scale(absmax_q, absmax2, code2, offset, k / bs, s2);
    const float v = NF4_CODE[nibble_at(packed, k)] * s;
    out[k] = dtype == 0 ? oracle_f32_to_bf16(v) : oracle_f32_to_f16(v);
  }
}

/* Same, for an arbitrary list of flat element indices (sampled checks on
 * large tensors). */
void oracle_dequant_at(const uint8_t* packed, const uint8_t* absmax_q,
                       const uint16_t* absmax2, const uint16_t* code2, float offset,
                       int64_t bs, int64_t s2, int dtype, const int64_t* idx,
                       int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) {
    const int64_t k = idx[i];
    const float s = oracle_block_scale(absmax_q, absmax2, code2, offset, k / bs, s2);
    const float v = NF4_CODE[nibble_at(packed, k)] * s;
    out[i] = dtype == 0 ? oracle_f32_to_bf16(v) : oracle_f32_to_f16(v);
  }
}

/* ------------------------------------------------------------------------ */
/* Decode GEMV with dequantization fused ([QTAX], fused kernel section):
 *   W is N x K row-major over the flattened quantized tensor (element
 *   (r, k) is flat index r*K + k), w_hat its binary32 dequantized value;
 *   y_ref[b][r] = sum_k w_hat[r][k] * x[b][k]   in binary64,
 *   s_abs[b][r] = sum_k |w_hat[r][k] * x[b][k]| in binary64,
 * with x given as bfloat16 bit patterns [batch][K].  Rows listed in `rows`
 * only (rows == NULL means all N rows); outputs are [batch][nrows].          */
void oracle_gemv(const uint8_t* packed, const uint8_t* absmax_q,
                 const uint16_t* absmax2, const uint16_t* code2, float offset,
                 int64_t N, int64_t K, int64_t bs, int64_t s2, const uint16_t* x,
                 int64_t batch, const int64_t* rows, int64_t nrows, double* y_ref,
                 double* s_abs) {
  const int64_t count = rows ? nrows : N;
  for (int64_t i = 0; i < count; ++i) {
    const int64_t r = rows ? rows[i] : i;
    for (int64_t b = 0; b < batch; ++b) {
      double acc = 0.0, acc_abs = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const int64_t flat = r * K + k;
        const float s = oracle_block_scale(absmax_q, absmax2, code2, offset, flat / bs, s2);
        const float w_hat = NF4_CODE[nibble_at(packed, flat)] * s;
        const double prod = (double)w_hat * (double)oracle_bf16_to_f32(x[b * K + k]);
        acc += prod;
        acc_abs += fabs(prod);
      }
      y_ref[b * count + i] = acc;
      s_abs[b * count + i] = acc_abs;
    }
  }
}

/* Magnitude GEMV for error bounds through chained layers:
 *   a[b][r] = sum_k |w_hat[r][k]| * e[b][k]   in binary64, e >= 0 given in
 * binary64 [batch][K]; outputs [batch][N].  A perturbation of the input by
 * at most e (elementwise) moves the exact product W_hat x by at most a.     */
void oracle_gemv_abs(const uint8_t* packed, const uint8_t* absmax_q,
                     const uint16_t* absmax2, const uint16_t* code2, float offset,
                     int64_t N, int64_t K, int64_t bs, int64_t s2, const double* e,
                     int64_t batch, double* a) {
  for (int64_t r = 0; r < N; ++r) {
    for (int64_t b = 0; b < batch; ++b) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const int64_t flat = r * K + k;
        const float s = oracle_block_scale(absmax_q, absmax2, code2, offset, flat / bs, s2);
        const float w_hat = NF4_CODE[nibble_at(packed, flat)] * s;
        acc += fabs((double)w_hat) * e[b * K + k];
      }
      a[b * N + r] = acc;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Output stage of a layer ([QTAX], fused kernel section: each binary32 row
 * sum is stored in the layer's 16-bit type and the layer's bias is added to
 * the stored row).  Types: 0 bfloat16, 1 binary16, 2 binary32.
 *   oracle_round_f64: the pattern of `dtype` nearest v (ties to even);
 *   oracle_decode:    the exact value of a pattern of `dtype`;
 *   oracle_gemv_output: v[b][i] = y_ref[b][i] + bias[r_i] in binary64, with
 *     the bias pattern widened exactly (bias == NULL: no bias; rows == NULL:
 *     r_i = i), and y_bits[b][i] = oracle_round_f64(v[b][i], dtype).        */
uint32_t oracle_round_f64(double v, int dtype) {
  if (dtype == 0) return oracle_f64_to_bf16(v);
  if (dtype == 1) return oracle_f64_to_f16(v);
  return oracle_f64_to_f32_bits(v);
}

double oracle_decode(uint32_t bits, int dtype) {
  if (dtype == 0) return (double)oracle_bf16_to_f32((uint16_t)bits);
  if (dtype == 1) return (double)oracle_f16_to_f32((uint16_t)bits);
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

void oracle_gemv_output(const double* y_ref, int64_t batch, int64_t count, const int64_t* rows,
                        const void* bias, int dtype, double* v, uint32_t* y_bits) {
  for (int64_t b = 0; b < batch; ++b) {
    for (int64_t i = 0; i < count; ++i) {
      const int64_t r = rows ? rows[i] : i;
      double bv = 0.0;
      if (bias) {
        const uint32_t bb = dtype == 2 ? ((const uint32_t*)bias)[r]
                                       : (uint32_t)((const uint16_t*)bias)[r];
        bv = oracle_decode(bb, dtype);
      }
      const double val = y_ref[b * count + i] + bv;
      v[b * count + i] = val;
      y_bits[b * count + i] = oracle_round_f64(val, dtype);
    }
  }
}
