/*
 * rlref.c — plain fp64 CPU oracle for the fused RL policy-loss step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it follows.  The three pages on RL.cu ("LLM Reinforcement Learning in
 * Pure CUDA") describe a fused PPO/GRPO update that turns per-token
 * vocabulary log-probabilities into a clipped-surrogate loss with a KL
 * penalty and an entropy bonus (ainews.cool RL.cu article, section
 * "技术深度解析" / technical deep dive, bullet "PPO 更新内核"; the KL penalty
 * and reward normalisation in the paragraph after its benchmark table).  The
 * pages print no formula, so each step here is the textbook definition
 * written out literally, in double precision, one row at a time, with no
 * blocking, fusion or reordering:
 *
 *   row statistics    M = max_v z_v, S = sum_v exp(z_v - M), lse = M + ln S,
 *                     logp = z_y - lse, H = -sum_v p_v ln p_v
 *   logits gradient   dz_v = scale * [ g (p_v - [v == y]) + c (p_v (ln p_v + H)) ]
 *
 * The per-token objective between the two (ratio, clip, KL, aggregation)
 * is written in numpy in oracle/__init__.py.
 *
 * Element formats.  Inputs are decoded exactly (bf16, fp16 and fp32 all embed
 * in double); outputs are rounded once from double, round-to-nearest-even,
 * with subnormals kept.  The decoders and the rounder are written from the
 * IEEE 754 binary16 and bfloat16 layouts, not from any library.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { RLREF_F32 = 0, RLREF_BF16 = 1, RLREF_F16 = 2, RLREF_F64 = 3 };

static size_t elem_size(int dtype) {
  switch (dtype) {
    case RLREF_F32: return 4;
    case RLREF_BF16: return 2;
    case RLREF_F16: return 2;
    case RLREF_F64: return 8;
  }
  return 0;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double decode_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25);  /* (1 + m/2^10) * 2^(e-15) */
  return sign ? -v : v;
}

static double load_elem(const void* base, int dtype, size_t i) {
  switch (dtype) {
    case RLREF_F32: return (double)((const float*)base)[i];
    case RLREF_BF16: return decode_bf16(((const uint16_t*)base)[i]);
    case RLREF_F16: return decode_f16(((const uint16_t*)base)[i]);
    case RLREF_F64: return ((const double*)base)[i];
  }
  return NAN;
}

/*
 * Round x to the nearest value of a binary format with `p` significand bits
 * (implicit bit included), minimum normal exponent `emin` and maximum
 * exponent `emax`; ties go to the even significand.  Values past the largest
 * finite number by half an ulp or more become infinity.
 */
static double round_to_format(double x, int p, int emin, int emax) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double a = fabs(x);
  int k;
  frexp(a, &k);                 /* a = f * 2^k with f in [0.5, 1): leading bit at 2^(k-1) */
  int lead = k - 1;
  if (lead < emin) lead = emin; /* subnormal range: fixed quantum */
  double q = ldexp(1.0, lead - (p - 1));
  double n = a / q;             /* exact: q is a power of two */
  double r = nearbyint(n);      /* default rounding mode: to nearest, ties to even */
  double y = r * q;
  double maxfin = ldexp(2.0 - ldexp(1.0, -(p - 1)), emax);
  if (y > maxfin) y = INFINITY;
  return x < 0 ? -y : y;
}

static uint16_t encode_bf16(double x) {
  if (isnan(x)) return 0x7fc0;
  float f = (float)round_to_format(x, 8, -126, 127); /* exact in binary32 */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

static uint16_t encode_f16(double x) {
  if (isnan(x)) return 0x7e00;
  double y = round_to_format(x, 11, -14, 15);
  uint16_t sign = signbit(y) ? 0x8000 : 0;
  double a = fabs(y);
  if (isinf(a)) return sign | 0x7c00;
  if (a == 0.0) return sign;
  if (a < ldexp(1.0, -14))                       /* subnormal */
    return sign | (uint16_t)(a / ldexp(1.0, -24));
  int k;
  double f = frexp(a, &k);                       /* a = f * 2^k, f in [0.5,1) */
  int e = k - 1 + 15;                            /* biased exponent of the leading bit */
  uint16_t m = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
  return sign | (uint16_t)(e << 10) | m;
}

static void store_elem(void* base, int dtype, size_t i, double x) {
  switch (dtype) {
    case RLREF_F32: ((float*)base)[i] = (float)x; break;   /* C conversion: correctly rounded, RNE */
    case RLREF_BF16: ((uint16_t*)base)[i] = encode_bf16(x); break;
    case RLREF_F16: ((uint16_t*)base)[i] = encode_f16(x); break;
    case RLREF_F64: ((double*)base)[i] = x; break;
  }
}

/* Exact decode of n elements to double. */
void rlref_decode(const void* src, int dtype, long long n, double* out) {
  for (long long i = 0; i < n; ++i) out[i] = load_elem(src, dtype, (size_t)i);
}

/* Round n doubles once to `dtype` (RNE, subnormals kept). */
void rlref_encode(const double* src, long long n, int dtype, void* out) {
  for (long long i = 0; i < n; ++i) store_elem(out, dtype, (size_t)i, src[i]);
}

/* Number of valid tokens: the count of nonzero mask bytes. */
long long rlref_count(const unsigned char* mask, long long n) {
  long long N = 0;
  for (long long i = 0; i < n; ++i) N += mask[i] != 0;
  return N;
}

/*
 * Row statistics (log-softmax over the vocabulary) for rows [row0, row1).
 * For a row with mask 0 all three outputs are 0 and its logits are not read.
 * A sampled id outside [0, V) gives logp = NaN.
 */
void rlref_row_stats(const void* logits, int dtype, long long ld, long long V,
                     const long long* ids, const unsigned char* mask,
                     long long row0, long long row1,
                     double* lse_out, double* logp_out, double* ent_out) {
  double* z = (double*)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
  size_t es = elem_size(dtype);
  for (long long r = row0; r < row1; ++r) {
    if (!mask[r]) { lse_out[r] = 0.0; logp_out[r] = 0.0; ent_out[r] = 0.0; continue; }
    const char* row = (const char*)logits + (size_t)r * (size_t)ld * es;
    for (long long v = 0; v < V; ++v) z[v] = load_elem(row, dtype, (size_t)v);
    double M = -INFINITY;
    for (long long v = 0; v < V; ++v) if (z[v] > M) M = z[v];
    double S = 0.0;
    for (long long v = 0; v < V; ++v) S += exp(z[v] - M);
    double lse = M + log(S);
    double H = 0.0;
    for (long long v = 0; v < V; ++v) {
      double lp = z[v] - lse;
      double p = exp(lp);
      if (p > 0.0) H -= p * lp;     /* 0 * log 0 = 0 */
    }
    long long y = ids[r];
    lse_out[r] = lse;
    logp_out[r] = (y >= 0 && y < V) ? z[y] - lse : NAN;
    ent_out[r] = H;
  }
  free(z);
}

/*
 * Gradient of the loss with respect to the logits of row r, for the rows
 * listed in rows[0..n_rows):
 *   dz_v = scale_r * [ g_r (p_v - [v == y_r]) + c_ent p_v (ln p_v + H_r) ]
 * with p_v = exp(z_v - lse_r).  scale_r already holds grad_scale * m_r / N
 * (0 for a masked row, which then writes an all-zero row without reading its
 * logits).  Row i of `out` (stride out_ld elements, format out_dtype) receives
 * the row rows[i]; each value is rounded once from double.
 */
void rlref_dlogits_rows(const void* logits, int dtype, long long ld, long long V,
                        const long long* ids, const long long* rows, long long n_rows,
                        const double* lse, const double* ent, const double* g,
                        const double* scale, double c_ent,
                        int out_dtype, void* out, long long out_ld) {
  size_t es = elem_size(dtype), os = elem_size(out_dtype);
  for (long long i = 0; i < n_rows; ++i) {
    long long r = rows[i];
    char* orow = (char*)out + (size_t)i * (size_t)out_ld * os;
    if (scale[i] == 0.0) {
      for (long long v = 0; v < V; ++v) store_elem(orow, out_dtype, (size_t)v, 0.0);
      continue;
    }
    const char* row = (const char*)logits + (size_t)r * (size_t)ld * es;
    long long y = ids[r];
    for (long long v = 0; v < V; ++v) {
      double lp = load_elem(row, dtype, (size_t)v) - lse[i];
      double p = exp(lp);
      double ent_term = (p > 0.0) ? p * (lp + ent[i]) : 0.0;
      double d = scale[i] * (g[i] * (p - (v == y ? 1.0 : 0.0)) + c_ent * ent_term);
      store_elem(orow, out_dtype, (size_t)v, d);
    }
  }
}
