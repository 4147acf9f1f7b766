/*
 * gq_oracle.c -- CPU oracle for per-token-group fp8 e4m3 quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct
 * statement of what the CUDA library computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load it; the product path
 * never does.  It shares no code, header, table or constant with the CUDA
 * library, and it includes nothing from it.
 *
 * The method (pytorch/ao pull-request pages):
 *   - "[moe training] use smaller block sizes for per group scaling kernels to
 *     improve perf" (#2668), intro: a kernel doing per-token-group scaling
 *     along dim0 -- the COLWISE variant: token groups are contiguous row
 *     ranges, one scale per (group, column).  The kernel arguments printed in
 *     the torch.compile failure report on the same page give the constants:
 *     fp8_dtype_max = 448.0, fp8_dtype_min = -448.0, EPS = 1e-12.
 *   - "[moe fp8 training] test and bench new faster method for per group
 *     rowwise scaling" (#2863), Summary: per-group ROWWISE scaling for the
 *     backward grad_weight GEMM -- groups are contiguous column ranges, one
 *     scale per (row, group) -- and the result is wanted transposed, so the
 *     fp8 output is written as A^T.
 * Further sections below: stacked expert weights along dim1 (#2863's PR
 * stack) and per row (#2668's PR stack), the mxfp8 cast along dim0 (#3114), and the grouped grad_weight
 * product of the two quantized operands (#2668's MoE fp8 training test).
 *
 * Per group g with token range [s_g, e_g) and each column (colwise) or row
 * (rowwise):
 *     amax  = max |x| over the group (0 for an empty group)
 *     scale = 448 / max(amax, 1e-12)                       IEEE fp32 division
 *     q     = e4m3( fp32(x * scale) )                       fp32 multiply, then
 *             round-to-nearest-even with saturation to +-448
 * The stored scale is the multiplier (448 / amax), not its reciprocal.
 *
 * Option round_scales_to_power_of_2 (a keyword argument of the same kernel
 * in #2668's failure report, True in that run): the scale becomes the power
 * of two at or below it, 2^floor(log2(scale)), before the multiply.
 *
 * Floating point: the precision is fixed to IEEE fp32 by the method, so the
 * scale and the product are computed in C `float` (FLT_EVAL_METHOD == 0 on
 * x86-64 and aarch64).  Build without -ffast-math and with
 * -ffp-contract=off.  The e4m3 encoder works in double, where every value it
 * touches is exact.
 *
 * Group bounds: offs[g] is the END offset of group g; group 0 starts at 0 and
 * group g at offs[g-1].  The contract is offs nondecreasing with values in
 * [0, extent]; to give out-of-contract offsets one defined meaning, each end
 * is taken as the running maximum of offs[0..g] clamped to [0, extent].
 * Elements past the last end belong to no group and are left untouched.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GQO_FP8_MAX 448.0f /* fp8_dtype_max in the kernel arguments  */
#define GQO_EPS 1e-12f     /* EPS in the kernel arguments             */

/* ---------------------------------------------------------------- bf16 --- */

/* A bf16 value is the top half of an IEEE binary32; widening is exact. */
float gqo_bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ---------------------------------------------------------------- e4m3 --- */

/*
 * OCP e4m3 ("fn") format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 holds the subnormals m * 2^-9; S.1111.111 is NaN;
 * there is no infinity; the largest finite magnitude, S.1111.110, is 448 --
 * the fp8_dtype_max the pages print.
 */
double gqo_e4m3_decode(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9); /* (m / 8) * 2^(1 - 7) */
  else
    mag = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Magnitudes of the 127 non-negative finite codes 0x00..0x7E, ascending. */
static double g_mag[127];
static int g_mag_ready = 0;

static void gqo_init_table(void) {
  int c;
  if (g_mag_ready) return;
  for (c = 0; c < 127; ++c) g_mag[c] = gqo_e4m3_decode((uint8_t)c);
  g_mag_ready = 1;
}

/*
 * Saturating round-to-nearest-even onto the e4m3 value set, from the
 * definition: find the two representable magnitudes that bracket |v|, take the
 * nearer one, and on an exact tie take the one whose code (hence mantissa) is
 * even.  |v| >= 448 saturates to 448 (clamping to [fp8_dtype_min,
 * fp8_dtype_max] before the cast).  The sign is kept, also on zero.  NaN is
 * outside the contract and maps to the NaN code.
 */
uint8_t gqo_e4m3_encode(float v) {
  uint32_t bits;
  uint8_t sign;
  double a, twice, mid;
  int lo, hi, c;
  gqo_init_table();
  memcpy(&bits, &v, sizeof bits);
  sign = (bits >> 31) ? 0x80 : 0x00;
  if (isnan(v)) return (uint8_t)(sign | 0x7F);
  a = fabs((double)v);
  if (a >= (double)GQO_FP8_MAX) return (uint8_t)(sign | 0x7E);
  /* invariant: g_mag[lo] <= a < g_mag[hi] */
  lo = 0;
  hi = 126;
  while (hi - lo > 1) {
    int m = (lo + hi) / 2;
    if (g_mag[m] <= a)
      lo = m;
    else
      hi = m;
  }
  /* |a - lo| vs |hi - a|  <=>  2a vs lo + hi; both sides are exact in double */
  twice = 2.0 * a;
  mid = g_mag[lo] + g_mag[hi];
  if (twice < mid)
    c = lo;
  else if (twice > mid)
    c = hi;
  else
    c = (lo % 2 == 0) ? lo : hi;
  return (uint8_t)(sign | c);
}

/* ------------------------------------------------------ scale, element --- */

/* scale = 448 / max(amax, 1e-12), IEEE fp32. */
float gqo_scale(float amax) {
  float d = amax > GQO_EPS ? amax : GQO_EPS;
  return GQO_FP8_MAX / d;
}

/* 2^floor(log2(scale)) for the positive finite scales gqo_scale returns:
 * frexp writes scale = m * 2^e with m in [0.5, 1), so floor(log2(scale)) is
 * e - 1. */
float gqo_scale_pow2(float amax) {
  int e;
  frexpf(gqo_scale(amax), &e);
  return ldexpf(1.0f, e - 1);
}

static float gqo_scale_opt(float amax, int pow2) {
  return pow2 ? gqo_scale_pow2(amax) : gqo_scale(amax);
}

/* q = e4m3(fp32(x * scale)). */
uint8_t gqo_quant(uint16_t x_bf16, float scale) {
  float v = gqo_bf16_to_float(x_bf16) * scale;
  return gqo_e4m3_encode(v);
}

/* ------------------------------------------------------------- groups --- */

static void gqo_group_bounds(const int32_t* offs, int32_t n_groups,
                             int64_t extent, int64_t* start, int64_t* end) {
  int64_t prev = 0;
  int32_t g;
  for (g = 0; g < n_groups; ++g) {
    int64_t e = offs[g];
    if (e < prev) e = prev;
    if (e > extent) e = extent;
    start[g] = prev;
    end[g] = e;
    prev = e;
  }
}

/* ------------------------------------------------------------ colwise --- */

/*
 * x: bf16 bits, (M, K) row-major.  Groups run along dim0 (rows).
 * q: e4m3 codes, (M, K) row-major.  scales: fp32, (n_groups, K) row-major.
 * Returns 0, or -1 on invalid arguments.
 */
int gqo_colwise_ex(const uint16_t* x, int64_t M, int64_t K, const int32_t* offs,
                   int32_t n_groups, int pow2, uint8_t* q, float* scales) {
  int64_t *start, *end;
  float* amax;
  int32_t g;
  if (M < 0 || K < 0 || n_groups < 1 || offs == NULL) return -1;
  if ((M * K > 0) && (x == NULL || q == NULL)) return -1;
  if (K > 0 && scales == NULL) return -1;
  start = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_groups);
  end = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_groups);
  amax = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
  if (!start || !end || !amax) {
    free(start);
    free(end);
    free(amax);
    return -1;
  }
  gqo_group_bounds(offs, n_groups, M, start, end);
  for (g = 0; g < n_groups; ++g) {
    int64_t r, k;
    for (k = 0; k < K; ++k) amax[k] = 0.0f;
    for (r = start[g]; r < end[g]; ++r)
      for (k = 0; k < K; ++k) {
        float a = fabsf(gqo_bf16_to_float(x[r * K + k]));
        if (a > amax[k]) amax[k] = a;
      }
    for (k = 0; k < K; ++k) scales[(int64_t)g * K + k] = gqo_scale_opt(amax[k], pow2);
    for (r = start[g]; r < end[g]; ++r)
      for (k = 0; k < K; ++k)
        q[r * K + k] = gqo_quant(x[r * K + k], scales[(int64_t)g * K + k]);
  }
  free(start);
  free(end);
  free(amax);
  return 0;
}

/* ---------------------------------------------------------- rowwise_t --- */

/*
 * a: bf16 bits, (N, Mg) row-major.  Groups run along dim1 (the Mg token
 * columns).  qt: e4m3 codes, (Mg, N) row-major, qt[m][n] = q(a[n][m]) -- the
 * transpose.  scales: fp32, (N, n_groups) row-major.
 * Returns 0, or -1 on invalid arguments.
 */
int gqo_rowwise_t_ex(const uint16_t* a, int64_t N, int64_t Mg,
                     const int32_t* offs, int32_t n_groups, int pow2, uint8_t* qt,
                     float* scales) {
  int64_t *start, *end;
  int64_t n;
  if (N < 0 || Mg < 0 || n_groups < 1 || offs == NULL) return -1;
  if ((N * Mg > 0) && (a == NULL || qt == NULL)) return -1;
  if (N > 0 && scales == NULL) return -1;
  start = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_groups);
  end = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_groups);
  if (!start || !end) {
    free(start);
    free(end);
    return -1;
  }
  gqo_group_bounds(offs, n_groups, Mg, start, end);
  for (n = 0; n < N; ++n) {
    int32_t g;
    for (g = 0; g < n_groups; ++g) {
      float amax = 0.0f, s;
      int64_t m;
      for (m = start[g]; m < end[g]; ++m) {
        float v = fabsf(gqo_bf16_to_float(a[n * Mg + m]));
        if (v > amax) amax = v;
      }
      s = gqo_scale_opt(amax, pow2);
      scales[n * n_groups + g] = s;
      for (m = start[g]; m < end[g]; ++m)
        qt[m * N + n] = gqo_quant(a[n * Mg + m], s);
    }
  }
  free(start);
  free(end);
  return 0;
}

/* -------------------------------------------------- expert weights --- */

/*
 * Stacked expert weights w: bf16 bits, (E, K, N) row-major.  For each expert
 * e and column n the amax is taken over the K rows of that expert (a
 * reduction along dim1, the "fused reduction kernel along dim1 for 3d expert
 * weights" of the #2863 page's PR stack); q has w's layout, scales are
 * (E, N) row-major.  Returns 0, or -1 on invalid arguments.
 */
int gqo_expert_dim1(const uint16_t* w, int64_t E, int64_t K, int64_t N, int pow2,
                    uint8_t* q, float* scales) {
  int64_t e, k, n;
  if (E < 1 || K < 0 || N < 0) return -1;
  if ((E * K * N > 0) && (w == NULL || q == NULL)) return -1;
  if (N > 0 && scales == NULL) return -1;
  for (e = 0; e < E; ++e)
    for (n = 0; n < N; ++n) {
      float amax = 0.0f, s;
      for (k = 0; k < K; ++k) {
        float a = fabsf(gqo_bf16_to_float(w[(e * K + k) * N + n]));
        if (a > amax) amax = a;
      }
      s = gqo_scale_opt(amax, pow2);
      scales[e * N + n] = s;
      for (k = 0; k < K; ++k)
        q[(e * K + k) * N + n] = gqo_quant(w[(e * K + k) * N + n], s);
    }
  return 0;
}

/*
 * Stacked expert weights w: bf16 bits, (E, N, K) row-major, scaled per row:
 * one scale for each expert e and row n, the amax taken over that row's K
 * elements (the "fp8 rowwise kernels for expert weights" of the #2668
 * page's PR stack, #2696); q has w's layout, scales are (E, N) row-major.
 * Returns 0, or -1 on invalid arguments.
 */
int gqo_expert_rowwise(const uint16_t* w, int64_t E, int64_t N, int64_t K, int pow2,
                       uint8_t* q, float* scales) {
  int64_t e, n, k;
  if (E < 1 || N < 0 || K < 0) return -1;
  if ((E * N * K > 0) && (w == NULL || q == NULL)) return -1;
  if (N > 0 && scales == NULL) return -1;
  for (e = 0; e < E; ++e)
    for (n = 0; n < N; ++n) {
      const int64_t row = (e * N + n) * K;
      float amax = 0.0f, s;
      for (k = 0; k < K; ++k) {
        float a = fabsf(gqo_bf16_to_float(w[row + k]));
        if (a > amax) amax = a;
      }
      s = gqo_scale_opt(amax, pow2);
      scales[e * N + n] = s;
      for (k = 0; k < K; ++k) q[row + k] = gqo_quant(w[row + k], s);
    }
  return 0;
}

/* ------------------------------------------------------ mxfp8 dim0 --- */

/*
 * mxfp8 cast along dim0 (the "dim0_mxfp8_floor" cast benchmark and the RCEIL
 * scaling type of the pytorch/ao "fix mxfp8 a2a bench script; set mxfp8 a2a
 * scaling type to RCEIL" page): every 32 consecutive elements of a row form
 * a block that shares one power-of-two scale 2^E, stored as an e8m0 byte
 * E + 127; elements are e4m3(fp32(x * 2^-E)).
 *   FLOOR (mode 0): E = floor(log2(amax)) - 8, 8 being the exponent of
 *                   e4m3's largest value (448 = 1.75 * 2^8);
 *   RCEIL (mode 1): E = ceil(log2(v)), v = fp32(amax / 448), the power of
 *                   two at or above the block's amax over 448.
 * E is clamped to [-127, 127]; a block whose amax is 0 gets E = -127 (byte
 * 0) and all-zero elements.
 */
static int gqo_mx_exponent(float amax, int mode) {
  int e, E;
  float v;
  if (amax == 0.0f) return -127;
  if (mode == 0) {
    frexpf(amax, &e);  /* amax = m * 2^e, m in [0.5, 1): floor(log2) = e - 1 */
    E = (e - 1) - 8;
  } else {
    v = amax / GQO_FP8_MAX;
    /* v = m * 2^e with m in [0.5, 1): ceil(log2 v) is e - 1 when m == 0.5
     * (v a power of two), else e */
    E = (frexpf(v, &e) == 0.5f) ? e - 1 : e;
  }
  if (E < -127) E = -127;
  if (E > 127) E = 127;
  return E;
}

/* x: bf16 bits (M, K) row-major, K % 32 == 0.  q: e4m3 (M, K); scales:
 * e8m0 bytes (M, K / 32).  Returns 0, or -1 on invalid arguments. */
int gqo_mxfp8_dim0(const uint16_t* x, int64_t M, int64_t K, int mode, uint8_t* q,
                   uint8_t* scales) {
  int64_t r, b, i, nb;
  if (M < 0 || K < 0 || K % 32 != 0 || (mode != 0 && mode != 1)) return -1;
  if (M * K > 0 && (x == NULL || q == NULL || scales == NULL)) return -1;
  nb = K / 32;
  for (r = 0; r < M; ++r)
    for (b = 0; b < nb; ++b) {
      const uint16_t* xb = x + r * K + b * 32;
      float amax = 0.0f, f;
      int E;
      for (i = 0; i < 32; ++i) {
        float a = fabsf(gqo_bf16_to_float(xb[i]));
        if (a > amax) amax = a;
      }
      E = gqo_mx_exponent(amax, mode);
      scales[r * nb + b] = (uint8_t)(E + 127);
      f = ldexpf(1.0f, -E);
      for (i = 0; i < 32; ++i) q[r * K + b * 32 + i] = gqo_e4m3_encode(gqo_bf16_to_float(xb[i]) * f);
    }
  return 0;
}

/* ------------------------------------------------ grouped grad_weight --- */

/*
 * The consumer of both quantized operands: the grad_weight GEMM of the MoE
 * backward pass, one product per token group ("[moe training] use smaller
 * block sizes for per group scaling kernels to improve perf" (#2668), MoE
 * fp8 training test: grad_weight = grad_output_t @ input, token groups
 * aligned to 16).  With
 *   qa_t: e4m3 codes (T, N) row-major -- the rowwise_t output, grad_output_t
 *         as a column-major (N, T) operand; sa: fp32 (N, G), its scales;
 *   qx:   e4m3 codes (T, K) row-major -- the colwise output of the layer
 *         input; sx: fp32 (G, K), its scales;
 * the result for group g = [s_g, e_g) is
 *   out[g][n][k] = ( sum over t in g of dec(qa_t[t][n]) * dec(qx[t][k]) )
 *                  / ( sa[n][g] * sx[g][k] ),
 * each quantized factor divided by the multiplier that produced it.
 *
 * Precision: double.  A product of two e4m3 values is exact (8 significant
 * bits, a multiple of 2^-18, below 2^17.7), and so is every partial sum for
 * T < 2^17 tokens (at most 53 bits); sa * sx is exact (two 24-bit
 * significands); the quotient is the only rounding.  absum (may be NULL)
 * receives the same quotient of the sum of |products|, the scale against
 * which an fp32 accumulation error is measured.  An empty group gives zeros;
 * tokens past the last end belong to no group.  Returns 0, or -1 on invalid
 * arguments.
 */
int gqo_grouped_wgrad(const uint8_t* qa_t, const float* sa, const uint8_t* qx,
                      const float* sx, int64_t T, int64_t N, int64_t K,
                      const int32_t* offs, int32_t n_groups, double* out, double* absum) {
  double dec[256];
  int64_t *start, *end;
  double *acc, *mag;
  int64_t t, n, k;
  int32_t g;
  int c;
  if (T < 0 || N < 0 || K < 0 || n_groups < 1 || offs == NULL) return -1;
  if (N * K > 0 && (out == NULL || sa == NULL || sx == NULL)) return -1;
  if (T * N > 0 && qa_t == NULL) return -1;
  if (T * K > 0 && qx == NULL) return -1;
  for (c = 0; c < 256; ++c) dec[c] = gqo_e4m3_decode((uint8_t)c);
  start = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_groups);
  end = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_groups);
  acc = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
  mag = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
  if (!start || !end || !acc || !mag) {
    free(start);
    free(end);
    free(acc);
    free(mag);
    return -1;
  }
  gqo_group_bounds(offs, n_groups, T, start, end);
  for (g = 0; g < n_groups; ++g) {
    for (n = 0; n < N * K; ++n) acc[n] = mag[n] = 0.0;
    for (t = start[g]; t < end[g]; ++t)
      for (n = 0; n < N; ++n) {
        const double a = dec[qa_t[t * N + n]];
        for (k = 0; k < K; ++k) {
          const double p = a * dec[qx[t * K + k]];
          acc[n * K + k] += p;
          mag[n * K + k] += fabs(p);
        }
      }
    for (n = 0; n < N; ++n)
      for (k = 0; k < K; ++k) {
        const double d = (double)sa[n * n_groups + g] * (double)sx[(int64_t)g * K + k];
        out[((int64_t)g * N + n) * K + k] = acc[n * K + k] / d;
        if (absum) absum[((int64_t)g * N + n) * K + k] = mag[n * K + k] / d;
      }
  }
  free(start);
  free(end);
  free(acc);
  free(mag);
  return 0;
}

/* The plain method: scales exactly 448 / max(amax, 1e-12). */
int gqo_colwise(const uint16_t* x, int64_t M, int64_t K, const int32_t* offs,
                int32_t n_groups, uint8_t* q, float* scales) {
  return gqo_colwise_ex(x, M, K, offs, n_groups, 0, q, scales);
}

int gqo_rowwise_t(const uint16_t* a, int64_t N, int64_t Mg, const int32_t* offs,
                  int32_t n_groups, uint8_t* qt, float* scales) {
  return gqo_rowwise_t_ex(a, N, Mg, offs, n_groups, 0, qt, scales);
}

/* ----------------------------------------------- array helpers (tests) --- */

void gqo_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = gqo_e4m3_encode(v[i]);
}

void gqo_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = gqo_e4m3_decode(c[i]);
}

void gqo_scale_array(const float* amax, int64_t n, float* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = gqo_scale(amax[i]);
}

void gqo_scale_pow2_array(const float* amax, int64_t n, float* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = gqo_scale_pow2(amax[i]);
}

void gqo_quant_array(const uint16_t* x, const float* scale, int64_t n,
                     uint8_t* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = gqo_quant(x[i], scale[i]);
}
