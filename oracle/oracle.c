/*
 * Oracle for the LLM.int8() mixed-precision decomposition linear.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain CPU statement of
 * what the CUDA path computes.  Only the test suite, the package's smoke
 * check and the CPU-baseline leg of the benchmark may load it.  It shares no
 * code with the CUDA path and the CUDA path never calls it.
 *
 * What the method computes, and where it is stated:
 *  - outliers are whole feature dimensions (columns of X) whose values are
 *    large; they are computed in 16-bit ("Hugging Face Quantization with
 *    bitsandbytes: 4-bit & 8-bit Models Explained", section 2 "LLM.int8():
 *    Quantizing Without Degrading Large Models");
 *  - the cut-off is llm_int8_threshold, default 6.0 (same page, section 3
 *    "Configuring 8-Bit Loading");
 *  - the bulk is quantized vector-wise to 8 bits and multiplied in int8, the
 *    outliers go through a 16-bit matrix multiplication ("bitsandbytes:
 *    GPU-Accelerated Inference and Training at Lower Bit Depths", section
 *    "How LLM.int8() quantizes weights and activations"; "Shrink LLMs to
 *    4-bit and train them anyway", "The interesting bit");
 *  - the int8 result is converted back to 16-bit only at the end (section 2
 *    of the Hugging Face page).
 * Readings where the pages are silent (all listed in the design notes):
 *  - a column is an outlier when ANY row has |x| >= tau (>=, not >);
 *  - row scale sx[t] = max |X[t,k]| over non-outlier k; weight scale
 *    sw[n] = max_k |W[n,k]| over all k (per output channel);
 *  - code q = rint(fl32(127*x) / a) in IEEE fp32, ties to even; a = 0 gives 0;
 *  - Y = fp16_rne(acc*sx*sw/127^2 + sum_j X[t,O_j]*W[n,O_j]), evaluated here
 *    in double, one final rounding to fp16;
 *  - the outlier weights are the fp16 weights W16, not dequantized codes; with
 *    W16 absent (only the int8 weight kept, half of fp16's bytes: Hugging
 *    Face page, "Quick Comparison" table; bitsandbytes GPU page, section
 *    "Why quantization matters for LLM deployment") they are the codes
 *    dequantized, Wq[n,k] * sw[n] / 127, exact real values carried in
 *    double;
 *  - an optional fp16 bias b[n] (the layer is a drop-in replacement for
 *    PyTorch's Linear: bitsandbytes GPU page, section "How LLM.int8()
 *    quantizes weights and activations") is added before the one rounding:
 *    Y = fp16_rne(acc*sx*sw/127^2 + sum_j X[t,O_j]*W[n,O_j] + b[n]).
 *
 * X, W16, the bias and Y are fp16, or all bf16 (the compute dtype the pages
 * prefer where the hardware supports it: Hugging Face page, section 5); the
 * arithmetic is the same, only the 16-bit format of inputs and output changes
 * -- except that bf16 codes scale x and a by one power of two first, since
 * bf16's range lets 127 x overflow fp32 (the code itself is unchanged).
 *
 * Codes are decided in fp32 because the kernel decides them in fp32; the
 * tests pin this rule against exact rational rounding.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -shared -fPIC
 * (oracle/build_oracle.py).
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_RANGE 1 /* an int32 accumulator would overflow */
#define ORC_ERR_ARG 2

/* Threads the OpenMP loops below use (for reporting a CPU baseline). */
int orc_num_threads(void) { return omp_get_max_threads(); }

/* ---- fp16 <-> double, written from the IEEE 754 binary16 definition ---- */

double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1.m) * 2^(e-15) */
  return sign ? -v : v;
}

/* Round a double to binary16, nearest-even, in one step (no float detour). */
uint16_t orc_double_to_half(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return 0x7e00;
  if (a >= 65520.0) return sign | 0x7c00; /* 65520 is the tie between 65504 and 2^16 */
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: quantum 2^-24 */
    double n = rint(a * 16777216.0); /* exact scaling by 2^24 */
    return sign | (uint16_t)n;      /* n == 1024 gives the smallest normal */
  }
  int e;
  frexp(a, &e);    /* a = f * 2^e, f in [0.5, 1) */
  int E = e - 1;   /* a in [2^E, 2^(E+1)) */
  double n = rint(ldexp(a, 10 - E)); /* significand in units of 2^(E-10), in [1024, 2048] */
  if (n >= 2048.0) {
    n = 1024.0;
    E += 1;
  }
  if (E + 15 >= 31) return sign | 0x7c00;
  return sign | (uint16_t)(((E + 15) << 10) | ((int)n - 1024));
}

/* ---- bfloat16 <-> double, from the format's definition: 1 sign bit, 8
 * exponent bits (bias 127), 7 fraction bits; the compute dtype the pages
 * prefer where the hardware has it (Hugging Face page, section 5 "Storage
 * Precision vs. Compute Precision") ---- */

double orc_bf16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int m = h & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)m, -133); /* subnormal: m * 2^-133 */
  else if (e == 255)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(128 + m), e - 134); /* (1.m) * 2^(e-127) */
  return sign ? -v : v;
}

/* Round a double to bfloat16, nearest-even, in one step. */
uint16_t orc_double_to_bf16(double v) {
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return 0x7fc0;
  if (a >= ldexp(511.0, 119)) return sign | 0x7f80; /* tie between the largest finite and 2^128 */
  if (a < ldexp(1.0, -126)) {
    /* subnormal range: quantum 2^-133 */
    double n = rint(ldexp(a, 133));
    return sign | (uint16_t)n; /* n == 128 gives the smallest normal */
  }
  int e;
  frexp(a, &e);
  int E = e - 1; /* a in [2^E, 2^(E+1)) */
  double n = rint(ldexp(a, 7 - E)); /* significand in units of 2^(E-7), in [128, 256] */
  if (n >= 256.0) {
    n = 128.0;
    E += 1;
  }
  if (E + 127 >= 255) return sign | 0x7f80;
  return sign | (uint16_t)(((E + 127) << 7) | ((int)n - 128));
}

/* The 16-bit element format of X, W16, the bias and Y: 0 fp16, 1 bf16. */
static double elem_to_double(uint16_t b, int fmt) {
  return fmt ? orc_bf16_to_double(b) : orc_half_to_double(b);
}
static uint16_t double_to_elem(double v, int fmt) {
  return fmt ? orc_double_to_bf16(v) : orc_double_to_half(v);
}

/* ---- vector-wise code: q = rint(fl32(127*x) / a), in fp32 ---- */
static int8_t code_of(float x, float a) {
  if (a == 0.0f) return 0;
  float num = 127.0f * x; /* exact for fp16 and bf16 x */
  float q = rintf(num / a);
  return (int8_t)q;
}

/* The same code for bf16 x and a, whose range (2^-133 .. 2^128) lets 127 x
 * and the quotient leave fp32's: x and a are first scaled by the same power
 * of two (exact; the code 127 x / a is unchanged) so that a lies in [1, 2).
 * A value whose scaled form underflows has a code of 0 either way. */
static int8_t code_of_scaled(float x, float a) {
  if (a == 0.0f) return 0;
  int e;
  frexpf(a, &e); /* a = f * 2^e, f in [0.5, 1) */
  return code_of(ldexpf(x, 1 - e), ldexpf(a, 1 - e));
}

static int8_t code_fmt(float x, float a, int fmt) {
  return fmt ? code_of_scaled(x, a) : code_of(x, a);
}

/* S1: per-output-channel absmax scale and int8 codes of the weight.
 * "quantizes weights on the fly as the model loads" (page "bitsandbytes",
 * d-central glossary); row-wise / per output channel. */
int orc_quantize_weight(const uint16_t *W16, int64_t N, int64_t K, int8_t *Wq,
                        float *sw, int fmt) {
  if (N < 0 || K < 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; n++) {
    float a = 0.0f;
    for (int64_t k = 0; k < K; k++) {
      float x = fabsf((float)elem_to_double(W16[n * K + k], fmt));
      if (x > a) a = x;
    }
    sw[n] = a;
    for (int64_t k = 0; k < K; k++)
      Wq[n * K + k] = code_fmt((float)elem_to_double(W16[n * K + k], fmt), a, fmt);
  }
  return ORC_OK;
}

/* S2: outlier feature columns.  Column k is an outlier when some row t has
 * |X[t,k]| >= tau.  O is ascending; *nO receives |O|. */
int orc_outlier_columns(const uint16_t *X, int64_t T, int64_t K, float tau,
                        int32_t *O, int32_t *nO, int fmt) {
  if (T < 0 || K < 0) return ORC_ERR_ARG;
  int32_t n = 0;
  for (int64_t k = 0; k < K; k++) {
    int hit = 0;
    for (int64_t t = 0; t < T && !hit; t++) {
      float x = fabsf((float)elem_to_double(X[t * K + k], fmt));
      if (x >= tau) hit = 1;
    }
    if (hit) O[n++] = (int32_t)k;
  }
  *nO = n;
  return ORC_OK;
}

/* S3: row scales over the non-outlier columns, int8 codes (0 in outlier
 * columns), and the fp16 outlier block XO[t, j] = X[t, O[j]] (T x nO). */
int orc_quantize_activations(const uint16_t *X, int64_t T, int64_t K,
                             const int32_t *O, int32_t nO, int8_t *Xq,
                             float *sx, uint16_t *XO, int fmt) {
  if (T < 0 || K < 0 || nO < 0) return ORC_ERR_ARG;
  /* column flags from the list */
  unsigned char *flag_buf = (unsigned char *)calloc((size_t)(K > 0 ? K : 1), 1);
  if (!flag_buf) return ORC_ERR_ARG;
  for (int32_t j = 0; j < nO; j++) flag_buf[O[j]] = 1;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; t++) {
    float a = 0.0f;
    for (int64_t k = 0; k < K; k++) {
      if (flag_buf[k]) continue;
      float x = fabsf((float)elem_to_double(X[t * K + k], fmt));
      if (x > a) a = x;
    }
    sx[t] = a;
    for (int64_t k = 0; k < K; k++)
      Xq[t * K + k] =
          flag_buf[k] ? 0 : code_fmt((float)elem_to_double(X[t * K + k], fmt), a, fmt);
    if (XO)
      for (int32_t j = 0; j < nO; j++) XO[t * nO + j] = X[t * K + O[j]];
  }
  free(flag_buf);
  return ORC_OK;
}

/* S4: acc[r, n] = sum_k Xq[rows[r], k] * Wq[n, k], exact, checked to fit int32. */
int orc_int8_matmul_rows(const int8_t *Xq, const int8_t *Wq, int64_t T, int64_t N,
                         int64_t K, const int64_t *rows, int64_t nrows,
                         int32_t *acc) {
  int bad = 0;
  (void)T;
#pragma omp parallel for collapse(2) schedule(static) reduction(| : bad)
  for (int64_t r = 0; r < nrows; r++) {
    for (int64_t n = 0; n < N; n++) {
      const int8_t *x = Xq + rows[r] * K;
      const int8_t *w = Wq + n * K;
      int64_t s = 0;
      for (int64_t k = 0; k < K; k++) s += (int64_t)x[k] * (int64_t)w[k];
      if (s > INT32_MAX || s < INT32_MIN) bad = 1;
      acc[r * N + n] = (int32_t)s;
    }
  }
  return bad ? ORC_ERR_RANGE : ORC_OK;
}

/* S5: out[r, n] = sum_j X[rows[r], O[j]] * W16[n, O[j]] in double (16-bit
 * operands, each product exact in double). */
void orc_outlier_matmul_rows(const uint16_t *X, const uint16_t *W16, int64_t T,
                             int64_t N, int64_t K, const int32_t *O, int32_t nO,
                             const int64_t *rows, int64_t nrows, double *out, int fmt) {
  (void)T;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t r = 0; r < nrows; r++) {
    for (int64_t n = 0; n < N; n++) {
      double s = 0.0;
      for (int32_t j = 0; j < nO; j++)
        s += elem_to_double(X[rows[r] * K + O[j]], fmt) *
             elem_to_double(W16[n * K + O[j]], fmt);
      out[r * N + n] = s;
    }
  }
}

/* S5 without W16: the outlier weights dequantized from the int8 codes,
 * w = Wq[n,k] * sw[n] / 127, then the same 16-bit-input product. */
void orc_outlier_matmul_rows_wq(const uint16_t *X, const int8_t *Wq, const float *sw,
                                int64_t N, int64_t K, const int32_t *O, int32_t nO,
                                const int64_t *rows, int64_t nrows, double *out, int fmt) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t r = 0; r < nrows; r++) {
    for (int64_t n = 0; n < N; n++) {
      double s = 0.0;
      for (int32_t j = 0; j < nO; j++) {
        double w = (double)Wq[n * K + O[j]] * (double)sw[n] / 127.0;
        s += elem_to_double(X[rows[r] * K + O[j]], fmt) * w;
      }
      out[r * N + n] = s;
    }
  }
}

/* S6: Y = fp16( acc * sx * sw / 127^2 + out ).  acc*sx*sw is exact in double
 * (at most 31 + 11 + 11 significant bits); one division, one addition, one
 * final rounding to fp16. */
void orc_dequant_rows(const int32_t *acc, const float *sx, const float *sw,
                      const double *out, const uint16_t *bias, const int64_t *rows,
                      int64_t nrows, int64_t N, uint16_t *Y, int fmt) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t r = 0; r < nrows; r++) {
    for (int64_t n = 0; n < N; n++) {
      double p = (double)acc[r * N + n] * (double)sx[rows[r]] * (double)sw[n];
      double v = p / 16129.0 + out[r * N + n];
      if (bias) v += elem_to_double(bias[n], fmt);  /* nn.Linear's bias, before the one rounding */
      Y[r * N + n] = double_to_elem(v, fmt);
    }
  }
}

/* The whole layer, S2..S6, for a chosen set of rows.  The outlier set and the
 * activation codes are computed over ALL T rows (the outlier set depends on
 * every row); S4..S6 only for `rows`.  Intermediates are optional outputs
 * (NULL to skip) except acc and out, which the caller provides as scratch.
 * W16 NULL: the outlier weights come from the int8 codes (above).  fmt: the
 * 16-bit format of X, W16, the bias and Y (0 fp16, 1 bf16). */
int orc_linear_rows(const uint16_t *X, int64_t T, int64_t K, const int8_t *Wq,
                    const float *sw, const uint16_t *W16, int64_t N, float tau,
                    const uint16_t *bias, const int64_t *rows, int64_t nrows, int8_t *Xq,
                    float *sx, int32_t *O, int32_t *nO, int32_t *acc, double *out,
                    uint16_t *Y, int fmt) {
  int rc = orc_outlier_columns(X, T, K, tau, O, nO, fmt);
  if (rc) return rc;
  rc = orc_quantize_activations(X, T, K, O, *nO, Xq, sx, NULL, fmt);
  if (rc) return rc;
  rc = orc_int8_matmul_rows(Xq, Wq, T, N, K, rows, nrows, acc);
  if (W16)
    orc_outlier_matmul_rows(X, W16, T, N, K, O, *nO, rows, nrows, out, fmt);
  else  /* only the int8 weight is kept */
    orc_outlier_matmul_rows_wq(X, Wq, sw, N, K, O, *nO, rows, nrows, out, fmt);
  orc_dequant_rows(acc, sx, sw, out, bias, rows, nrows, N, Y, fmt);
  return rc;
}

/* ---- the blockwise 8-bit codec of optimizer states ----
 * 8-bit optimizers keep their states quantized block-wise ("bitsandbytes:
 * GPU-Accelerated Inference and Training at Lower Bit Depths", section
 * "8-bit optimizers for full-model training"); each block carries its own
 * scaling factor, which limits what one outlier does to its neighbours (page
 * "bitsandbytes", section "What it provides").  Readings (the pages give no
 * block size and no code map): fp32 values in blocks of B consecutive
 * elements (the last block may be short), the block's scale is its absmax
 * a, the code is q = rint(fl32(fl32(127 * x) / a)) in IEEE fp32, ties to
 * even (0 when a = 0), and the decoded value is fl32(fl32(q * a) / 127).
 * For a >= 2^120 those formulas leave fp32's range (127 x and q a reach
 * 2^127 * 127 > FLT_MAX), so such a block is coded and decoded with x and a
 * first multiplied by 2^-8 and the decoded value multiplied back by 2^8.
 * A power-of-two factor commutes with every IEEE rounding in the normal
 * range, so the scaled formulas give the plain ones' results wherever those
 * are finite; values that the factor pushes below the normal range have
 * code 0 either way (|127 x / a| < 2^-100 there). */
static float codec_scale(float a) { return a >= 0x1p120f ? 0x1p-8f : 1.0f; }

int orc_quantize_blockwise(const float *x, int64_t n, int64_t B, int8_t *q, float *absmax) {
  if (n < 0 || B <= 0) return ORC_ERR_ARG;
  const int64_t nb = (n + B - 1) / B;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nb; b++) {
    const int64_t i0 = b * B, i1 = i0 + B < n ? i0 + B : n;
    float a = 0.0f;
    for (int64_t i = i0; i < i1; i++) {
      const float v = fabsf(x[i]);
      if (v > a) a = v;
    }
    absmax[b] = a;
    const float s = codec_scale(a);
    const float as = a * s;
    for (int64_t i = i0; i < i1; i++) {
      if (a == 0.0f) {
        q[i] = 0;
      } else {
        const float num = 127.0f * (x[i] * s);
        q[i] = (int8_t)rintf(num / as);
      }
    }
  }
  return ORC_OK;
}

int orc_dequantize_blockwise(const int8_t *q, const float *absmax, int64_t n, int64_t B,
                             float *y) {
  if (n < 0 || B <= 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) {
    const float a = absmax[i / B], s = codec_scale(a);
    const float prod = (float)q[i] * (a * s);
    y[i] = (prod / 127.0f) / s;
  }
  return ORC_OK;
}
