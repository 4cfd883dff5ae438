/*
 * Plain CPU oracle of C = relu(A·B) for fp16 A (M,K), B (K,N), row-major.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
 * leg may load this library.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (TileLang paper-reading page, section 2, the matmul_relu example):
 *   the accumulator fragment is float32 and starts cleared (T.clear); every k-step adds
 *   A_tile·B_tile into it (T.gemm); the epilogue replaces each element x by max(x, 0)
 *   (the T.Parallel loop with T.max) and the copy to the float16 C rounds it.
 * The practitioner page (section 3.2) states why the accumulator is float32 and not float16.
 *
 * So, element by element,
 *     C[i,j] = fp16_rne( relu( sum_{k=0}^{K-1} A[i,k]*B[k,j] ) )
 * with the sum formed in float32 in increasing k.  Every fp16*fp16 product has at most 22
 * significant bits and an exponent inside float32's range, so each product is exact in
 * float32 and the only roundings are the K-1 additions (FMA contraction cannot change the
 * result).  A second accumulator in float64 (same order) gives the near-exact reference
 * that the tolerance is measured against; it is rounded to fp16 directly, once.
 *
 * relu(x) = (x > 0) ? x : +0, so -0 and NaN give +0.  fp16 rounding: IEEE 754 binary16,
 * round to nearest with ties to even, subnormals kept, overflow to infinity.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- IEEE 754 binary16 encode / decode, written from the format's definition ---- */

/* Round a non-negative double q (< 2^53) to the nearest integer, ties to even. */
static double round_half_even(double q) {
  double fl = floor(q);
  double diff = q - fl; /* exact: q and fl share exponent range */
  if (diff > 0.5) return fl + 1.0;
  if (diff < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* binary64 -> binary16 bits, round to nearest even. NaN -> quiet NaN 0x7E00 with the sign. */
uint16_t tg_oracle_f64_to_f16(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
  double a = fabs(x);
  /* largest finite is 65504 = (2 - 2^-10) * 2^15; the midpoint to 2^16 is 65520 and the tie
     goes to the even neighbour 2^16, which overflows: so a >= 65520 -> infinity. */
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
  if (a < 0x1p-14) {
    /* subnormal range: value = m * 2^-24 with m in [0, 1024]; m == 1024 is the smallest normal
       and its bit pattern 0x0400 follows on directly. */
    double m = round_half_even(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)m);
  }
  int e2;
  double fr = frexp(a, &e2);         /* a = fr * 2^e2, fr in [0.5, 1) */
  int e = e2 - 1;                    /* a = s * 2^e, s in [1, 2), e in [-14, 15] */
  double q = ldexp(fr, 11);          /* s * 2^10 in [1024, 2048), exact */
  double r = round_half_even(q);
  if (r == 2048.0) { r = 1024.0; e += 1; }
  if (e > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(r - 1024.0));
}

/* binary32 -> binary16: every float is exactly a double, so this is the same rounding. */
uint16_t tg_oracle_f32_to_f16(float x) { return tg_oracle_f64_to_f16((double)x); }

/* binary16 bits -> exact double value. */
double tg_oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 0x1F;
  int man = h & 0x3FF;
  double v;
  if (ex == 0x1F) {
    v = man ? NAN : INFINITY;
  } else if (ex == 0) {
    v = ldexp((double)man, -24);
  } else {
    v = ldexp((double)(1024 + man), ex - 25);
  }
  return sign ? -v : v;
}

void tg_oracle_f32_to_f16_array(const float* x, uint16_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = tg_oracle_f32_to_f16(x[i]);
}
void tg_oracle_f64_to_f16_array(const double* x, uint16_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = tg_oracle_f64_to_f16(x[i]);
}
void tg_oracle_f16_to_f64_array(const uint16_t* x, double* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = tg_oracle_f16_to_f64(x[i]);
}

static float relu32(float x) { return (x > 0.0f) ? x : 0.0f; }
static double relu64(double x) { return (x > 0.0) ? x : 0.0; }

/*
 * relu(A·B) on a sub-grid of C: rows rows[0..nr-1] and columns cols[0..nc-1] (nr*nc outputs,
 * row-major in the outputs).  With every row and column selected this is the whole C.
 *
 *   out16_f32acc[r*nc+c]  fp16 bits of relu(float32 sum)          (may be NULL)
 *   acc_f32[r*nc+c]       float32 sum before relu                  (may be NULL)
 *   out16_f64acc[r*nc+c]  fp16 bits of relu(float64 sum)          (may be NULL)
 *   acc_f64[r*nc+c]       float64 sum before relu                  (may be NULL)
 *   relu                  1: apply relu; 0: identity epilogue
 *   nthreads              OpenMP threads over rows (0 = runtime default)
 *
 * Returns 0, or -1 on a bad argument or allocation failure.
 */
int tg_oracle_gemm_relu(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, const int64_t* rows, int64_t nr,
                        const int64_t* cols, int64_t nc, int relu, uint16_t* out16_f32acc,
                        float* acc_f32, uint16_t* out16_f64acc, double* acc_f64, int nthreads) {
  if (M < 0 || N < 0 || K < 0 || nr < 0 || nc < 0) return -1;
  if (K > 0 && (lda < K || ldb < N)) return -1;
  for (int64_t r = 0; r < nr; ++r)
    if (rows[r] < 0 || rows[r] >= M) return -1;
  for (int64_t c = 0; c < nc; ++c)
    if (cols[c] < 0 || cols[c] >= N) return -1;
  if (nr == 0 || nc == 0) return 0;
  const int want32 = (out16_f32acc != NULL) || (acc_f32 != NULL);
  const int want64 = (out16_f64acc != NULL) || (acc_f64 != NULL);

  /* decode the selected columns of B once: Bsel[k*nc + c] = B[k, cols[c]] (exact) */
  float* Bsel = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1) * (size_t)nc);
  if (!Bsel) return -1;
  for (int64_t k = 0; k < K; ++k)
    for (int64_t c = 0; c < nc; ++c)
      Bsel[k * nc + c] = (float)tg_oracle_f16_to_f64(B[k * ldb + cols[c]]);

  int failed = 0;
#ifdef _OPENMP
  int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
  for (int64_t r = 0; r < nr; ++r) {
    float* s32 = (float*)calloc((size_t)nc, sizeof(float));
    double* s64 = (double*)calloc((size_t)nc, sizeof(double));
    if (!s32 || !s64) {
      failed = 1;
    } else {
      const uint16_t* arow = A + rows[r] * lda;
      for (int64_t k = 0; k < K; ++k) {
        float a = (float)tg_oracle_f16_to_f64(arow[k]);
        const float* brow = Bsel + k * nc;
        if (want32)
          for (int64_t c = 0; c < nc; ++c) s32[c] = s32[c] + a * brow[c];
        if (want64)
          for (int64_t c = 0; c < nc; ++c) s64[c] = s64[c] + (double)a * (double)brow[c];
      }
      for (int64_t c = 0; c < nc; ++c) {
        int64_t o = r * nc + c;
        if (acc_f32) acc_f32[o] = s32[c];
        if (out16_f32acc) out16_f32acc[o] = tg_oracle_f32_to_f16(relu ? relu32(s32[c]) : s32[c]);
        if (acc_f64) acc_f64[o] = s64[c];
        if (out16_f64acc) out16_f64acc[o] = tg_oracle_f64_to_f16(relu ? relu64(s64[c]) : s64[c]);
      }
    }
    free(s32);
    free(s64);
  }
  free(Bsel);
  return failed ? -1 : 0;
}

int tg_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- fused epilogue: C = fp16( act( sum + bias[j] ) + residual[i, j] ) ----
 *
 * The pages motivate fusing the elementwise epilogue into the GEMM (the practitioner page,
 * section 2) and use relu as the example (the paper-reading page, section 2).  Activations:
 *   relu(x)      = x > 0 ? x : +0
 *   gelu(x)      = x/2 * (1 + erf(x / sqrt 2))
 *   gelu_tanh(x) = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))
 * (GELU and its tanh form: Hendrycks & Gimpel, "Gaussian Error Linear Units", 2016.)
 * The float64 result adds bias, applies the activation with libm's erf/tanh and adds the
 * residual in double, then rounds once to fp16; the float32 result does the same steps in
 * float (activation evaluated in double and rounded to float).
 */
static double act64(double x, int act) {
  switch (act) {
    case 1: return (x > 0.0) ? x : 0.0;
    case 2: return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
    case 3: return 0.5 * x * (1.0 + tanh(sqrt(2.0 / acos(-1.0)) * (x + 0.044715 * x * x * x)));
    default: return x;
  }
}

int tg_oracle_gemm_epilogue(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, const int64_t* rows, int64_t nr,
                            const int64_t* cols, int64_t nc, int act, const uint16_t* bias,
                            const uint16_t* residual, int64_t ldr, uint16_t* out16_f32acc,
                            uint16_t* out16_f64acc, double* pre_f64, int nthreads) {
  if (act < 0 || act > 3) return -1;
  if (residual && ldr < N) return -1;
  if (nr == 0 || nc == 0) return 0;
  float* s32 = (float*)malloc(sizeof(float) * (size_t)nr * (size_t)nc);
  double* s64 = (double*)malloc(sizeof(double) * (size_t)nr * (size_t)nc);
  if (!s32 || !s64) {
    free(s32);
    free(s64);
    return -1;
  }
  int rc = tg_oracle_gemm_relu(A, B, M, N, K, lda, ldb, rows, nr, cols, nc, 0, NULL, s32, NULL,
                               s64, nthreads);
  if (rc == 0) {
    for (int64_t r = 0; r < nr; ++r) {
      for (int64_t c = 0; c < nc; ++c) {
        const int64_t o = r * nc + c;
        const int64_t i = rows[r], j = cols[c];
        double b = bias ? tg_oracle_f16_to_f64(bias[j]) : 0.0;
        double res = residual ? tg_oracle_f16_to_f64(residual[i * ldr + j]) : 0.0;
        /* float64 reference */
        double x = s64[o] + b;
        if (pre_f64) pre_f64[o] = x;
        double y = act64(x, act) + res;
        if (out16_f64acc) out16_f64acc[o] = tg_oracle_f64_to_f16(y);
        /* float32 steps */
        float xf = s32[o] + (float)b;
        float yf = (float)act64((double)xf, act);
        yf = yf + (float)res;
        if (out16_f32acc) out16_f32acc[o] = tg_oracle_f32_to_f16(yf);
      }
    }
  }
  free(s32);
  free(s64);
  return rc;
}

/* ---- int4 weight dequantisation (W_INT4 / A_FP16 GEMM) ----
 *
 * The paper-reading page (section 5) evaluates a dequantising GEMM with 4-bit integer weights
 * and fp16 activations.  Format used here: Wq holds K rows of ceil(N/8) uint32 words; word
 * (k, c) carries columns 8c..8c+7, column 8c+e in bits [4e, 4e+4); q is unsigned in [0, 15]
 * with the zero point 8.  scales holds ceil(K/group) rows of N fp16 values (leading dimension
 * lds).  The weight is
 *     w[k][n] = fp16_rne( (q[k][n] - 8) * scales[k / group][n] )
 * (the product is exact in double; one rounding).  out16 is K x N fp16 bits, row-major.
 */
int tg_oracle_dequant_w4(const uint32_t* Wq, const uint16_t* scales, int64_t K, int64_t N,
                         int64_t ldq, int64_t lds, int64_t group, uint16_t* out16) {
  if (K < 0 || N < 0 || group <= 0 || ldq < (N + 7) / 8 || lds < N) return -1;
  for (int64_t k = 0; k < K; ++k) {
    for (int64_t n = 0; n < N; ++n) {
      const uint32_t word = Wq[k * ldq + n / 8];
      const int q = (int)((word >> (4 * (n % 8))) & 0xFu);
      const double s = tg_oracle_f16_to_f64(scales[(k / group) * lds + n]);
      out16[k * N + n] = tg_oracle_f64_to_f16((double)(q - 8) * s);
    }
  }
  return 0;
}

/* ---- NF4 weight dequantisation (W_NF4 / A_FP16 GEMM) ----
 *
 * The paper-reading page (section 5) names a second dequantising GEMM beside W_INT4 / A_FP16:
 * 4-bit NormalFloat weights with fp16 activations.  NF4 (Dettmers, Pagnoni, Holtzman and
 * Zettlemoyer, "QLoRA: Efficient Finetuning of Quantized LLMs", NeurIPS 2023, section 3 and
 * Appendix E) maps a 4-bit code q to one of 16 values spread like the quantiles of a standard
 * normal distribution, normalised to [-1, 1], with an exact zero.  The table below is the one
 * printed in that appendix.
 *
 * Storage, the same as the int4 format above: Wq holds K rows of ceil(N/8) uint32 words;
 * column 8c+e of row k is the nibble in bits [4e, 4e+4) of word (k, c).  scales holds
 * ceil(K/group) rows of N fp16 values (leading dimension lds).  The weight is
 *     w[k][n] = fp16_rne( fp16_rne(nf4[q[k][n]]) * scales[k / group][n] )
 * the code value rounded to fp16 once (it is held in the activations' precision), then the
 * product (exact in double) rounded once.  out16 is K x N fp16 bits, row-major.
 */
static const double kNf4Codes[16] = {
    -1.0,
    -0.6961928009986877,
    -0.5250730514526367,
    -0.39491748809814453,
    -0.28444138169288635,
    -0.18477343022823334,
    -0.09105003625154495,
    0.0,
    0.07958029955625534,
    0.16093020141124725,
    0.24611230194568634,
    0.33791524171447754,
    0.44070982933044434,
    0.5626170039176941,
    0.7229568362236023,
    1.0,
};

/* The NF4 code value of q (0..15) as printed; NaN for any other q. */
double tg_oracle_nf4_code(int q) { return (q >= 0 && q < 16) ? kNf4Codes[q] : NAN; }

int tg_oracle_dequant_nf4(const uint32_t* Wq, const uint16_t* scales, int64_t K, int64_t N,
                          int64_t ldq, int64_t lds, int64_t group, uint16_t* out16) {
  if (K < 0 || N < 0 || group <= 0 || ldq < (N + 7) / 8 || lds < N) return -1;
  for (int64_t k = 0; k < K; ++k) {
    const int64_t g = k / group; /* scale row */
    for (int64_t n = 0; n < N; ++n) {
      const uint32_t word = Wq[k * ldq + n / 8];
      const unsigned nib = (word >> (4u * (uint32_t)(n % 8))) & 15u;
      const double code = tg_oracle_f16_to_f64(tg_oracle_f64_to_f16(kNf4Codes[nib]));
      const double s = tg_oracle_f16_to_f64(scales[g * lds + n]);
      out16[k * N + n] = tg_oracle_f64_to_f16(code * s);
    }
  }
  return 0;
}
