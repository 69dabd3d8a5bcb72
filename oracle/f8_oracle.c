/*
 * CPU oracle for the Float8 training linear with dynamic tensorwise scaling.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file: only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg use it. It shares no code, header, table or
 * constant generator with the CUDA library.
 *
 * What it follows:
 *   - "TorchTitan: One-stop PyTorch native solution for production ready LLM
 *     pretraining" (atlas.scime.ai summary), Approach and the ablation table:
 *     Float8 is one of the composable training transformations, measured on
 *     Llama 3.1 8B on top of torch.compile.
 *   - wassimseifeddine.com/posts/torchtitan, section "Float8 Training": the
 *     feature is torchao's Float8 training.
 *   - stanleyjacob.dev/oss/torchtitan, Part XI (reading list), item 9: the
 *     number formats are the E4M3 / E5M2 encodings of "FP8 Formats for Deep
 *     Learning" (Micikevicius et al., 2022).  The E4M3 bit layout used here is
 *     the one that paper defines: 1 sign, 4 exponent (bias 7) and 3 mantissa
 *     bits, no infinities, S.1111.111 is NaN, largest finite value 448.
 *   - The pages never spell out the scaling recipe.  The plainest reading,
 *     and the one this oracle takes, is dynamic tensorwise scaling:
 *     amax = max|x| over the whole tensor, s = 448 / amax in fp32 (with the
 *     clamp amax >= 1e-12 so that an all-zero tensor stays finite),
 *     q = satfinite_rne_e4m3(fl32(x * s)), three GEMMs with exact
 *     accumulation, then division by the two scales and round-to-nearest-even
 *     to bf16.
 *
 * Everything here is written from those definitions, in exact arithmetic
 * where the definition is exact: fp64 holds every fp32, every e4m3 value and
 * every partial sum below 2^53 exactly, and the GEMM sums are formed in int64.
 * Built with -ffp-contract=off so that the one fp32 multiply of the cast is a
 * plain IEEE multiply.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16                                                                      */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an fp32 bit pattern, so widening is exact. */
float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Round a double to the nearest bf16, ties to even, from the definition of
 * the format: 8 exponent bits (bias 127), 7 stored mantissa bits, gradual
 * underflow with spacing 2^-133 below 2^-126, and overflow to infinity for
 * anything that rounds to 2^128 or beyond.
 */
uint16_t or_f64_to_bf16(double y)
{
    if (isnan(y))
        return 0x7FC0;
    uint16_t sign = signbit(y) ? 0x8000 : 0;
    double a = fabs(y);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);

    int e;
    frexp(a, &e);          /* a = f * 2^e with f in [0.5, 1) */
    int E = e - 1;         /* a in [2^E, 2^(E+1)) */
    double ulp = (E < -126) ? ldexp(1.0, -133) : ldexp(1.0, E - 7);

    double n = a / ulp;    /* exact: division by a power of two */
    double fl = floor(n);
    double r = n - fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) == 1.0))
        fl += 1.0;
    double v = fl * ulp;   /* the rounded magnitude, exact */

    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    if (v < ldexp(1.0, -126))
        return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -133)));

    int e2;
    frexp(v, &e2);
    int E2 = e2 - 1;
    int mant = (int)(v / ldexp(1.0, E2) * 128.0) - 128;
    return (uint16_t)(sign | ((E2 + 127) << 7) | mant);
}

/* ------------------------------------------------------------------------ */
/* E4M3 ("float8_e4m3fn")                                                    */
/* ------------------------------------------------------------------------ */

/* Value of an E4M3 byte S.EEEE.MMM; NaN for S.1111.111. */
double or_e4m3_decode(uint8_t c)
{
    int s = c >> 7;
    int E = (c >> 3) & 0xF;
    int M = c & 0x7;
    if (E == 15 && M == 7)
        return NAN;
    double mag = (E == 0) ? (double)M * ldexp(1.0, -9)
                          : (double)(8 + M) * ldexp(1.0, E - 10);
    return s ? -mag : mag;
}

/*
 * Saturating round-to-nearest-even of an fp32 value to E4M3.
 *   |v| >= 448 (and +-inf) -> +-448: no finite code lies above 448.
 *   otherwise the nearest point of the E4M3 grid, ties to the even code.
 * The grid spacing is 2^-9 below 2^-6 (subnormals and the first normal
 * binade share it) and 2^(E-3) in the binade [2^E, 2^(E+1)).  Within a
 * spacing-uniform stretch consecutive grid points are consecutive codes, so
 * "even multiple of the spacing" is "even code".  The sign is kept, also for
 * results that round to zero.
 */
uint8_t or_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);

    double ulp;
    if (a < ldexp(1.0, -6)) {
        ulp = ldexp(1.0, -9);
    } else {
        int e;
        frexp(a, &e);
        ulp = ldexp(1.0, (e - 1) - 3);
    }
    double n = a / ulp;
    double fl = floor(n);
    double r = n - fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) == 1.0))
        fl += 1.0;
    double q = fl * ulp;   /* a grid value in [0, 448] */

    if (q < ldexp(1.0, -6))
        return (uint8_t)(sign | (uint8_t)(q / ldexp(1.0, -9)));
    int e2;
    frexp(q, &e2);
    int E2 = e2 - 1;
    int mant = (int)(q / ldexp(1.0, E2) * 8.0) - 8;
    return (uint8_t)(sign | ((E2 + 7) << 3) | mant);
}

/* ------------------------------------------------------------------------ */
/* E5M2 ("float8_e5m2")                                                      */
/* ------------------------------------------------------------------------ */

/*
 * Value of an E5M2 byte S.EEEEE.MM (bias 15, IEEE-like): E=0 subnormals
 * M * 2^-16; E=1..30 (4+M) * 2^(E-17); E=31: M=0 is +-inf, else NaN.
 */
double or_e5m2_decode(uint8_t c)
{
    int s = c >> 7;
    int E = (c >> 2) & 0x1F;
    int M = c & 0x3;
    double mag;
    if (E == 31)
        mag = (M == 0) ? INFINITY : NAN;
    else if (E == 0)
        mag = (double)M * ldexp(1.0, -16);
    else
        mag = (double)(4 + M) * ldexp(1.0, E - 17);
    return s ? -mag : mag;
}

/*
 * Saturating round-to-nearest-even of an fp32 value to E5M2: |v| >= 57344
 * (the largest finite value, 1.75 * 2^15) and +-inf give +-57344; NaN gives
 * a NaN code; otherwise the nearest grid point, ties to the even code.  The
 * spacing is 2^-16 below 2^-14 and 2^(E-2) in the binade [2^E, 2^(E+1)).
 */
uint8_t or_e5m2_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a >= 57344.0)
        return (uint8_t)(sign | 0x7B);

    double ulp;
    if (a < ldexp(1.0, -14)) {
        ulp = ldexp(1.0, -16);
    } else {
        int e;
        frexp(a, &e);
        ulp = ldexp(1.0, (e - 1) - 2);
    }
    double n = a / ulp;
    double fl = floor(n);
    double r = n - fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) == 1.0))
        fl += 1.0;
    double q = fl * ulp;   /* a grid value in [0, 57344] */

    if (q < ldexp(1.0, -14))
        return (uint8_t)(sign | (uint8_t)(q / ldexp(1.0, -16)));
    int e2;
    frexp(q, &e2);
    int E2 = e2 - 1;
    int mant = (int)(q / ldexp(1.0, E2) * 4.0) - 4;
    return (uint8_t)(sign | ((E2 + 15) << 2) | mant);
}

/* ------------------------------------------------------------------------ */
/* Dynamic tensorwise scaling                                                */
/* ------------------------------------------------------------------------ */

/*
 * amax = max_i |x_i| over a bf16 tensor, in fp32 (exact, order-free).
 * Non-finite entries are left out of the maximum and reported through
 * *nonfinite (1 if any entry is +-inf or NaN).
 */
float or_amax(const uint16_t *x, int64_t n, int *nonfinite)
{
    float m = 0.0f;
    int nf = 0;
#pragma omp parallel for reduction(max : m) reduction(| : nf) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(or_bf16_to_f32(x[i]));
        if (!isfinite(a))
            nf = 1;
        else if (a > m)
            m = a;
    }
    if (nonfinite)
        *nonfinite = nf;
    return m;
}

/* s = fl32(448 / max(amax, 1e-12)), one IEEE fp32 division. */
float or_scale(float amax)
{
    float d = (amax > 1e-12f) ? amax : 1e-12f;
    return 448.0f / d;
}

/* The same with the largest finite value of the format: 448 (E4M3, fmt 0)
 * or 57344 (E5M2, fmt 1). */
float or_scale_fmt(float amax, int fmt)
{
    float d = (amax > 1e-12f) ? amax : 1e-12f;
    return (fmt == 1 ? 57344.0f : 448.0f) / d;
}

/*
 * q = satfinite_rne_e4m3(fl32(x * s)) for a row-major bf16 [rows, cols]
 * tensor, written row-major into q [rows, cols] and column-major into
 * qt [cols, rows] (either may be NULL).
 */
void or_cast_transpose(const uint16_t *x, int64_t rows, int64_t cols, float s,
                       uint8_t *q, uint8_t *qt)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            float v = or_bf16_to_f32(x[r * cols + c]) * s;
            uint8_t b = or_e4m3_encode(v);
            if (q)
                q[r * cols + c] = b;
            if (qt)
                qt[c * rows + r] = b;
        }
    }
}

/* q = satfinite_rne_<fmt>(fl32(x * s)), both layouts, fmt 0 = E4M3, 1 = E5M2. */
void or_cast_transpose_fmt(const uint16_t *x, int64_t rows, int64_t cols, float s, int fmt,
                           uint8_t *q, uint8_t *qt)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            float v = or_bf16_to_f32(x[r * cols + c]) * s;
            uint8_t b = (fmt == 1) ? or_e5m2_encode(v) : or_e4m3_encode(v);
            if (q)
                q[r * cols + c] = b;
            if (qt)
                qt[c * rows + r] = b;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM: C[m,n] = bf16( sum_k dec(A[m,k]) * dec(B[n,k]) / (sa * sb) )         */
/* ------------------------------------------------------------------------ */

/*
 * Every E4M3 value is an integer multiple of 2^-9 with magnitude at most
 * 448 * 2^9 = 229376 < 2^18, so z = value * 2^9 is an exact int32.  A NaN
 * code has no value; the encoder above never emits one, and it is mapped
 * to 0 here.
 */
static void decode_row_z(const uint8_t *src, int64_t n, int32_t *z)
{
    for (int64_t i = 0; i < n; ++i) {
        double v = or_e4m3_decode(src[i]);
        z[i] = isnan(v) ? 0 : (int32_t)(v * 512.0);
    }
}

/*
 * One output: the exact sum, then the exact dequantised value
 * acc * 2^-18 / (sa * sb) rounded once to fp64 (sa * sb is exact in fp64)
 * and then to nearest-even bf16.
 */
static uint16_t finish(int64_t acc, float sa, float sb)
{
    double y = (double)acc * ldexp(1.0, -18) / ((double)sa * (double)sb);
    return or_f64_to_bf16(y);
}

static uint16_t finish_f64(double acc, float sa, float sb)
{
    double y = acc * ldexp(1.0, -18) / ((double)sa * (double)sb);
    return or_f64_to_bf16(y);
}

/*
 * Full GEMM.  a: [M,K] row-major E4M3 bytes, b: [N,K] row-major E4M3 bytes,
 * c: [M,N] row-major bf16.  route 0 sums in int64, route 1 in fp64; with
 * |z_a z_b| < 2^36 and K < 2^17 both sums are exact and therefore equal.
 */
void or_gemm(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
             float sa, float sb, uint16_t *c, int route)
{
    int32_t *zb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N * K > 0 ? N * K : 1));
    for (int64_t n = 0; n < N; ++n)
        decode_row_z(b + n * K, K, zb + n * K);
#pragma omp parallel
    {
        int32_t *za = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            decode_row_z(a + m * K, K, za);
            for (int64_t n = 0; n < N; ++n) {
                const int32_t *zr = zb + n * K;
                if (route == 0) {
                    int64_t acc = 0;
                    for (int64_t k = 0; k < K; ++k)
                        acc += (int64_t)za[k] * (int64_t)zr[k];
                    c[m * N + n] = finish(acc, sa, sb);
                } else {
                    double acc = 0.0;
                    for (int64_t k = 0; k < K; ++k)
                        acc += (double)za[k] * (double)zr[k];
                    c[m * N + n] = finish_f64(acc, sa, sb);
                }
            }
        }
        free(za);
    }
    free(zb);
}

/*
 * Selected rows of the same GEMM: out[i, n] = C[rows[i], n] for n < N.
 * Used to check outputs of shapes too large for the full product.
 */
void or_gemm_rows(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                  float sa, float sb, const int64_t *rows, int64_t nrows, uint16_t *out)
{
    (void)M;
    int32_t *za = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nrows * K > 0 ? nrows * K : 1));
    for (int64_t i = 0; i < nrows; ++i)
        decode_row_z(a + rows[i] * K, K, za + i * K);
#pragma omp parallel
    {
        int32_t *zr = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t n = 0; n < N; ++n) {
            decode_row_z(b + n * K, K, zr);
            for (int64_t i = 0; i < nrows; ++i) {
                const int32_t *zi = za + i * K;
                int64_t acc = 0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (int64_t)zi[k] * (int64_t)zr[k];
                out[i * N + n] = finish(acc, sa, sb);
            }
        }
        free(zr);
    }
    free(za);
}

/* Selected columns: out[j, m] = C[m, cols[j]] for m < M. */
void or_gemm_cols(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                  float sa, float sb, const int64_t *cols, int64_t ncols, uint16_t *out)
{
    (void)N;
    int32_t *zb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(ncols * K > 0 ? ncols * K : 1));
    for (int64_t j = 0; j < ncols; ++j)
        decode_row_z(b + cols[j] * K, K, zb + j * K);
#pragma omp parallel
    {
        int32_t *za = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t m = 0; m < M; ++m) {
            decode_row_z(a + m * K, K, za);
            for (int64_t j = 0; j < ncols; ++j) {
                const int32_t *zj = zb + j * K;
                int64_t acc = 0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (int64_t)za[k] * (int64_t)zj[k];
                out[j * M + m] = finish(acc, sa, sb);
            }
        }
        free(za);
    }
    free(zb);
}

/*
 * Mixed formats.  Every E5M2 value is an integer multiple of 2^-16 with
 * magnitude at most 57344 * 2^16 < 2^32 and every E4M3 value one of 2^-9, so
 * z = value * 2^16 (E5M2) or value * 2^9 (E4M3) is an exact int64, and the
 * dot product is summed exactly in __int128 (a product is below 2^64 and a
 * row has fewer than 2^31 terms).  The exact sum times 2^-(ea+eb) is then
 * rounded to fp64 (exact while it stays below 2^53, one rounding beyond),
 * divided by sa*sb (exact in fp64) with one more rounding, and rounded to
 * nearest-even bf16.  fmt: 0 = E4M3, 1 = E5M2.
 */
static void decode_row_z64(const uint8_t *src, int64_t n, int fmt, int64_t *z)
{
    for (int64_t i = 0; i < n; ++i) {
        double v = fmt == 1 ? or_e5m2_decode(src[i]) : or_e4m3_decode(src[i]);
        z[i] = (isnan(v) || isinf(v)) ? 0 : (int64_t)(v * (fmt == 1 ? 65536.0 : 512.0));
    }
}

static uint16_t finish128(__int128 acc, int shift, float sa, float sb)
{
    double y = (double)acc * ldexp(1.0, -shift) / ((double)sa * (double)sb);
    return or_f64_to_bf16(y);
}

/* Rows `rows` of C = A B^T with A in format fa, B in format fb. */
void or_gemm_rows_fmt(const uint8_t *a, int fa, const uint8_t *b, int fb, int64_t M, int64_t N,
                      int64_t K, float sa, float sb, const int64_t *rows, int64_t nrows,
                      uint16_t *out)
{
    (void)M;
    const int shift = (fa == 1 ? 16 : 9) + (fb == 1 ? 16 : 9);
    int64_t *za = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nrows * K > 0 ? nrows * K : 1));
    for (int64_t i = 0; i < nrows; ++i)
        decode_row_z64(a + rows[i] * K, K, fa, za + i * K);
#pragma omp parallel
    {
        int64_t *zr = (int64_t *)malloc(sizeof(int64_t) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t n = 0; n < N; ++n) {
            decode_row_z64(b + n * K, K, fb, zr);
            for (int64_t i = 0; i < nrows; ++i) {
                const int64_t *zi = za + i * K;
                __int128 acc = 0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (__int128)zi[k] * (__int128)zr[k];
                out[i * N + n] = finish128(acc, shift, sa, sb);
            }
        }
        free(zr);
    }
    free(za);
}

/* ------------------------------------------------------------------------ */
/* SwiGLU input of the w2 linear: h = bf16( silu(a) * b )                     */
/* ------------------------------------------------------------------------ */

/*
 * The pages name the SwiGLU FFN of Llama 3.1 (the ablation table's model)
 * but print no arithmetic for it, so the oracle takes the definition itself:
 * silu(a) = a / (1 + exp(-a)) = a * sigma(a), with h = silu(a) * b, each
 * formed in fp64 from the exact bf16 inputs (libm exp) and rounded once to
 * bf16.  fp64 carries 29 more bits than the bf16 result needs, so this is
 * the correctly rounded h except within ~2^-50 (relative) of a bf16
 * rounding boundary.  exp(-a) overflows fp64 only for a < -709, where
 * a / inf gives the correctly signed zero (and -inf / inf the NaN of
 * -inf * sigma(-inf) = -inf * 0).
 */
double or_silu(double a)
{
    return a / (1.0 + exp(-a));
}

/* h = bf16(silu(a) * b) elementwise over n values, in fp64. */
void or_swiglu_h(const uint16_t *a, const uint16_t *b, int64_t n, uint16_t *h)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const double fa = (double)or_bf16_to_f32(a[i]);
        const double fb = (double)or_bf16_to_f32(b[i]);
        h[i] = or_f64_to_bf16(or_silu(fa) * fb);
    }
}

/*
 * The gradient of h = silu(a) * b for an upstream gradient dh, elementwise
 * over n values, from the derivative of the definition above:
 *   sigma    = 1 / (1 + exp(-a))
 *   dh/db    = silu(a) = a sigma
 *   dh/da    = b silu'(a),   silu'(a) = sigma (1 + a (1 - sigma))
 *   db = bf16(dh * a * sigma),  da = bf16(dh * b * silu'(a))
 * all in fp64, each output rounded once to bf16.
 */
void or_swiglu_bwd(const uint16_t *dh, const uint16_t *a, const uint16_t *b, int64_t n,
                   uint16_t *da, uint16_t *db)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const double fa = (double)or_bf16_to_f32(a[i]);
        const double fb = (double)or_bf16_to_f32(b[i]);
        const double fdh = (double)or_bf16_to_f32(dh[i]);
        const double sigma = 1.0 / (1.0 + exp(-fa));
        const double dsilu = sigma * (1.0 + fa * (1.0 - sigma));
        db[i] = or_f64_to_bf16(fdh * (fa * sigma));
        da[i] = or_f64_to_bf16(fdh * fb * dsilu);
    }
}

/* Number of threads the parallel loops above use. */
int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
