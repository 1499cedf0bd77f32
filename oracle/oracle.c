/*
 * oracle.c -- plain CPU definition of the skinny decode projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library.
 *
 * What it computes
 * ----------------
 * The projection of low-batch decode: y = x . W^T, optionally followed by the
 * attention-residual add that the output projection is fused with.
 *   - "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly"
 *     (papercache.org deep notes), method details 1 "Tune shapes for the
 *     workload": the attention input projections, computed by small-matrix
 *     kernels at batch 1-2 and by split-K kernels at larger batch.  Split-K
 *     only reorders the sum over the reduction dimension, so the definition
 *     below is the plain sum in k order.
 *   - same page, method details 2 "Overlap computation and communication":
 *     the output projection fused with the attention residual add.
 *
 *   y_ref[m,n] = sum_{k<K} x[m,k] * W[n,k]   (+ res[m,n])          (fp64)
 *   s1[m,n]    = sum_{k<K} |x[m,k]| * |W[n,k]|                      (fp64)
 *   y_bf16     = round-to-nearest-even(y_ref) to bfloat16, once.
 *
 * W is [N,K] row-major (an nn.Linear weight), x is [M,K], res and y are
 * [M,N], all row-major and dense; every operand is bfloat16 given as raw
 * 16-bit patterns.  The residual is added to the complete fp64 sum and the
 * result is rounded to bf16 exactly once (there is no intermediate rounding
 * of x.W^T).  The pages print no formula, data type or layout; these are the
 * plainest reading of the method they describe, with bf16 operands and the
 * nn.Linear layout.
 *
 * The accumulation is a plain fp64 loop in increasing k; bf16 values are
 * decoded and the RNE rounding is done here by hand (no CUDA, no bf16
 * library type).  OpenMP parallelises over output elements only.
 *
 * Every function here is pinned by the CPU test suite: exact integer brute
 * force, identity and permutation closed forms, linearity in x, invariance to
 * splitting K, exact x16 row scaling, and bit-for-bit agreement of the bf16
 * decode/encode with an independent library conversion.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp64.  A bf16 value is the top half of an IEEE binary32. */
double oracle_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The spacing of bf16 values at |v|: 2^(e-7) for 2^e <= |v| < 2^(e+1) when
 * |v| is normal (e >= -126), and the subnormal spacing 2^-133 below that. */
double oracle_ulp_bf16(double v)
{
    double a = fabs(v);
    if (!(a >= 0x1p-126)) /* zero, subnormal (and NaN) */
        return 0x1p-133;
    if (isinf(a))
        return INFINITY;
    int e;
    frexp(a, &e); /* a = f * 2^e, 0.5 <= f < 1, so 2^(e-1) <= a < 2^e */
    return ldexp(1.0, (e - 1) - 7);
}

/* fp64 -> bf16, round to nearest, ties to even, with one rounding step.
 * Overflow goes to +-inf (the largest finite bf16 is (2 - 2^-7) * 2^127;
 * anything at or above the midpoint to 2^128 rounds up to infinity). */
uint16_t oracle_bf16_round(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    double ulp = oracle_ulp_bf16(a);
    double q = a / ulp;          /* exact: division by a power of two */
    double qi = floor(q);        /* integer part, exact */
    double frac = q - qi;        /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(qi, 2.0) != 0.0))
        qi += 1.0;
    double r = qi * ulp;         /* exact, representable as bf16 */
    if (r >= 0x1p128)
        return sign | 0x7F80;
    float f = (float)r;          /* exact: every bf16 value is a float */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* One output element: the fp64 dot product of row m of x with row n of W. */
static void oracle_point(int64_t K, const uint16_t *xrow, const uint16_t *wrow,
                         double *y, double *s1)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double a = oracle_bf16_decode(xrow[k]);
        double b = oracle_bf16_decode(wrow[k]);
        acc += a * b;
        mag += fabs(a) * fabs(b);
    }
    *y = acc;
    *s1 = mag;
}

static void oracle_set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads the next parallel region will use. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full projection.  x [M,K], W [N,K], res [M,N] or NULL.
 * Outputs (each may be NULL): y_ref [M,N] fp64 (residual included),
 * s1 [M,N] fp64, y_bf16 [M,N] = RNE(y_ref).  Returns 0, or -1 on bad sizes.
 */
int oracle_linear(int64_t M, int64_t N, int64_t K,
                  const uint16_t *x, const uint16_t *W, const uint16_t *res,
                  double *y_ref, double *s1, uint16_t *y_bf16, int nthreads)
{
    if (M < 0 || N < 0 || K < 0)
        return -1;
    oracle_set_threads(nthreads);
    int64_t total = M * N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < total; ++i) {
        int64_t n = i / M, m = i % M; /* n outer keeps a W row hot */
        double y, mag;
        oracle_point(K, x + m * K, W + n * K, &y, &mag);
        if (res)
            y += oracle_bf16_decode(res[m * N + n]);
        if (y_ref)
            y_ref[m * N + n] = y;
        if (s1)
            s1[m * N + n] = mag;
        if (y_bf16)
            y_bf16[m * N + n] = oracle_bf16_round(y);
    }
    return 0;
}

/*
 * The same definition at chosen output points only (for spot checks of
 * full-size launches): point j is element (ms[j], ns[j]).
 */
int oracle_linear_points(int64_t M, int64_t N, int64_t K,
                         const uint16_t *x, const uint16_t *W,
                         const uint16_t *res, int64_t npts,
                         const int64_t *ms, const int64_t *ns,
                         double *y_ref, double *s1, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || npts < 0)
        return -1;
    for (int64_t j = 0; j < npts; ++j)
        if (ms[j] < 0 || ms[j] >= M || ns[j] < 0 || ns[j] >= N)
            return -1;
    oracle_set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < npts; ++j) {
        int64_t m = ms[j], n = ns[j];
        double y, mag;
        oracle_point(K, x + m * K, W + n * K, &y, &mag);
        if (res)
            y += oracle_bf16_decode(res[m * N + n]);
        y_ref[j] = y;
        if (s1)
            s1[j] = mag;
    }
    return 0;
}

/* Element-wise array forms of the three bf16 helpers above. */
void oracle_bf16_decode_array(int64_t n, const uint16_t *in, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_decode(in[i]);
}

void oracle_bf16_round_array(int64_t n, const double *in, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_round(in[i]);
}

void oracle_ulp_bf16_array(int64_t n, const double *in, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_ulp_bf16(in[i]);
}
