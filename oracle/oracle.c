/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU implementation of the all-gather
 * matmul, used to check the CUDA path.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * What it computes (the definition, not the schedule):
 *
 *   Xcat = concat over r = 0..P-1 of X_r          -- rank order along rows
 *   Ycan = Y            if rhs_transpose == 0      -- Y stored [k, n]
 *        = transpose(Y) if rhs_transpose != 0      -- Y stored [n, k]
 *   O[i, j] = round_bf16( sum_{kk = 0..k-1} Xcat[i, kk] * Ycan[kk, j] )
 *
 * Sources:
 *  - "tpu_inference/kernels/collectives/all_gather_matmul.py", docstring of
 *    all_gather_matmul: the result is all-gather(x, axis=0) @ y; the
 *    rhs_transpose branch of _do_mxu contracts dimension 1 of both operands,
 *    i.e. uses Y stored [n, k]; every dot uses preferred_element_type=float32
 *    and the result is cast to x.dtype (bf16 here).
 *  - "AllGather-GEMM" (Triton-distributed Ascend tutorial), function
 *    torch_allgather_gemm: all_gather, then torch.cat along dim 0, then
 *    torch.matmul -- the same concatenation order.
 *
 * Readings where the pages are silent:
 *  - The float32 accumulation order is not fixed by the pages; this oracle
 *    sums in ascending kk.  Products of two bf16 values are exact in float32
 *    (8-bit x 8-bit significands), so contraction to FMA does not change any
 *    result.
 *  - The float32 -> bf16 cast is round-to-nearest-even; NaN stays NaN.
 *
 * The same definition with fp16 inputs and output (oracle_agmm_typed): the
 * element type changes only the two conversions, each written from the IEEE
 * binary16 layout.
 *
 * A second accumulation mode sums in double precision.  It is not the pages'
 * arithmetic; the tests use it as a near-exact reference for error bounds.
 *
 * Parallelism: rows are split across OpenMP threads; each output element is
 * still summed by one thread in ascending kk, so the thread count never
 * changes a result.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE-754 binary32 bit pattern. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 value to the nearest bf16, ties to even. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) {
        /* NaN: keep sign, force a quiet NaN payload that survives truncation. */
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    /* Adding 0x7FFF plus the kept LSB rounds the discarded half to nearest,
     * breaking a tie toward an even kept LSB.  A carry into the exponent is
     * the correct rounding (up to infinity at the top). */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* IEEE-754 binary16 (fp16): 1 sign bit, 5 exponent bits (bias 15), 10
 * fraction bits.  Exponent 0 encodes zero and the subnormals f * 2^-24;
 * exponent 31 encodes infinity (fraction 0) and NaN. */
float oracle_f16_to_f32(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1F;
    const int f = h & 0x3FF;
    float v;
    if (e == 0) {
        v = (float)f * (1.0f / 16777216.0f); /* f * 2^-24, exact in binary32 */
    } else if (e == 31) {
        uint32_t u = f ? 0x7FC00000u : 0x7F800000u;
        memcpy(&v, &u, sizeof v);
    } else {
        /* (1024 + f) * 2^(e - 25): build the binary32 pattern directly */
        uint32_t u = ((uint32_t)(e - 15 + 127) << 23) | ((uint32_t)f << 13);
        memcpy(&v, &u, sizeof v);
    }
    return sign ? -v : v;
}

/* Round a binary32 value to the nearest fp16, ties to even.  Overflow
 * rounds to infinity; NaN stays NaN (quiet, sign kept). */
uint16_t oracle_f32_to_f16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    const int exp = (int)((u >> 23) & 0xFF);
    const uint32_t frac = u & 0x7FFFFFu;
    if (exp == 255) return (uint16_t)(sign | (frac ? 0x7E00u : 0x7C00u));
    if (exp == 0) return sign; /* binary32 zero or subnormal: far below 2^-25 */
    const int e = exp - 127 + 15; /* fp16 exponent field if the result is normal */
    if (e >= 31) return (uint16_t)(sign | 0x7C00u);
    const uint32_t m = frac | 0x800000u; /* 24-bit significand, value m * 2^(exp-150) */
    /* Units of the result's last place: 2^(e-25) when normal, 2^-24 when subnormal. */
    const int shift = e >= 1 ? 13 : 14 - e;
    if (shift > 31) return sign;
    const uint32_t q = m >> shift;
    const uint32_t rem = m & ((1u << shift) - 1u);
    const uint32_t half = 1u << (shift - 1);
    const uint32_t up = (rem > half || (rem == half && (q & 1u))) ? 1u : 0u;
    if (e >= 1) {
        /* q holds the implicit bit at 0x400; a carry into the exponent is correct */
        return (uint16_t)(sign | (uint32_t)(((uint32_t)(e - 1) << 10) + q + up));
    }
    return (uint16_t)(sign | (q + up)); /* subnormal; a carry makes the smallest normal */
}

void oracle_f16_array_to_f32(const uint16_t *src, float *dst, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) dst[i] = oracle_f16_to_f32(src[i]);
}

void oracle_f32_array_to_f16(const float *src, uint16_t *dst, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) dst[i] = oracle_f32_to_f16(src[i]);
}

void oracle_bf16_array_to_f32(const uint16_t *src, float *dst, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) dst[i] = oracle_bf16_to_f32(src[i]);
}

void oracle_f32_array_to_bf16(const float *src, uint16_t *dst, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) dst[i] = oracle_f32_to_bf16(src[i]);
}

/*
 * Rows [row_begin, row_end) of O = concat(X_0..X_{P-1}) @ Ycan.
 *
 *   x_shards[r]  : P pointers, each to a row-major [m_per_device, k] bf16 array
 *   y            : bf16, row-major [k, n] (rhs_transpose == 0) or [n, k] (!= 0)
 *   acc_double   : 0 -> float32 accumulation (the pages' precision),
 *                  1 -> double accumulation (test reference only)
 *   out_f32      : [rows, n] float32 sums (acc_double == 0), or NULL
 *   out_bf16     : [rows, n] bf16 bit patterns of out_f32, or NULL
 *   out_f64      : [rows, n] double sums (acc_double == 1), or NULL
 *   nthreads     : OpenMP threads (<= 0: library default)
 *
 * Returns 0 on success, -1 on invalid arguments, -2 on allocation failure.
 */
/* Element types of the 16-bit inputs and output. */
enum { ORACLE_BF16 = 0, ORACLE_F16 = 1 };

static float elem_to_f32(uint16_t b, int elem)
{
    return elem == ORACLE_F16 ? oracle_f16_to_f32(b) : oracle_bf16_to_f32(b);
}

static uint16_t f32_to_elem(float f, int elem)
{
    return elem == ORACLE_F16 ? oracle_f32_to_f16(f) : oracle_f32_to_bf16(f);
}

/*
 * The same product with the element type of X, Y and the 16-bit output given
 * by `elem` (ORACLE_BF16 or ORACLE_F16); out_bf16 then receives that type's
 * bit patterns.  Products of two fp16 values (11-bit significands) are also
 * exact in float32.
 */
int oracle_agmm_typed(int P, int64_t m_per_device, int64_t k, int64_t n, int rhs_transpose,
                      const uint16_t *const *x_shards, const uint16_t *y,
                      int64_t row_begin, int64_t row_end, int acc_double,
                      float *out_f32, uint16_t *out_bf16, double *out_f64, int nthreads, int elem);

int oracle_agmm(int P, int64_t m_per_device, int64_t k, int64_t n, int rhs_transpose,
                const uint16_t *const *x_shards, const uint16_t *y,
                int64_t row_begin, int64_t row_end, int acc_double,
                float *out_f32, uint16_t *out_bf16, double *out_f64, int nthreads)
{
    return oracle_agmm_typed(P, m_per_device, k, n, rhs_transpose, x_shards, y, row_begin, row_end,
                             acc_double, out_f32, out_bf16, out_f64, nthreads, ORACLE_BF16);
}

int oracle_agmm_typed(int P, int64_t m_per_device, int64_t k, int64_t n, int rhs_transpose,
                      const uint16_t *const *x_shards, const uint16_t *y,
                      int64_t row_begin, int64_t row_end, int acc_double,
                      float *out_f32, uint16_t *out_bf16, double *out_f64, int nthreads, int elem)
{
    if (elem != ORACLE_BF16 && elem != ORACLE_F16) return -1;
    if (P < 1 || m_per_device < 1 || k < 1 || n < 1 || !x_shards || !y) return -1;
    const int64_t M = (int64_t)P * m_per_device;
    if (row_begin < 0 || row_end > M || row_begin > row_end) return -1;
    for (int r = 0; r < P; ++r)
        if (!x_shards[r]) return -1;
    if (acc_double && !out_f64) return -1;
    if (!acc_double && !out_f32 && !out_bf16) return -1;
    const int64_t rows = row_end - row_begin;
    if (rows == 0) return 0;

    /* Step 1: the gathered LHS, written out explicitly (only the rows asked
     * for): global row i is row (i mod m_per_device) of shard i / m_per_device. */
    float *xcat = (float *)malloc((size_t)(rows * k) * sizeof(float));
    /* Step 2: Ycan = Y or its transpose, as a [k, n] float32 array. */
    float *ycan = (float *)malloc((size_t)(k * n) * sizeof(float));
    if (!xcat || !ycan) {
        free(xcat);
        free(ycan);
        return -2;
    }
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t g = row_begin + i;
        const uint16_t *src = x_shards[g / m_per_device] + (g % m_per_device) * k;
        for (int64_t kk = 0; kk < k; ++kk) xcat[i * k + kk] = elem_to_f32(src[kk], elem);
    }
    for (int64_t kk = 0; kk < k; ++kk)
        for (int64_t j = 0; j < n; ++j)
            ycan[kk * n + j] = elem_to_f32(rhs_transpose ? y[j * k + kk] : y[kk * n + j], elem);

    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < rows; ++i) {
        /* Step 3: O[i, :] = sum over kk, ascending, of Xcat[i, kk] * Ycan[kk, :]. */
        const float *xr = xcat + i * k;
        if (acc_double) {
            double *acc = out_f64 + i * n;
            for (int64_t j = 0; j < n; ++j) acc[j] = 0.0;
            for (int64_t kk = 0; kk < k; ++kk) {
                const double a = (double)xr[kk];
                const float *yr = ycan + kk * n;
                for (int64_t j = 0; j < n; ++j) acc[j] += a * (double)yr[j];
            }
        } else {
            float *acc = out_f32 ? out_f32 + i * n : (float *)malloc((size_t)n * sizeof(float));
            if (!acc) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                failed = 1;
                continue;
            }
            for (int64_t j = 0; j < n; ++j) acc[j] = 0.0f;
            for (int64_t kk = 0; kk < k; ++kk) {
                const float a = xr[kk];
                const float *yr = ycan + kk * n;
                for (int64_t j = 0; j < n; ++j) acc[j] += a * yr[j];
            }
            /* Step 4: cast to the output dtype (bf16 or fp16, round to nearest even). */
            if (out_bf16)
                for (int64_t j = 0; j < n; ++j) out_bf16[i * n + j] = f32_to_elem(acc[j], elem);
            if (!out_f32) free(acc);
        }
    }
    free(xcat);
    free(ycan);
    return failed ? -2 : 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
