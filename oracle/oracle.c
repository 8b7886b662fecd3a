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
int oracle_agmm(int P, int64_t m_per_device, int64_t k, int64_t n, int rhs_transpose,
                const uint16_t *const *x_shards, const uint16_t *y,
                int64_t row_begin, int64_t row_end, int acc_double,
                float *out_f32, uint16_t *out_bf16, double *out_f64, int nthreads)
{
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
        for (int64_t kk = 0; kk < k; ++kk) xcat[i * k + kk] = oracle_bf16_to_f32(src[kk]);
    }
    for (int64_t kk = 0; kk < k; ++kk)
        for (int64_t j = 0; j < n; ++j)
            ycan[kk * n + j] = oracle_bf16_to_f32(rhs_transpose ? y[j * k + kk] : y[kk * n + j]);

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
            /* Step 4: cast to the output dtype (bf16, round to nearest even). */
            if (out_bf16)
                for (int64_t j = 0; j < n; ++j) out_bf16[i * n + j] = oracle_f32_to_bf16(acc[j]);
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
