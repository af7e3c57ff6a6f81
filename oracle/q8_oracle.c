/*
 * Q8_0 product oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow fp64 CPU statement of what the Q8_0 product computes, used to check the CUDA library. Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg load it; the library never does, and this file shares no code,
 * header or constant with it.
 *
 * Source: "logicaffeine_compile/spatial/passes/from_q8.rs", module doc (the product
 *   y[r, n] = sum_b s[b, n] * sum_i x[r, 32b + i] * q[32b + i, n],
 * Q8_0 blocks of 32 rows, one fp32 scale per block and column) and `q8_fold` (the fp32 carry starts at zero and every
 * block's sums are folded in).  Here every step is done in fp64:
 *   - bf16 -> fp64, int8 -> fp64 and fp32 -> fp64 are exact conversions;
 *   - x * q is exact in fp64 (8-bit by 7-bit significands);
 *   - the 32-term inner sum is formed first, then multiplied by the block's scale, then added to the carry, in the
 *     order of the formula (block b ascending, lane i ascending).
 * Beside y the oracle returns the error scale A[r, n] = sum_b |s[b, n]| * sum_i |x[r, 32b + i] * q[32b + i, n]|,
 * against which a GPU result is judged.
 *
 * Layouts (the pages' `W__q8`, `K x N` int8, and `W__q8_scale`, `K/32 x N` fp32, with N padded to whole 32-column
 * tiles, Np):  x is bf16 bit patterns [m][K]; q is int8 [K][Np]; s is fp32 [K/32][Np]; the output columns are the
 * `ncols` entries of `cols` (every n < Np when cols is NULL); y and a are fp64 [m][ncols].
 */
#include <stdint.h>
#include <string.h>

#define ORACLE_BLOCK 32 /* rows of a Q8_0 block (from_q8.rs, `Q8_BLOCK`) */

/* bf16 is the top half of an IEEE binary32: widen the bit pattern, then the float to double (both exact). */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t wide = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &wide, sizeof f);
    return (double)f;
}

static double absd(double v) { return v < 0.0 ? -v : v; }

/* One output: row r of x against column n of the Q8_0 weight. */
static void one_output(const uint16_t *x, const int8_t *q, const float *s, int K, int Np, int r, int64_t n,
                       double *y_out, double *a_out) {
    const int nblocks = K / ORACLE_BLOCK;
    double y = 0.0, a = 0.0; /* the carry starts at zero */
    for (int b = 0; b < nblocks; ++b) {
        double inner = 0.0, inner_abs = 0.0;
        for (int i = 0; i < ORACLE_BLOCK; ++i) {
            const int k = ORACLE_BLOCK * b + i;
            const double xv = bf16_bits_to_double(x[(int64_t)r * K + k]);
            const double qv = (double)q[(int64_t)k * Np + n];
            inner += xv * qv;
            inner_abs += absd(xv * qv);
        }
        const double sv = (double)s[(int64_t)b * Np + n];
        y += sv * inner;
        a += absd(sv) * inner_abs;
    }
    *y_out = y;
    *a_out = a;
}

/* y[r][j], a[r][j] for r < m and the j-th requested column.  Returns 0, or -1 on a shape the product does not take
 * (the applicability rule of from_q8.rs, `q8_gemv_applies`: m >= 1, K > 0 and a whole number of 32-row blocks). */
int oracle_q8_gemv(const uint16_t *x, const int8_t *q, const float *s, int m, int K, int Np, const int64_t *cols,
                   int64_t ncols, double *y, double *a) {
    if (m < 1 || K <= 0 || K % ORACLE_BLOCK != 0 || Np <= 0 || Np % ORACLE_BLOCK != 0) return -1;
    const int64_t count = cols ? ncols : Np;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t j = 0; j < count; ++j) {
        const int64_t n = cols ? cols[j] : j;
        for (int r = 0; r < m; ++r) one_output(x, q, s, K, Np, r, n, &y[(int64_t)r * count + j], &a[(int64_t)r * count + j]);
    }
    return 0;
}

/* The number of threads the OpenMP runtime will use (reported beside the CPU baseline). */
int oracle_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
