/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain, slow, double-precision CPU reference for causal grouped-query
 * attention of a prefill chunk against a cached prefix. Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never does. It shares no code, header or constant with the CUDA path.
 *
 * What it computes (exact attention, no tiling, no online update):
 *   for every chunk row i (query position P + i) and query head h, with
 *   g = h / (HQ / HKV)                         [page 1, Lesson: head h reads KV head h/4]
 *     s_j  = scale * sum_d q[i][h][d] * k[j][g][d],   j = 0 .. P + i
 *                                              [page 1, Lesson: row i sees keys j <= P + i]
 *     m    = max_j s_j
 *     w_j  = exp(s_j - m)
 *     Z    = sum_j w_j
 *     out[i][h][d] = (sum_j w_j * v[j][g][d]) / Z
 * in double, as the attention-v1 oracle is described ("double sums") on page 1
 * ("Inference Attention 2: Flash Prefill Against a Cached Prefix", Lesson), and
 * in the two-pass shape (maximum first, then exponentials and sums, then the
 * weighted values) of the double CPU reference in "FlashAttention and inference
 * kernels" (A working FlashAttention forward kernel). The score -> softmax ->
 * weighted-sum order is the one "Inference Attention 1: The Full Score Matrix"
 * (Lesson) names. The core is generic in HQ, HKV, D and scale so that small
 * hand-checkable cases (the worked example of "FlashAttention and inference
 * kernels", Exercises 1, has D = 1 and scale 1) run through the same code.
 *
 * Layouts: q [C][HQ][D], k and v [P + C][HKV][D], all fp32 row-major.
 * out is double [nrows][HQ][D], one block per requested chunk row.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

/* One (row, head) output: the definition above, written out. `s` is scratch
 * for the visible scores (n doubles). */
static void one_row_head(const float *q_row, const float *k, const float *v,
                         double *out_row, long n, int HKV, int D, int g,
                         double scale, double *s)
{
    long j;
    int d;
    double m = -INFINITY;
    for (j = 0; j < n; ++j) {
        const float *kj = k + ((size_t)j * HKV + g) * D;
        double dot = 0.0;
        for (d = 0; d < D; ++d)
            dot += (double)q_row[d] * (double)kj[d];
        s[j] = dot * scale;
        if (s[j] > m)
            m = s[j];
    }
    double Z = 0.0;
    for (j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        Z += s[j];
    }
    for (d = 0; d < D; ++d) {
        double acc = 0.0;
        for (j = 0; j < n; ++j)
            acc += s[j] * (double)v[((size_t)j * HKV + g) * D + d];
        out_row[d] = acc / Z;
    }
}

/*
 * oracle_prefill: out[r][h][:] for the chunk rows listed in rows[0..nrows).
 * rows == NULL means all C rows in order (nrows must then equal C).
 * nthreads <= 0 leaves the OpenMP default.
 * Returns 0, or a negative code for bad arguments / allocation failure.
 */
int oracle_prefill(const float *q, const float *k, const float *v, double *out,
                   long C, long P, int HQ, int HKV, int D, double scale,
                   const int *rows, long nrows, int nthreads)
{
    if (!q || !k || !v || !out || C < 0 || P < 0 || HQ <= 0 || HKV <= 0 ||
        D <= 0 || HQ % HKV != 0 || nrows < 0)
        return ORACLE_EINVAL;
    if (rows == NULL && nrows != C)
        return ORACLE_EINVAL;
    if (rows != NULL) {
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= C)
                return ORACLE_EINVAL;
    }
    const int group = HQ / HKV;
    const long pairs = nrows * (long)HQ;
    int failed = 0;

#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(P + C > 0 ? P + C : 1));
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < pairs; ++t) {
            if (!s) {
#pragma omp atomic write
                failed = 1;
                continue;
            }
            const long r = t / HQ;
            const int h = (int)(t % HQ);
            const long i = rows ? rows[r] : r;
            const long n = P + i + 1;
            one_row_head(q + ((size_t)i * HQ + h) * D, k, v,
                         out + ((size_t)r * HQ + h) * D, n, HKV, D,
                         h / group, scale, s);
        }
        free(s);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/* The number of OpenMP threads a parallel region would use. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
