/*
 * CPU oracle for the heterogeneous-rank LoRA delta -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package smoke check and the benchmark's CPU-baseline leg
 * may load this file's library.  It shares no code, header or constant with the
 * CUDA library: it decodes fp16 itself, reads the adapters from the caller's
 * host-store arrays (never from a device pool) and computes in fp64 with plain
 * loops, so that a reader can check each line against the definition.
 *
 * Definition followed (written out, no blocking, fusion or reordering):
 *
 *   h = x W + s * x A B                     per token, with its own adapter
 *
 *   - S-LoRA: Serving Thousands of Concurrent LoRA Adapters (explainer),
 *     "What this paper explains": A is d_in x r, B is r x d_out, and the delta is
 *     kept separate from the base instead of merged;  "How to read the paper",
 *     item 2: the forward is h = xW + xAB.
 *   - S-LoRA: Multiplexing Thousands of Fine-Tuned Adapters on a Single GPU,
 *     section 2 pseudocode ("Batched S-LoRA Vector Matrix Addition"): for each
 *     token i, look up that token's adapter factors, form (x_i A) B, multiply by
 *     the adapter's scaling and add it to the base output.
 *
 * The base output x W is an input here (y0): the base model is not part of the
 * delta.  With At[j][k] = A[k][j] (one hidden-length row per rank index j, the
 * layout a pool page holds), for a token t whose adapter is a:
 *
 *   u_j      = sum_{k < d} x[t][k] * At_a[j][k]                 (j < r_a)
 *   ref[t][n] = y0[t][n] + s_a * sum_{j < r_a} u_j * B_a[j][n]
 *
 * and a token whose adapter index is -1 keeps ref[t][n] = y0[t][n].
 * Every input is an fp16 value, upcast exactly; every sum is fp64.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, from the format's definition:
 * sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double slora_oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);                /* subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25);    /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* OpenMP threads for later calls (n > 0); the arithmetic does not depend on it. */
void slora_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int slora_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * ref[i][n] for the tokens listed in sel[0..n_sel) (sel == NULL: every token,
 * n_sel must then equal T).
 *
 *   x, y0       fp16 bits, [T][d] row-major
 *   idx         adapter index per token, -1 = base only
 *   rank[a], scaling[a]          for a < n_adapters
 *   At[a], B[a] fp16 bits, [rank[a]][d] row-major (NULL allowed if unused)
 *   out         double [n_sel][d]
 *
 * Returns 0, or -1 on an index outside [−1, n_adapters) / a NULL factor that a
 * token needs.
 */
int slora_oracle_delta(int32_t T, int32_t d,
                       const uint16_t *x, const uint16_t *y0, const int32_t *idx,
                       int32_t n_adapters, const int32_t *rank, const double *scaling,
                       const uint16_t *const *At, const uint16_t *const *B,
                       int64_t n_sel, const int32_t *sel, double *out)
{
    int bad = 0;
    if (sel == NULL && n_sel != T)
        return -1;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < n_sel; ++i) {
        int32_t t = sel ? sel[i] : (int32_t)i;
        double *o = out + (size_t)i * (size_t)d;
        if (t < 0 || t >= T) { bad = 1; continue; }
        const uint16_t *xt = x + (size_t)t * (size_t)d;
        const uint16_t *yt = y0 + (size_t)t * (size_t)d;
        for (int32_t n = 0; n < d; ++n)
            o[n] = slora_oracle_half_to_double(yt[n]);
        int32_t a = idx[t];
        if (a == -1)
            continue;
        if (a < 0 || a >= n_adapters || At[a] == NULL || B[a] == NULL) { bad = 1; continue; }
        int32_t r = rank[a];
        double s = scaling[a];
        double *u = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
        /* shrink: u = x_t A */
        for (int32_t j = 0; j < r; ++j) {
            const uint16_t *arow = At[a] + (size_t)j * (size_t)d;
            double acc = 0.0;
            for (int32_t k = 0; k < d; ++k)
                acc += slora_oracle_half_to_double(xt[k]) * slora_oracle_half_to_double(arow[k]);
            u[j] = acc;
        }
        /* expand: ref = y0 + s * u B */
        for (int32_t n = 0; n < d; ++n) {
            double acc = 0.0;
            for (int32_t j = 0; j < r; ++j)
                acc += u[j] * slora_oracle_half_to_double(B[a][(size_t)j * (size_t)d + n]);
            o[n] += s * acc;
        }
        free(u);
    }
    return bad ? -1 : 0;
}
