/* The oracle's loops on every host core (OpenMP) -- TEST INFRASTRUCTURE ONLY:
 * the bench's all-core CPU baseline.  Same arithmetic per element as
 * oracle.c (binary64, explicit fma, no contraction), split over threads:
 *
 *   copy, AXPY, BS5's vector updates, scatter: static chunks of the index
 *   range, results written to fresh arrays inside the loop (no separate copy
 *   of the inputs); every element is computed exactly as in oracle.c, so the
 *   results are bitwise the oracle's.
 *
 *   gather: one global row per iteration (CSR rowStarts/localIds, local ids
 *   ascending within a row), summed from +0.0 in ascending local order --
 *   bitwise the oracle's pass over the scatter table.
 *
 *   norm, dot: Dot2 [ORO] over each thread's contiguous chunk, the chunks'
 *   (sum, error) pairs combined in chunk order by TwoSum -- the sequential
 *   order within each chunk; the result agrees with the one-thread Dot2 to
 *   its accuracy, not bit for bit.
 *
 * [ORO] T. Ogita, S. M. Rump, S. Oishi, "Accurate sum and dot product",
 *       SIAM J. Sci. Comput. 26(6), 2005 -- Algorithm Dot2.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>

int oracle_omp_threads(void) { return omp_get_max_threads(); }

void oracle_omp_copy(int64_t n, const double *x, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        y[i] = x[i];
}

/* out_i = fma(alpha, x_i, beta * y_i) (out may be y). */
void oracle_omp_axpy(int64_t n, double alpha, const double *x, double beta, const double *y,
                     double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double by = beta * y[i];
        out[i] = fma(alpha, x[i], by);
    }
}

/* Dot2 over [lo, hi): *p + *s is the chunk's value (p the running sum, s the
 * accumulated errors). */
static void dot2_chunk(int64_t lo, int64_t hi, const double *x, const double *y, double *p_out,
                       double *s_out)
{
    double p = 0.0, s = 0.0;
    for (int64_t i = lo; i < hi; ++i) {
        double h = x[i] * y[i];
        double q = fma(x[i], y[i], -h);
        double t = p + h;
        double z = t - p;
        double e = (p - (t - z)) + (h - z);
        p = t;
        s = s + (e + q);
    }
    *p_out = p;
    *s_out = s;
}

double oracle_omp_dot2(int64_t n, const double *x, const double *y)
{
    int nt = omp_get_max_threads();
    double *part = (double *)malloc(sizeof(double) * 2 * (size_t)nt);
    if (!part)
        return NAN;
#pragma omp parallel num_threads(nt)
    {
        int t = omp_get_thread_num(), k = omp_get_num_threads();
        int64_t lo = n * t / k, hi = n * (t + 1) / k;
        dot2_chunk(lo, hi, x, y, &part[2 * t], &part[2 * t + 1]);
        if (k < nt && t == 0)  /* fewer threads than asked: empty chunks for the rest */
            for (int u = k; u < nt; ++u)
                part[2 * u] = part[2 * u + 1] = 0.0;
    }
    /* combine in chunk order: TwoSum of the running sums, errors summed */
    double p = 0.0, s = 0.0;
    for (int t = 0; t < nt; ++t) {
        double h = part[2 * t];
        double u = p + h;
        double z = u - p;
        double e = (p - (u - z)) + (h - z);
        p = u;
        s = s + (e + part[2 * t + 1]);
    }
    free(part);
    return p + s;
}

/* xo_i = fma(alpha, p_i, x_i), ro_i = fma(-alpha, Ap_i, r_i) (xo may be x,
 * ro may be r). */
void oracle_omp_cg_update(int64_t n, double alpha, const double *p, const double *Ap,
                          const double *x, const double *r, double *xo, double *ro)
{
    double nalpha = -alpha;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        xo[i] = fma(alpha, p[i], x[i]);
        ro[i] = fma(nalpha, Ap[i], r[i]);
    }
}

void oracle_omp_scatter(int64_t NL, const int32_t *ids, const double *qG, double *qL)
{
#pragma omp parallel for schedule(static)
    for (int64_t l = 0; l < NL; ++l)
        qL[l] = ids[l] >= 0 ? qG[ids[l]] : 0.0;
}

/* rowStarts[NG + 1], localIds[rowStarts[NG]]: row g holds locals
 * localIds[rowStarts[g] .. rowStarts[g+1]) in ascending order; only locals
 * below NL (the length of qL) contribute. */
void oracle_omp_gather(int64_t NL, int64_t NG, const int64_t *rowStarts, const int32_t *localIds,
                       const double *qL, double *qG)
{
#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < NG; ++g) {
        double s = 0.0;
        for (int64_t k = rowStarts[g]; k < rowStarts[g + 1]; ++k)
            if (localIds[k] < NL)
                s += qL[localIds[k]];
        qG[g] = s;
    }
}

/* Rows of a local-to-global table (setup, not an operation): rowStarts[NG+1]
 * and localIds[rowStarts[NG]] with each row's local ids ascending -- a
 * counting sort over ids (negative ids, the masked locals, belong to no
 * row).  rowStarts must hold NG + 1 zeros on entry; returns 0, or -1 when out
 * of memory. */
int oracle_rows(int64_t NL, int64_t NG, const int32_t *ids, int64_t *rowStarts, int32_t *localIds)
{
    for (int64_t l = 0; l < NL; ++l)
        if (ids[l] >= 0)
            ++rowStarts[ids[l] + 1];
    for (int64_t g = 0; g < NG; ++g)
        rowStarts[g + 1] += rowStarts[g];
    int64_t *next = (int64_t *)malloc(sizeof(int64_t) * (size_t)(NG > 0 ? NG : 1));
    if (!next)
        return -1;
    for (int64_t g = 0; g < NG; ++g)
        next[g] = rowStarts[g];
    for (int64_t l = 0; l < NL; ++l)
        if (ids[l] >= 0)
            localIds[next[ids[l]]++] = (int32_t)l;
    free(next);
    return 0;
}
