/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the seven Benchmark
 * Streaming (BS) operations and the box-mesh numbering they run on.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg
 * use it.  It shares no source with the CUDA path.
 *
 * Arithmetic: IEEE binary64, round to nearest even, compiled with
 * -ffp-contract=off so that every fused multiply-add is an explicit fma().
 *
 * Sources (paper titles, with the part of each that a function follows):
 *   [P1] "Portable high-order finite element kernels I: Streaming Operations"
 *        -- BS tests list, CG vector operations, eq. (3) (v_L = Z v_G),
 *        the gather/scatter kernel descriptions (BS6 CSR gather, BS7
 *        scatterIds with negative = masked).
 *   [P2] "GPU accelerated spectral finite elements on all-hex meshes"
 *        -- local-to-global table I_{l->g} (scatter) and global-to-local
 *        table I_{g->l} (gather sums the local copies of a global node).
 *   [ORO] T. Ogita, S. M. Rump, S. Oishi, "Accurate sum and dot product",
 *        SIAM J. Sci. Comput. 26(6), 2005 -- Algorithm Dot2 (TwoProduct by
 *        fma, TwoSum by Knuth).
 */
#include <math.h>
#include <stdint.h>

/* BS1 copy [P1, BS test list]: y_i = x_i. */
void oracle_copy(int64_t n, const double *x, double *y)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = x[i];
}

/* BS2 AXPY [P1, CG vector operations, "vector addition y = alpha x + beta y"]:
 * y_i = fma(alpha, x_i, beta * y_i), the product beta*y_i rounded first. */
void oracle_axpy(int64_t n, double alpha, const double *x, double beta, double *y)
{
    for (int64_t i = 0; i < n; ++i) {
        double by = beta * y[i];
        y[i] = fma(alpha, x[i], by);
    }
}

/* Plain sequential dot product: s = (((0 + x0 y0) + x1 y1) + ...), every
 * product and sum rounded.  Reported beside the accurate value. */
double oracle_dot_plain(int64_t n, const double *x, const double *y)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double p = x[i] * y[i];
        s = s + p;
    }
    return s;
}

/* BS4 inner product / BS3 norm (x.x) [P1, CG vector operations "dot
 * product" and "norm: alpha = x.x"], evaluated by Dot2 [ORO]: the result is
 * as accurate as a dot product computed in twice the working precision and
 * then rounded.  The sum order is i = 0, 1, ..., n-1. */
double oracle_dot2(int64_t n, const double *x, const double *y)
{
    double p = 0.0, s = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        /* TwoProduct: h + q == x_i * y_i exactly. */
        double h = x[i] * y[i];
        double q = fma(x[i], y[i], -h);
        /* TwoSum: t + e == p + h exactly. */
        double t = p + h;
        double z = t - p;
        double e = (p - (t - z)) + (h - z);
        p = t;
        s = s + (e + q);
    }
    return p + s;
}

/* BS5 fused CG update [P1, BS test list: steps 8-10 of the CG method fused
 * into one operation]: x_i <- x_i + alpha p_i, r_i <- r_i - alpha Ap_i, each
 * by one fma.  The residual norm r.r of the updated r is taken separately by
 * oracle_dot2(r, r). */
void oracle_cg_update(int64_t n, double alpha, const double *p, const double *Ap,
                      double *x, double *r)
{
    double nalpha = -alpha;
    for (int64_t i = 0; i < n; ++i) {
        x[i] = fma(alpha, p[i], x[i]);
        r[i] = fma(nalpha, Ap[i], r[i]);
    }
}

/* BS7 scatter [P1, eq. (3) v_L = Z v_G and the scatterIds description; P2,
 * I_{l->g}]: q_L[l] = q_G[ids[l]]; a negative id marks a masked local degree
 * of freedom, whose value is +0.0. */
void oracle_scatter(int64_t NL, const int32_t *ids, const double *qG, double *qL)
{
    for (int64_t l = 0; l < NL; ++l)
        qL[l] = ids[l] >= 0 ? qG[ids[l]] : 0.0;
}

/* BS6 gather [P1, gather operator Z^T; P2, I_{g->l}: a global node receives
 * the sum of its local copies]: q_G = Z^T q_L.  Written as one pass over the
 * scatter table in ascending local index, so that every global value is
 * ((+0.0 + q_L[l1]) + q_L[l2]) + ... with l1 < l2 < ...  Masked locals do
 * not contribute. */
void oracle_gather(int64_t NL, int64_t NG, const int32_t *ids, const double *qL, double *qG)
{
    for (int64_t g = 0; g < NG; ++g)
        qG[g] = 0.0;
    for (int64_t l = 0; l < NL; ++l)
        if (ids[l] >= 0)
            qG[ids[l]] += qL[l];
}

/* The 24 proper rotations of the reference cube, in a fixed order (mesh
 * numbering convention): the axis permutations pi of (0, 1, 2) in
 * lexicographic order, and for each the flip masks f = 0 .. 7 (bit a:
 * output axis a reversed), keeping those whose signed permutation matrix
 * has determinant sign(pi) (-1)^popcount(f) = +1.  Index 0 is the identity. */
static void cube_rotations(int perm[24][3], int flip[24][3])
{
    static const int P[6][3] = {{0, 1, 2}, {0, 2, 1}, {1, 0, 2}, {1, 2, 0}, {2, 0, 1}, {2, 1, 0}};
    static const int sign[6] = {1, -1, -1, 1, 1, -1};
    int o = 0;
    for (int p = 0; p < 6; ++p)
        for (int f = 0; f < 8; ++f) {
            int flips = (f & 1) + ((f >> 1) & 1) + ((f >> 2) & 1);
            if (sign[p] * ((flips & 1) ? -1 : 1) != 1)
                continue;
            for (int a = 0; a < 3; ++a) {
                perm[o][a] = P[p][a];
                flip[o][a] = (f >> a) & 1;
            }
            ++o;
        }
}

/* Box-mesh local-to-global table [P1, eq. (1) K hexahedra, (p+1)^3 GLL
 * nodes per element, N_L = K(p+1)^3; P2, I_{l->g}].
 *
 * The mesh is E x E x E hexahedra of degree N on a box.  Lattice element
 * (ex, ey, ez) has number ex + E (ey + E ez).  Storage slot s holds lattice
 * element e = elemPerm[s], with orientation o = orient[e] (0 if orient is
 * NULL).  Its local node (i, j, k), 0 <= i, j, k <= N, has local index
 * l = s (N+1)^3 + i + (N+1)(j + (N+1) k); with v = (i, j, k) and rotation o
 * of cube_rotations, w_a = v[perm_a], or N - v[perm_a] if axis a is
 * flipped, and the node sits on lattice node (ex N + w_0, ey N + w_1,
 * ez N + w_2) of the (E N + 1)^3 lattice, numbered x fastest; that lattice
 * node's global id is nodePerm[lattice number].  With mask_boundary != 0
 * every local node on the box boundary gets -1. */
void oracle_box_scatter_ids(int E, int N, const int32_t *elemPerm, const int32_t *nodePerm,
                            int mask_boundary, const uint8_t *orient, int32_t *ids)
{
    int perm[24][3], flip[24][3];
    cube_rotations(perm, flip);
    int64_t K = (int64_t)E * E * E;
    int64_t q = N + 1;
    int64_t M = (int64_t)E * N + 1;
    for (int64_t s = 0; s < K; ++s) {
        int64_t e = elemPerm[s];
        int64_t ex = e % E;
        int64_t ey = (e / E) % E;
        int64_t ez = e / ((int64_t)E * E);
        int o = orient ? orient[e] : 0;
        for (int64_t k = 0; k < q; ++k)
            for (int64_t j = 0; j < q; ++j)
                for (int64_t i = 0; i < q; ++i) {
                    int64_t v[3] = {i, j, k}, w[3];
                    for (int a = 0; a < 3; ++a)
                        w[a] = flip[o][a] ? N - v[perm[o][a]] : v[perm[o][a]];
                    int64_t gx = ex * N + w[0], gy = ey * N + w[1], gz = ez * N + w[2];
                    int64_t L = gx + M * (gy + M * gz);
                    int64_t l = s * q * q * q + i + q * (j + q * k);
                    int on_boundary = gx == 0 || gy == 0 || gz == 0 ||
                                      gx == M - 1 || gy == M - 1 || gz == M - 1;
                    ids[l] = (mask_boundary && on_boundary) ? -1 : nodePerm[L];
                }
    }
}
