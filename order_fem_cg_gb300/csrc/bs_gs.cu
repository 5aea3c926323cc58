// bs_gs.cu -- BS6 gather (q_G = Z^T q_L), BS7 scatter (q_L = Z q_G), and the
// streaming sequence of one CG iteration.
//
// "Portable high-order finite element kernels I: Streaming Operations":
// Z is the N_L x N_G Boolean scatter operator of eq. (3) with one nonzero
// per row; BS7 reads it as the table scatterIds (negative = masked), BS6
// reads Z^T as a CSR matrix without values whose rows (global nodes) are
// grouped by blockStarts so that each thread block stages about
// NODES_PER_BLOCK entries in shared memory.  "GPU accelerated spectral
// finite elements on all-hex meshes": the local-to-global and
// global-to-local tables these are.
//
// GB300 design:
//  * gather: one block of 256 threads per row segment (<= SEG CSR entries).
//    Phase 1 loads the segment's local ids coalesced, issues all of its
//    random q_L reads at once (SEG/256 independent 8-byte loads per
//    thread, no L1 allocation) and parks the values in shared memory with
//    the segment's row starts.  Phase 2 gives each thread whole rows: it
//    sums a row's values in ascending local index from +0.0 and stores q_G
//    coalesced.  No atomics; the sum order is the definition's.
//  * scatter: persistent grid over groups of 4 local entries: one 16-byte
//    id load, 4 independent random q_G reads, one 32-byte q_L store;
//    UNROLL groups in flight per thread.
//  * every table entry is range-checked; a bad entry is skipped (never
//    dereferenced) and raises the context's device error flag.
#include <cuda_runtime.h>

#include "bs_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kScatterUnroll = 2;

__device__ __forceinline__ double ld_random(const double *p)
{
    double v;
    asm volatile("ld.global.nc.L1::no_allocate.f64 %0, [%1];" : "=d"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ int32_t ld_index(const int32_t *p)
{
    int32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ int4 ld_index4(const int32_t *p)
{
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_vec4(double *p, double a, double b, double c, double d)
{
    asm volatile("st.global.L1::no_allocate.v4.f64 [%0], {%1,%2,%3,%4};" ::"l"(p), "d"(a), "d"(b),
                 "d"(c), "d"(d)
                 : "memory");
}

__device__ __forceinline__ bool in_range(int32_t i, int64_t n)
{
    return static_cast<uint64_t>(static_cast<uint32_t>(i)) < static_cast<uint64_t>(n) && i >= 0;
}

// ------------------------------------------------------------------ BS6
template <int SEG>
__global__ void __launch_bounds__(kThreads)
    gather_kernel(const int32_t *__restrict__ rowStarts, const int32_t *__restrict__ localIds,
                  const int32_t *__restrict__ blockStarts, const double *__restrict__ qL,
                  double *__restrict__ qG, int64_t NL, int64_t NG, int64_t nnz, int *err)
{
    constexpr int PER = SEG / kThreads;
    __shared__ double vals[SEG];
    __shared__ uint16_t rs[SEG + 1];  // row starts relative to the segment, <= SEG
    static_assert(SEG < 65536, "row offsets are staged as 16-bit");

    const int32_t r0 = blockStarts[blockIdx.x];
    const int32_t r1 = blockStarts[blockIdx.x + 1];
    const int32_t nrows = r1 - r0;
    if (r0 < 0 || nrows < 0 || r1 > NG || nrows > SEG) {
        if (threadIdx.x == 0)
            atomicOr(err, BS_DEVERR_BOUNDS);
        return;
    }
    const int32_t e0 = rowStarts[r0];
    const int32_t e1 = rowStarts[r1];
    const int32_t ne = e1 - e0;
    if (e0 < 0 || ne < 0 || e1 > nnz || ne > SEG) {
        if (threadIdx.x == 0)
            atomicOr(err, BS_DEVERR_BOUNDS);
        return;
    }

    bool bad = false;
    int32_t id[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int j = threadIdx.x + k * kThreads;
        id[k] = j < ne ? ld_index(localIds + e0 + j) : 0;
    }
    for (int j = threadIdx.x; j <= nrows; j += kThreads) {
        const int32_t o = rowStarts[r0 + j] - e0;
        if (o < 0 || o > ne)
            bad = true;
        rs[j] = static_cast<uint16_t>(o < 0 ? 0 : (o > ne ? ne : o));
    }
    double v[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int j = threadIdx.x + k * kThreads;
        v[k] = 0.0;
        if (j < ne) {
            if (in_range(id[k], NL))
                v[k] = ld_random(qL + id[k]);
            else
                bad = true;
        }
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int j = threadIdx.x + k * kThreads;
        if (j < ne)
            vals[j] = v[k];
    }
    __syncthreads();

    for (int k = threadIdx.x; k < nrows; k += kThreads) {
        const int32_t a = rs[k], z = rs[k + 1];
        double s = 0.0;
        if (z < a) {
            bad = true;
        } else if (z > a) {
            // (+0.0 + v_a) + ... equals v_a + ... except that it is never
            // -0.0: skip the first addition, then map -0.0 to +0.0.
            s = vals[a];
            for (int32_t j = a + 1; j < z; ++j)
                s += vals[j];
            if ((__double_as_longlong(s) << 1) == 0)
                s = 0.0;
        }
        qG[r0 + k] = s;
    }
    if (bad)
        atomicOr(err, BS_DEVERR_BOUNDS);
}

// ------------------------------------------------------------------ BS7
// ids 16-byte aligned, qL 32-byte aligned; groups of 4 entries.
template <int UNROLL>
__global__ void __launch_bounds__(kThreads)
    scatter4_kernel(const int32_t *__restrict__ ids, const double *__restrict__ qG,
                    double *__restrict__ qL, int64_t ngroups, int64_t NL, int64_t NG, int *err)
{
    const int64_t gid = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    bool bad = false;
    for (int64_t b = gid; b < ngroups; b += stride * UNROLL) {
        int4 id[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < ngroups)
                id[u] = ld_index4(ids + 4 * (b + u * stride));
        double v[UNROLL][4];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < ngroups) {
                const int32_t g[4] = {id[u].x, id[u].y, id[u].z, id[u].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    v[u][c] = 0.0;
                    if (g[c] >= 0) {
                        if (g[c] < NG)
                            v[u][c] = ld_random(qG + g[c]);
                        else
                            bad = true;
                    }
                }
            }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < ngroups)
                st_vec4(qL + 4 * (b + u * stride), v[u][0], v[u][1], v[u][2], v[u][3]);
    }
    const int64_t l = 4 * ngroups + gid;
    if (l < NL) {
        const int32_t g = ids[l];
        double v = 0.0;
        if (g >= 0) {
            if (g < NG)
                v = qG[g];
            else
                bad = true;
        }
        qL[l] = v;
    }
    if (bad)
        atomicOr(err, BS_DEVERR_BOUNDS);
}

// Any alignment: one entry per thread and step.
__global__ void __launch_bounds__(kThreads)
    scatter1_kernel(const int32_t *__restrict__ ids, const double *__restrict__ qG,
                    double *__restrict__ qL, int64_t NL, int64_t NG, int *err)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    bool bad = false;
    for (int64_t l = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; l < NL;
         l += stride) {
        const int32_t g = ids[l];
        double v = 0.0;
        if (g >= 0) {
            if (g < NG)
                v = ld_random(qG + g);
            else
                bad = true;
        }
        qL[l] = v;
    }
    if (bad)
        atomicOr(err, BS_DEVERR_BOUNDS);
}

int check_tables(bs_ctx *ctx, const char *name, const bs_gs_dev *t, bool need_csr)
{
    if (!t)
        return bs_set_error(ctx, BS_EINVAL, "%s: NULL table struct", name);
    if (t->NL < 0 || t->NG < 0 || t->NL > INT32_MAX || t->NG >= INT32_MAX)
        return bs_set_error(ctx, BS_EINVAL, "%s: bad table sizes", name);
    if (t->NL > 0 && !t->scatterIds)
        return bs_set_error(ctx, BS_EINVAL, "%s: NULL scatterIds", name);
    if (need_csr) {
        if (t->nnz < 0 || t->nnz > t->NL || t->nblocks < 0 || t->nblocks >= INT32_MAX ||
            (t->NG > 0 && t->nblocks == 0))
            return bs_set_error(ctx, BS_EINVAL, "%s: bad CSR sizes", name);
        if (t->seg_max < 1 || t->seg_max > BS_GATHER_SEG_MAX)
            return bs_set_error(ctx, BS_EINVAL, "%s: seg_max %d outside [1, %d]", name,
                                t->seg_max, BS_GATHER_SEG_MAX);
        if (!t->rowStarts || !t->blockStarts || (t->nnz > 0 && !t->localIds))
            return bs_set_error(ctx, BS_EINVAL, "%s: NULL CSR table", name);
    }
    return BS_OK;
}

template <int SEG>
void launch_gather(const bs_ctx *ctx, const bs_gs_dev *t, const double *qL, double *qG,
                   cudaStream_t s)
{
    gather_kernel<SEG><<<static_cast<unsigned>(t->nblocks), kThreads, 0, s>>>(
        t->rowStarts, t->localIds, t->blockStarts, qL, qG, t->NL, t->NG, t->nnz, ctx->dev_err);
}

} // namespace

extern "C" int bs_gather(bs_ctx *ctx, const bs_gs_dev *t, const double *qL, double *qG,
                         void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (int st = check_tables(ctx, "bs_gather", t, true))
        return st;
    if ((t->NL > 0 && !qL) || (t->NG > 0 && !qG))
        return bs_set_error(ctx, BS_EINVAL, "bs_gather: NULL vector");
    if (bs_overlap(qL, 8 * t->NL, qG, 8 * t->NG))
        return bs_set_error(ctx, BS_EINVAL, "bs_gather: qL and qG overlap");
    if ((reinterpret_cast<uintptr_t>(qL) | reinterpret_cast<uintptr_t>(qG)) & 7u)
        return bs_set_error(ctx, BS_EINVAL, "bs_gather: vectors must be 8-byte aligned");
    if (int st = bs_check_device(ctx))
        return st;
    if (t->NG == 0)
        return BS_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (t->plan && !(ctx->tune.small_onepass && 8 * t->NL <= kOnePassGatherBytes))
        return bs_gather_planned(ctx, t, qL, qG, s);
    if (t->seg_max <= 1024)
        launch_gather<1024>(ctx, t, qL, qG, s);
    else if (t->seg_max <= 2048)
        launch_gather<2048>(ctx, t, qL, qG, s);
    else
        launch_gather<4096>(ctx, t, qL, qG, s);
    BS_LAUNCH_CHECK(ctx, "gather_kernel");
    return BS_OK;
}

extern "C" int bs_scatter(bs_ctx *ctx, const bs_gs_dev *t, const double *qG, double *qL,
                          void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (int st = check_tables(ctx, "bs_scatter", t, false))
        return st;
    if ((t->NL > 0 && !qL) || (t->NG > 0 && !qG))
        return bs_set_error(ctx, BS_EINVAL, "bs_scatter: NULL vector");
    if (bs_overlap(qL, 8 * t->NL, qG, 8 * t->NG))
        return bs_set_error(ctx, BS_EINVAL, "bs_scatter: qL and qG overlap");
    if ((reinterpret_cast<uintptr_t>(qL) | reinterpret_cast<uintptr_t>(qG)) & 7u)
        return bs_set_error(ctx, BS_EINVAL, "bs_scatter: vectors must be 8-byte aligned");
    if (int st = bs_check_device(ctx))
        return st;
    if (t->NL == 0)
        return BS_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (t->plan && !(ctx->tune.small_onepass && 8 * t->NG <= kOnePassScatterBytes))
        return bs_scatter_planned(ctx, t, qG, qL, s);
    const bool vec = (reinterpret_cast<uintptr_t>(t->scatterIds) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(qL) & 31u) == 0;
    const int64_t cap = static_cast<int64_t>(ctx->sms) * ctx->tune.scatter_blocks_per_sm;
    if (vec) {
        const int64_t ngroups = t->NL / 4;
        int64_t need = (ngroups / kScatterUnroll + kThreads) / kThreads;
        const int grid = static_cast<int>(need < cap ? (need < 1 ? 1 : need) : cap);
        scatter4_kernel<kScatterUnroll><<<grid, kThreads, 0, s>>>(t->scatterIds, qG, qL, ngroups,
                                                                  t->NL, t->NG, ctx->dev_err);
    } else {
        const int64_t need = (t->NL + kThreads - 1) / kThreads;
        const int grid = static_cast<int>(need < cap ? need : cap);
        scatter1_kernel<<<grid, kThreads, 0, s>>>(t->scatterIds, qG, qL, t->NL, t->NG,
                                                  ctx->dev_err);
    }
    BS_LAUNCH_CHECK(ctx, "scatter_kernel");
    return BS_OK;
}

extern "C" int bs_cg_iteration(bs_ctx *ctx, const bs_gs_dev *t, const double *pG, double *pL,
                               double *ApG, double *xG, double *rG, const double *rr_dev,
                               double *pAp_dev, double *rr_new_dev, double *rnorm_dev,
                               void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (int st = check_tables(ctx, "bs_cg_iteration", t, true))
        return st;
    if (!rr_dev || !pAp_dev || !rr_new_dev || !rnorm_dev)
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_iteration: NULL scalar pointer");
    if (bs_overlap(pG, 8 * t->NG, ApG, 8 * t->NG))
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_iteration: pG and ApG overlap");
    const int64_t n = t->NG;
    int st;
    if ((st = bs_scatter(ctx, t, pG, pL, stream)))
        return st;
    if ((st = bs_gather(ctx, t, pL, ApG, stream)))
        return st;
    if ((st = bs_dot(ctx, n, pG, ApG, pAp_dev, stream)))
        return st;
    if ((st = bs_cg_update(ctx, n, rr_dev, pAp_dev, 0.0, pG, ApG, xG, rG, rr_new_dev, stream)))
        return st;
    return bs_norm(ctx, n, rG, rnorm_dev, stream);
}

extern "C" int bs_cg_solve(bs_ctx *ctx, const bs_gs_dev *t, const double *dL, const double *bG,
                           double *xG, double *rG, double *pG, double *ApG, int32_t iters,
                           double *scal_dev, void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (!t || iters < 0 || !scal_dev)
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve: NULL tables/scalars or iters < 0");
    const int64_t n = t->NG;
    if (n > 0 && (!bG || !xG || !rG || !pG || !ApG))
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve: NULL vector");
    const double *vin[2] = {bG, xG};
    double *vout[3] = {rG, pG, ApG};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 2; ++j)
            if (bs_overlap(vout[i], 8 * n, vin[j], 8 * n))
                return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve: work vectors overlap b or x");
        for (int j = i + 1; j < 3; ++j)
            if (bs_overlap(vout[i], 8 * n, vout[j], 8 * n))
                return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve: r, p and Ap overlap");
        if (bs_overlap(vout[i], 8 * n, scal_dev, 8 * (2ll * iters + 1)))
            return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve: scalars overlap a vector");
    }
    if (bs_overlap(bG, 8 * n, xG, 8 * n))
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve: b and x overlap");
    double *rr = scal_dev, *pAp = scal_dev + iters + 1;
    int st;
    // r = b - A x; p = r; rr_0 = r.r
    if ((st = bs_apply_diag(ctx, t, xG, dL, ApG, stream)) ||
        (st = bs_copy(ctx, n, bG, rG, stream)) ||
        (st = bs_axpy(ctx, n, -1.0, ApG, 1.0, rG, stream)) ||
        (st = bs_copy(ctx, n, rG, pG, stream)) || (st = bs_norm(ctx, n, rG, rr, stream)))
        return st;
    for (int32_t k = 0; k < iters; ++k) {
        // Ap = A p; alpha = rr_k / p.Ap; x += alpha p, r -= alpha Ap, rr_k+1 = r.r;
        // p = r + (rr_k+1 / rr_k) p
        if ((st = bs_apply_diag(ctx, t, pG, dL, ApG, stream)) ||
            (st = bs_dot(ctx, n, pG, ApG, pAp + k, stream)) ||
            (st = bs_cg_update(ctx, n, rr + k, pAp + k, 0.0, pG, ApG, xG, rG, rr + k + 1,
                               stream)) ||
            (st = bs_axpy_dev(ctx, n, 1.0, rG, rr + k + 1, rr + k, pG, stream)))
            return st;
    }
    return BS_OK;
}

extern "C" int bs_apply_diag(bs_ctx *ctx, const bs_gs_dev *t, const double *xG, const double *dL,
                             double *yG, void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (int st = check_tables(ctx, "bs_apply_diag", t, true))
        return st;
    if (!t->plan)
        return bs_set_error(ctx, BS_EINVAL, "bs_apply_diag: needs a two-pass plan");
    if (t->NG > 0 && (!xG || !yG))
        return bs_set_error(ctx, BS_EINVAL, "bs_apply_diag: NULL vector");
    if (bs_overlap(xG, 8 * t->NG, yG, 8 * t->NG) ||
        (dL && bs_overlap(dL, 8 * t->NL, yG, 8 * t->NG)))
        return bs_set_error(ctx, BS_EINVAL, "bs_apply_diag: yG overlaps xG or dL");
    if ((reinterpret_cast<uintptr_t>(xG) | reinterpret_cast<uintptr_t>(dL) |
         reinterpret_cast<uintptr_t>(yG)) & 7u)
        return bs_set_error(ctx, BS_EINVAL, "bs_apply_diag: vectors must be 8-byte aligned");
    if (int st = bs_check_device(ctx))
        return st;
    if (t->NG == 0)
        return BS_OK;
    return bs_apply_diag_planned(ctx, t, xG, dL, yG, static_cast<cudaStream_t>(stream));
}
