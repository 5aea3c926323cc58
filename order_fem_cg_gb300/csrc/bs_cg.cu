// bs_cg.cu -- the CG solve of bs_cg_solve in one cooperative kernel.
//
// For sizes where launches, not bytes, set the time ("Portable high-order
// finite element kernels I", eqs. (8)-(10): T0 dominates below the
// Fischer-Brown point), the whole iteration runs inside one kernel whose
// blocks are all resident (cooperative launch) and meet at grid barriers:
//
//   Ap = Z^T diag(d) Z p    scatter with the local operator into q_L, then
//                           the CSR gather, with p.Ap summed in the same pass
//   x += alpha p, r -= alpha Ap, r.r     (BS5)
//   p = r + beta p                        (BS2)
//
// four barriers per iteration.  The gather/scatter phases are the one-pass
// forms (random 8-byte accesses): right for meshes that fit L2, not for the
// bench-scale meshes (use bs_cg_solve there).
//
// The barrier is this file's own: an arrival counter and a generation word
// in the context's scratch, polled with a bounded count; a block that gives
// up raises the abort word (so every other block gives up at its next poll)
// and the context's timeout flag, and the kernel ends.
#include <cuda_runtime.h>

#include "bs_internal.h"

namespace {

constexpr int kCT = 256;                      // threads per block
constexpr long long kMaxPolls = 1ll << 22;    // per barrier wait (x >= 32 ns sleep)

// Barrier words: arrival count, generation, abort, each on its own 64-byte
// line of the context's 256-byte counter block (word 0 is the reductions'
// completion counter); zeroed on the stream before every launch.
struct Bar {
    unsigned int *count, *gen, *abort;
};

struct CgArgs {
    int64_t NL, NG, nnz;
    const int32_t *ids, *rowStarts, *localIds;
    const double *dL, *b;
    double *x, *r, *p, *Ap, *qL, *scal;
    double mzero;  // -0 (for mul_rn)
    int32_t iters;
    double *part_a, *part_b;  // per-block partials of p.Ap and of r.r
    Bar bar;
    int *err;
};

__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_down_sync(0xffffffffu, v, o);
    return v;
}

// Sum over the block; the result is valid in thread 0.
__device__ double block_sum(double v, double *sh)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();  // sh may still be read from a previous call
    if (lane == 0)
        sh[w] = v;
    __syncthreads();
    if (w == 0) {
        v = lane < kCT / 32 ? sh[lane] : 0.0;
        v = warp_sum(v);
    }
    return v;
}

// All blocks arrive, then all leave; false (in every thread of the block)
// if the wait gave up.  Writes before the barrier are visible after it.
__device__ bool grid_sync(const Bar &b, int *err)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        volatile unsigned int *gen = b.gen;
        volatile unsigned int *abort = b.abort;
        const unsigned int g = *gen;
        __threadfence();
        if (atomicAdd(b.count, 1u) == gridDim.x - 1) {
            *b.count = 0u;
            __threadfence();
            atomicAdd(b.gen, 1u);
        } else {
            long long polls = 0;
            while (*gen == g) {
                if (*abort || ++polls > kMaxPolls) {
                    ok = 0;
                    atomicExch(b.abort, 1u);
                    atomicOr(err, BS_DEVERR_TIMEOUT);
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// sum of part[0 .. gridDim.x) in a fixed order: every block gets the same
// value (valid in every thread).
__device__ double grid_total(const double *part, double *sh)
{
    __shared__ double s_tot;
    double v = 0.0;
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += kCT)
        v += __ldcg(part + i);
    v = block_sum(v, sh);
    if (threadIdx.x == 0)
        s_tot = v;
    __syncthreads();
    return s_tot;
}

__device__ __forceinline__ double quotient(double num, double den)
{
    return den != 0.0 ? __ddiv_rn(num, den) : 0.0;
}

__device__ __forceinline__ void flag(int *err)
{
    atomicOr(err, BS_DEVERR_BOUNDS);
}

// q_L[l] = d[l] * v[ids[l]] (or v[ids[l]]) for every unmasked local.
__device__ void scatter_scaled(const CgArgs &a, const double *v)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kCT;
    bool bad = false;
    for (int64_t l = blockIdx.x * static_cast<int64_t>(kCT) + threadIdx.x; l < a.NL; l += stride) {
        const int32_t g = a.ids[l];
        if (g < 0)
            continue;
        if (g >= a.NG) {
            bad = true;
            continue;
        }
        a.qL[l] = a.dL ? mul_rn(a.dL[l], v[g], a.mzero) : v[g];
    }
    if (bad)
        flag(a.err);
}

// y[g] = (+0.0 + q_L[l1]) + q_L[l2] + ... (ascending l) for every row;
// returns this thread's sum of w[g] y[g] (if w) for the p.Ap reduction.
__device__ double gather_rows(const CgArgs &a, double *y, const double *w)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kCT;
    double acc = 0.0;
    bool bad = false;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(kCT) + threadIdx.x; g < a.NG; g += stride) {
        const int32_t e0 = a.rowStarts[g], e1 = a.rowStarts[g + 1];
        double s = 0.0;
        if (e0 < 0 || e1 < e0 || e1 > a.nnz) {
            bad = true;
        } else {
            for (int32_t e = e0; e < e1; ++e) {
                const int32_t l = a.localIds[e];
                if (l < 0 || l >= a.NL)
                    bad = true;
                else
                    s += a.qL[l];
            }
        }
        y[g] = s;
        if (w)
            acc = __fma_rn(w[g], s, acc);
    }
    if (bad)
        flag(a.err);
    return acc;
}

__global__ void __launch_bounds__(kCT) cg_fused_kernel(CgArgs a)
{
    __shared__ double sh[kCT / 32];
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kCT;
    const int64_t t0 = blockIdx.x * static_cast<int64_t>(kCT) + threadIdx.x;

    // r = b - A x; p = r; rr_0 = r.r
    scatter_scaled(a, a.x);
    if (!grid_sync(a.bar, a.err))
        return;
    gather_rows(a, a.Ap, nullptr);
    if (!grid_sync(a.bar, a.err))
        return;
    double acc = 0.0;
    for (int64_t i = t0; i < a.NG; i += stride) {
        const double ri = __fma_rn(-1.0, a.Ap[i], a.b[i]);
        a.r[i] = ri;
        a.p[i] = ri;
        acc = __fma_rn(ri, ri, acc);
    }
    acc = block_sum(acc, sh);
    if (threadIdx.x == 0)
        a.part_b[blockIdx.x] = acc;
    if (!grid_sync(a.bar, a.err))
        return;
    double rr = grid_total(a.part_b, sh);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        a.scal[0] = rr;

    for (int32_t k = 0; k < a.iters; ++k) {
        // Ap = A p, with p.Ap
        scatter_scaled(a, a.p);
        if (!grid_sync(a.bar, a.err))
            return;
        acc = block_sum(gather_rows(a, a.Ap, a.p), sh);
        if (threadIdx.x == 0)
            a.part_a[blockIdx.x] = acc;
        if (!grid_sync(a.bar, a.err))
            return;
        const double pAp = grid_total(a.part_a, sh);
        const double alpha = quotient(rr, pAp), nalpha = -alpha;
        // BS5: x += alpha p, r -= alpha Ap, r.r over the updated r
        acc = 0.0;
        for (int64_t i = t0; i < a.NG; i += stride) {
            a.x[i] = __fma_rn(alpha, a.p[i], a.x[i]);
            const double ri = __fma_rn(nalpha, a.Ap[i], a.r[i]);
            a.r[i] = ri;
            acc = __fma_rn(ri, ri, acc);
        }
        acc = block_sum(acc, sh);
        if (threadIdx.x == 0)
            a.part_b[blockIdx.x] = acc;
        if (!grid_sync(a.bar, a.err))
            return;
        const double rr_new = grid_total(a.part_b, sh);
        const double beta = quotient(rr_new, rr);
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            a.scal[k + 1] = rr_new;
            a.scal[a.iters + 1 + k] = pAp;
        }
        // BS2: p = r + beta p
        for (int64_t i = t0; i < a.NG; i += stride)
            a.p[i] = __fma_rn(1.0, a.r[i], mul_rn(beta, a.p[i], a.mzero));
        rr = rr_new;
        if (!grid_sync(a.bar, a.err))
            return;
    }
}

// Two rounds of the grid barrier; block `absent` (if >= 0) leaves before
// the first, so that the other blocks' waits run out.
__global__ void __launch_bounds__(kCT) barrier_probe_kernel(Bar bar, int absent, int *err)
{
    if (static_cast<int>(blockIdx.x) == absent)
        return;
    if (!grid_sync(bar, err))
        return;
    grid_sync(bar, err);
}

int barrier_setup(bs_ctx *ctx, cudaStream_t s, Bar *bar)
{
    unsigned int *words = ctx->counter;
    BS_CUDA_TRY(ctx, cudaMemsetAsync(words + 16, 0, 3 * 64, s));
    bar->count = words + 16;
    bar->gen = words + 32;
    bar->abort = words + 48;
    return BS_OK;
}

} // namespace

extern "C" int bs_probe_grid_barrier(bs_ctx *ctx, int absent_block, void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (int st = bs_check_device(ctx))
        return st;
    const int grid = ctx->sms;
    if (absent_block >= grid)
        return bs_set_error(ctx, BS_EINVAL, "bs_probe_grid_barrier: no block %d", absent_block);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Bar bar;
    if (int st = barrier_setup(ctx, s, &bar))
        return st;
    int *err = ctx->dev_err;
    void *args[3] = {&bar, &absent_block, &err};
    BS_CUDA_TRY(ctx, cudaLaunchCooperativeKernel(reinterpret_cast<void *>(barrier_probe_kernel),
                                                 dim3(grid), dim3(kCT), args, 0, s));
    return BS_OK;
}

extern "C" int bs_cg_solve_fused(bs_ctx *ctx, const bs_gs_dev *t, const double *dL,
                                 const double *bG, double *xG, double *rG, double *pG,
                                 double *ApG, double *pL, int32_t iters, double *scal_dev,
                                 void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (!t || iters < 0 || !scal_dev)
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve_fused: NULL tables/scalars or iters < 0");
    const int64_t NG = t->NG, NL = t->NL;
    if (NG < 1 || NL < 1 || !t->scatterIds || !t->rowStarts || (t->nnz > 0 && !t->localIds))
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve_fused: bad tables");
    if (!bG || !xG || !rG || !pG || !ApG || !pL)
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve_fused: NULL vector");
    const void *ptr[7] = {bG, xG, rG, pG, ApG, pL, scal_dev};
    const int64_t len[7] = {8 * NG, 8 * NG, 8 * NG, 8 * NG, 8 * NG, 8 * NL, 8 * (2ll * iters + 1)};
    for (int i = 0; i < 7; ++i) {
        if (reinterpret_cast<uintptr_t>(ptr[i]) & 7u)
            return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve_fused: pointers must be 8-byte aligned");
        for (int j = i + 1; j < 7; ++j)
            if (bs_overlap(ptr[i], len[i], ptr[j], len[j]))
                return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve_fused: vectors overlap");
    }
    if (dL && (bs_overlap(dL, 8 * NL, rG, 8 * NG) || bs_overlap(dL, 8 * NL, pL, 8 * NL)))
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_solve_fused: dL overlaps a written vector");
    if (int st = bs_check_device(ctx))
        return st;

    int per_sm = 0;
    BS_CUDA_TRY(ctx, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cg_fused_kernel, kCT, 0));
    if (per_sm < 1)
        return bs_set_error(ctx, BS_ECUDA, "bs_cg_solve_fused: kernel cannot be resident");
    int grid = ctx->sms * (per_sm < 2 ? per_sm : 2);
    if (2 * grid > kMaxReduceBlocks)
        grid = kMaxReduceBlocks / 2;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CgArgs a;
    if (int st = barrier_setup(ctx, s, &a.bar))
        return st;
    a.NL = NL;
    a.NG = NG;
    a.nnz = t->nnz;
    a.ids = t->scatterIds;
    a.rowStarts = t->rowStarts;
    a.localIds = t->localIds;
    a.dL = dL;
    a.mzero = -0.0;
    a.b = bG;
    a.x = xG;
    a.r = rG;
    a.p = pG;
    a.Ap = ApG;
    a.qL = pL;
    a.scal = scal_dev;
    a.iters = iters;
    a.part_a = ctx->partials;
    a.part_b = ctx->partials + grid;
    a.err = ctx->dev_err;
    void *args[1] = {&a};
    BS_CUDA_TRY(ctx, cudaLaunchCooperativeKernel(reinterpret_cast<void *>(cg_fused_kernel),
                                                 dim3(grid), dim3(kCT), args, 0, s));
    return BS_OK;
}
