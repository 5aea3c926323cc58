// bs_gs2.cu -- two-pass tiled BS6 gather and BS7 scatter.
//
// Same results as the one-pass kernels of bs_gs.cu ("Portable high-order
// finite element kernels I: Streaming Operations", BS6/BS7; eq. (3)), bit
// for bit, with a different data movement.  On GB300 a scattered 8-byte
// access costs one SM-to-L2 request whether it hits L2 or not, and the
// memory system serves about 5e10 such requests per second -- a random
// gather or scatter of N_L values cannot beat N_L / 5e10 seconds.  The plan
// (bs_plan.cpp) instead routes every value through shared memory twice:
//
//   scatter pass 1 (per tile of global rows): stage the tile's q_G values in
//     shared memory, then write the work array in contiguous runs, one run
//     per bucket of locals;
//   scatter pass 2 (per bucket of locals): place the bucket's runs by local
//     offset in shared memory (pre-zeroed: masked locals stay +0.0) and
//     write q_L coalesced;
//   gather pass 1 (per tile of locals): stage q_L, write runs per bucket of
//     rows;
//   gather pass 2 (per bucket of rows): place values by CSR position, then
//     sum each row in ascending local order from +0.0 and write q_G
//     coalesced.
//
// Global traffic is about twice the algorithmic bytes, all of it in runs.
// One 1024-thread block per SM, up to 227 KB of dynamic shared memory.
// Every table-derived index is checked; a bad one is skipped and raises the
// context's device error flag.
#include <cuda_runtime.h>

#include "bs_internal.h"

namespace {

constexpr int kT = 1024;  // threads per block
constexpr int kU = 8;     // independent loads per thread per step

struct PlanArgs {
    int64_t NL, NG, nnz;
    int32_t s_ntiles, s_nbuckets, s_tile_rows, s_bucket_len;
    int32_t g_ntiles, g_nbuckets, g_tile_len, g_bucket_entries_max, g_bucket_rows_max;
    const int32_t *rowStarts;
    const int32_t *s_tileRows, *s_runStart;
    const uint16_t *s_src, *s_dst;
    const int32_t *g_bucketRows, *g_tileSlot, *g_runStart;
    const uint16_t *g_src, *g_pos;
    double *work;
    int *err;
};

__device__ __forceinline__ uint16_t ld_u16(const uint16_t *p)
{
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ double ld_seq(const double *p)
{
    double v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.f64 %0, [%1];" : "=d"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void flag(int *err)
{
    atomicOr(err, BS_DEVERR_BOUNDS);
}

// Copies n consecutive doubles from global memory into shared memory, kU
// loads in flight per thread.
__device__ __forceinline__ void stage(double *dst, const double *src, int n)
{
    for (int i0 = threadIdx.x; i0 < n; i0 += kU * kT) {
        double v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
            v[u] = i0 + u * kT < n ? ld_seq(src + i0 + u * kT) : 0.0;
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (i0 + u * kT < n)
                dst[i0 + u * kT] = v[u];
    }
}

// In-place exclusive scan of a[0..n); a[n] receives the total.  All
// threads of the block call it; it ends with a barrier.
__device__ void block_exclusive_scan(int32_t *a, int n)
{
    __shared__ int32_t warp_tot[kT / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (n + kT - 1) / kT;
    const int i0 = threadIdx.x * per;
    int32_t local = 0;
    for (int k = 0; k < per; ++k)
        if (i0 + k < n)
            local += a[i0 + k];
    int32_t v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += y;
    }
    if (lane == 31)
        warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int32_t w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    int32_t prefix = (v - local) + (warp > 0 ? warp_tot[warp - 1] : 0);
    for (int k = 0; k < per; ++k)
        if (i0 + k < n) {
            const int32_t x = a[i0 + k];
            a[i0 + k] = prefix;
            prefix += x;
        }
    if (threadIdx.x == 0)
        a[n] = warp_tot[kT / 32 - 1];
    __syncthreads();
}

// (+0.0 + v[0]) + v[1] + ... + v[n-1], n >= 1, in that order.  A sum
// started from +0.0 is never -0.0 and otherwise equals the same sum started
// from v[0], so the first addition is replaced by mapping -0.0 to +0.0
// with integer operations (binary64 adds are scarce on this GPU).
__device__ __forceinline__ double row_sum(const double *v, int n)
{
    double s = v[0];
    for (int j = 1; j < n; ++j)
        s += v[j];
    const long long b = __double_as_longlong(s);
    return (b << 1) == 0 ? 0.0 : s;
}

// Largest c in [0, n) with off[c] <= k, for 0 <= k < off[n].
__device__ __forceinline__ int find_run(const int32_t *off, int n, int32_t k)
{
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= k)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Loads the (tile, bucket) run table row of tile `t` into shared memory:
// runPos[b] = work position of run (t, b), runOff = exclusive scan of the
// run lengths (runOff[nb] = total).  Returns false (uniformly) on a bad
// table; the caller flags and leaves.
__device__ bool load_runs(const int32_t *runStart, int t, int nb, int64_t nnz, int32_t *runPos,
                          int32_t *runOff)
{
    __shared__ int bad_runs;
    if (threadIdx.x == 0)
        bad_runs = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += kT) {
        const int32_t p0 = runStart[static_cast<int64_t>(t) * nb + b];
        const int32_t p1 = runStart[static_cast<int64_t>(t + 1) * nb + b];
        const bool ok = p0 >= 0 && p1 >= p0 && p1 <= nnz;
        runPos[b] = ok ? p0 : 0;
        runOff[b] = ok ? p1 - p0 : 0;
        if (!ok)
            bad_runs = 1;
    }
    __syncthreads();
    block_exclusive_scan(runOff, nb);
    return bad_runs == 0;
}

// Writes the tile's slots [0, total) to the work array run by run: slot k
// of run c goes to work[runPos[c] + k - runOff[c]], its value taken from
// the staged tile at offset src[base + k].  Each warp takes chunks of
// 32 kU consecutive slots (lane i: slots i, i+32, ...), so the src loads
// and the work stores of a warp instruction are contiguous; a lane finds
// its run by one binary search per chunk and then walks forward.
__device__ __forceinline__ bool emit_runs(const int32_t *runPos, const int32_t *runOff, int nb,
                                          int32_t total, const uint16_t *src, int64_t base,
                                          const double *vals, int nvals, double *work)
{
    constexpr int kChunk = 32 * kU;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    bool bad = false;
    for (int32_t c0 = warp * kChunk; c0 < total; c0 += (kT / 32) * kChunk) {
        uint16_t o[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t k = c0 + lane + 32 * u;
            o[u] = k < total ? ld_u16(src + base + k) : 0;
        }
        int c = find_run(runOff, nb, c0 + lane < total ? c0 + lane : total - 1);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t k = c0 + lane + 32 * u;
            if (k < total) {
                while (c + 1 < nb && runOff[c + 1] <= k)
                    ++c;
                double v = 0.0;
                if (o[u] < nvals)
                    v = vals[o[u]];
                else
                    bad = true;
                work[runPos[c] + (k - runOff[c])] = v;
            }
        }
    }
    return bad;
}

// --------------------------------------------------------------- scatter
__global__ void __launch_bounds__(kT, 1) scatter_tile_kernel(PlanArgs a, const double *__restrict__ qG)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *vals = reinterpret_cast<double *>(smem);
    int32_t *runPos = reinterpret_cast<int32_t *>(vals + a.s_tile_rows);
    int32_t *runOff = runPos + a.s_nbuckets;
    const int t = blockIdx.x;
    const int32_t r0 = a.s_tileRows[t], r1 = a.s_tileRows[t + 1];
    const int32_t nrows = r1 - r0;
    if (r0 < 0 || nrows < 0 || nrows > a.s_tile_rows || r1 > a.NG) {
        if (threadIdx.x == 0)
            flag(a.err);
        return;
    }
    const int32_t e0 = a.rowStarts[r0], e1 = a.rowStarts[r1];
    if (e0 < 0 || e1 < e0 || e1 > a.nnz) {
        if (threadIdx.x == 0)
            flag(a.err);
        return;
    }
    stage(vals, qG + r0, nrows);
    if (!load_runs(a.s_runStart, t, a.s_nbuckets, a.nnz, runPos, runOff) ||
        runOff[a.s_nbuckets] != e1 - e0) {
        if (threadIdx.x == 0)
            flag(a.err);
        return;
    }
    if (emit_runs(runPos, runOff, a.s_nbuckets, e1 - e0, a.s_src, e0, vals, nrows, a.work))
        flag(a.err);
}

__global__ void __launch_bounds__(kT, 1) scatter_bucket_kernel(PlanArgs a, double *__restrict__ qL)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *out = reinterpret_cast<double *>(smem);
    const int b = blockIdx.x;
    const int64_t l0 = static_cast<int64_t>(b) * a.s_bucket_len;
    const int32_t len = static_cast<int32_t>(
        a.NL - l0 < a.s_bucket_len ? a.NL - l0 : a.s_bucket_len);
    const int32_t j0 = a.s_runStart[b];
    const int32_t j1 = a.s_runStart[static_cast<int64_t>(a.s_ntiles) * a.s_nbuckets + b];
    if (len <= 0 || j0 < 0 || j1 < j0 || j1 > a.nnz || j1 - j0 > len) {
        if (threadIdx.x == 0)
            flag(a.err);
        return;
    }
    for (int32_t i = threadIdx.x; i < len; i += kT)
        out[i] = 0.0;
    __syncthreads();
    bool bad = false;
    for (int32_t j = j0 + threadIdx.x; j < j1; j += kU * kT) {
        uint16_t d[kU];
        double v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t jj = j + u * kT;
            d[u] = jj < j1 ? ld_u16(a.s_dst + jj) : 0;
            v[u] = jj < j1 ? ld_seq(a.work + jj) : 0.0;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (j + u * kT < j1) {
                if (d[u] < len)
                    out[d[u]] = v[u];
                else
                    bad = true;
            }
    }
    __syncthreads();
    for (int32_t i = threadIdx.x; i < len; i += kT)
        qL[l0 + i] = out[i];
    if (bad)
        flag(a.err);
}

// ---------------------------------------------------------------- gather
__global__ void __launch_bounds__(kT, 1) gather_tile_kernel(PlanArgs a, const double *__restrict__ qL)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *vals = reinterpret_cast<double *>(smem);
    int32_t *runPos = reinterpret_cast<int32_t *>(vals + a.g_tile_len);
    int32_t *runOff = runPos + a.g_nbuckets;
    const int u = blockIdx.x;
    const int64_t l0 = static_cast<int64_t>(u) * a.g_tile_len;
    const int32_t len = static_cast<int32_t>(a.NL - l0 < a.g_tile_len ? a.NL - l0 : a.g_tile_len);
    const int32_t s0 = a.g_tileSlot[u], s1 = a.g_tileSlot[u + 1];
    if (len <= 0 || s0 < 0 || s1 < s0 || s1 > a.nnz || s1 - s0 > len) {
        if (threadIdx.x == 0)
            flag(a.err);
        return;
    }
    stage(vals, qL + l0, len);
    if (!load_runs(a.g_runStart, u, a.g_nbuckets, a.nnz, runPos, runOff) ||
        runOff[a.g_nbuckets] != s1 - s0) {
        if (threadIdx.x == 0)
            flag(a.err);
        return;
    }
    if (emit_runs(runPos, runOff, a.g_nbuckets, s1 - s0, a.g_src, s0, vals, len, a.work))
        flag(a.err);
}

__global__ void __launch_bounds__(kT, 1) gather_bucket_kernel(PlanArgs a, double *__restrict__ qG)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *vals = reinterpret_cast<double *>(smem);
    uint16_t *rs = reinterpret_cast<uint16_t *>(vals + a.g_bucket_entries_max);
    const int c = blockIdx.x;
    const int32_t r0 = a.g_bucketRows[c], r1 = a.g_bucketRows[c + 1];
    const int32_t nrows = r1 - r0;
    if (r0 < 0 || nrows < 0 || nrows > a.g_bucket_rows_max || r1 > a.NG) {
        if (threadIdx.x == 0)
            flag(a.err);
        return;
    }
    const int32_t e0 = a.rowStarts[r0], e1 = a.rowStarts[r1];
    const int32_t ne = e1 - e0;
    const int32_t j0 = a.g_runStart[c];
    const int32_t j1 = a.g_runStart[static_cast<int64_t>(a.g_ntiles) * a.g_nbuckets + c];
    if (e0 < 0 || ne < 0 || e1 > a.nnz || ne > a.g_bucket_entries_max || j0 != e0 || j1 != e1) {
        if (threadIdx.x == 0)
            flag(a.err);
        return;
    }
    bool bad = false;
    for (int32_t j = threadIdx.x; j < ne; j += kU * kT) {
        uint16_t p[kU];
        double v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t jj = j + u * kT;
            p[u] = jj < ne ? ld_u16(a.g_pos + e0 + jj) : 0;
            v[u] = jj < ne ? ld_seq(a.work + e0 + jj) : 0.0;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (j + u * kT < ne) {
                if (p[u] < ne)
                    vals[p[u]] = v[u];
                else
                    bad = true;
            }
    }
    for (int32_t k0 = threadIdx.x; k0 <= nrows; k0 += kU * kT) {
        int32_t o[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
            o[u] = k0 + u * kT <= nrows ? a.rowStarts[r0 + k0 + u * kT] - e0 : 0;
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (k0 + u * kT <= nrows) {
                if (o[u] < 0 || o[u] > ne)
                    bad = true;
                rs[k0 + u * kT] = static_cast<uint16_t>(o[u] < 0 ? 0 : (o[u] > ne ? ne : o[u]));
            }
    }
    __syncthreads();
    for (int32_t k = threadIdx.x; k < nrows; k += kT) {
        const int32_t lo = rs[k], hi = rs[k + 1];
        if (hi < lo)
            bad = true;
        qG[r0 + k] = hi > lo ? row_sum(vals + lo, hi - lo) : 0.0;
    }
    if (bad)
        flag(a.err);
}

int64_t smem_s1(const bs_plan_dev *p) { return 8ll * p->s_tile_rows + 4ll * p->s_nbuckets + 4ll * (p->s_nbuckets + 1); }
int64_t smem_s2(const bs_plan_dev *p) { return 8ll * p->s_bucket_len; }
int64_t smem_g1(const bs_plan_dev *p) { return 8ll * p->g_tile_len + 4ll * p->g_nbuckets + 4ll * (p->g_nbuckets + 1); }
int64_t smem_g2(const bs_plan_dev *p) { return 8ll * p->g_bucket_entries_max + 2ll * (p->g_bucket_rows_max + 1); }

constexpr int64_t kSmemMax = 232448;

template <class K>
int set_smem(bs_ctx *ctx, K kernel, int64_t bytes)
{
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (e != cudaSuccess)
        return bs_set_error(ctx, BS_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return BS_OK;
}

int check_plan(bs_ctx *ctx, const char *name, const bs_gs_dev *t, const void *qL, const void *qG)
{
    const bs_plan_dev *p = t->plan;
    if (!t->rowStarts)
        return bs_set_error(ctx, BS_EINVAL, "%s: the plan needs rowStarts", name);
    if (p->s_ntiles < 1 || p->s_nbuckets < 1 || p->s_tile_rows < 1 || p->s_bucket_len < 1 ||
        p->g_ntiles < 1 || p->g_nbuckets < 1 || p->g_tile_len < 1 || p->g_bucket_entries_max < 1 ||
        p->g_bucket_rows_max < 1)
        return bs_set_error(ctx, BS_EINVAL, "%s: bad plan sizes", name);
    if (static_cast<int64_t>(p->s_nbuckets) * p->s_bucket_len < t->NL ||
        static_cast<int64_t>(p->g_ntiles) * p->g_tile_len < t->NL)
        return bs_set_error(ctx, BS_EINVAL, "%s: plan does not cover the mesh", name);
    if (smem_s1(p) > kSmemMax || smem_s2(p) > kSmemMax || smem_g1(p) > kSmemMax ||
        smem_g2(p) > kSmemMax)
        return bs_set_error(ctx, BS_EINVAL, "%s: plan needs too much shared memory", name);
    if (!p->s_tileRows || !p->s_runStart || !p->g_bucketRows || !p->g_tileSlot ||
        !p->g_runStart || !p->work || (t->nnz > 0 && (!p->s_src || !p->s_dst || !p->g_src || !p->g_pos)))
        return bs_set_error(ctx, BS_EINVAL, "%s: NULL plan table", name);
    if (p->work_len < t->nnz)
        return bs_set_error(ctx, BS_EINVAL, "%s: work buffer shorter than nnz", name);
    if (bs_overlap(p->work, 8 * p->work_len, qL, 8 * t->NL) ||
        bs_overlap(p->work, 8 * p->work_len, qG, 8 * t->NG))
        return bs_set_error(ctx, BS_EINVAL, "%s: work buffer overlaps qL or qG", name);
    if (reinterpret_cast<uintptr_t>(p->work) & 7u)
        return bs_set_error(ctx, BS_EINVAL, "%s: work buffer must be 8-byte aligned", name);
    return BS_OK;
}

PlanArgs make_args(const bs_ctx *ctx, const bs_gs_dev *t)
{
    const bs_plan_dev *p = t->plan;
    PlanArgs a;
    a.NL = t->NL;
    a.NG = t->NG;
    a.nnz = t->nnz;
    a.s_ntiles = p->s_ntiles;
    a.s_nbuckets = p->s_nbuckets;
    a.s_tile_rows = p->s_tile_rows;
    a.s_bucket_len = p->s_bucket_len;
    a.g_ntiles = p->g_ntiles;
    a.g_nbuckets = p->g_nbuckets;
    a.g_tile_len = p->g_tile_len;
    a.g_bucket_entries_max = p->g_bucket_entries_max;
    a.g_bucket_rows_max = p->g_bucket_rows_max;
    a.rowStarts = t->rowStarts;
    a.s_tileRows = p->s_tileRows;
    a.s_runStart = p->s_runStart;
    a.s_src = p->s_src;
    a.s_dst = p->s_dst;
    a.g_bucketRows = p->g_bucketRows;
    a.g_tileSlot = p->g_tileSlot;
    a.g_runStart = p->g_runStart;
    a.g_src = p->g_src;
    a.g_pos = p->g_pos;
    a.work = p->work;
    a.err = ctx->dev_err;
    return a;
}

} // namespace

int bs_scatter_planned(bs_ctx *ctx, const bs_gs_dev *t, const double *qG, double *qL,
                       cudaStream_t s)
{
    if (int st = check_plan(ctx, "bs_scatter", t, qL, qG))
        return st;
    const bs_plan_dev *p = t->plan;
    const PlanArgs a = make_args(ctx, t);
    if (int st = set_smem(ctx, scatter_tile_kernel, smem_s1(p)))
        return st;
    if (int st = set_smem(ctx, scatter_bucket_kernel, smem_s2(p)))
        return st;
    scatter_tile_kernel<<<p->s_ntiles, kT, smem_s1(p), s>>>(a, qG);
    BS_LAUNCH_CHECK(ctx, "scatter_tile_kernel");
    scatter_bucket_kernel<<<p->s_nbuckets, kT, smem_s2(p), s>>>(a, qL);
    BS_LAUNCH_CHECK(ctx, "scatter_bucket_kernel");
    return BS_OK;
}

int bs_gather_planned(bs_ctx *ctx, const bs_gs_dev *t, const double *qL, double *qG,
                      cudaStream_t s)
{
    if (int st = check_plan(ctx, "bs_gather", t, qL, qG))
        return st;
    const bs_plan_dev *p = t->plan;
    const PlanArgs a = make_args(ctx, t);
    if (int st = set_smem(ctx, gather_tile_kernel, smem_g1(p)))
        return st;
    if (int st = set_smem(ctx, gather_bucket_kernel, smem_g2(p)))
        return st;
    gather_tile_kernel<<<p->g_ntiles, kT, smem_g1(p), s>>>(a, qL);
    BS_LAUNCH_CHECK(ctx, "gather_tile_kernel");
    gather_bucket_kernel<<<p->g_nbuckets, kT, smem_g2(p), s>>>(a, qG);
    BS_LAUNCH_CHECK(ctx, "gather_bucket_kernel");
    return BS_OK;
}
