// bs_gs2.cu -- two-pass tiled BS6 gather and BS7 scatter.
//
// Same results as the one-pass kernels of bs_gs.cu ("Portable high-order
// finite element kernels I: Streaming Operations", BS6/BS7; eq. (3)), bit
// for bit, with a different data movement.  On GB300 a scattered 8-byte
// access into a vector larger than L2 pulls a whole sector from HBM, which
// serves about 5e10 of them per second -- a random gather or scatter of N_L
// values over such vectors cannot beat N_L / 5e10 seconds.  The plan
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
// Pass 1 writes runs of ~10-18 values, so a warp's 32 stores cost ~5 line
// requests instead of 2; these fragmented writes set its time, and runs grow
// only with tile x bucket, which one SM's shared memory caps.
// One 1024-thread block per SM, up to 227 KB of dynamic shared memory.
// Every table-derived index is checked; a bad one is skipped and raises the
// context's device error flag.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "bs_internal.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kT = 1024;  // threads per block
constexpr int kU = 8;     // independent loads per thread per step
constexpr int kMaxRow = 32;  // longest row of the grouped gather layout

struct PlanArgs {
    int64_t NL, NG, nnz;
    int32_t s_ntiles, s_nbuckets, s_tile_rows, s_bucket_len;
    int32_t g_ntiles, g_nbuckets, g_tile_len, g_bucket_entries_max, g_bucket_rows_max, g_mmax;
    const int32_t *rowStarts;
    const int32_t *s_tileRows, *s_runStart;
    const uint16_t *s_src, *s_dst;
    const int32_t *g_subRows, *g_tileSlot, *g_runStart;
    const uint16_t *g_src, *g_pos, *g_groupStart, *g_rowPos;
    double *work;
    int *err;
    int pf_next;  // persistent grids: prefetch a block's next tile/bucket into L2
    double mzero;  // -0 (for mul_rn)
    int pf_s2;     // scatter pass 2 prefetches its bucket's later entries into L2
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

// Two consecutive values (16-byte aligned) and two consecutive 16-bit
// entries (4-byte aligned), read once, not kept in L1.
__device__ __forceinline__ double2 ld_pair(const double *p)
{
    double2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.f64 {%0, %1}, [%2];"
                 : "=d"(v.x), "=d"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_u16x2(const uint16_t *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Four consecutive values (32-byte aligned) and four consecutive 16-bit
// entries (8-byte aligned), read once, not kept in L1.
struct Quad {
    double x, y, z, w;
};

__device__ __forceinline__ Quad ld_quad(const double *p)
{
    Quad v;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.f64 {%0, %1, %2, %3}, [%4];"
                 : "=d"(v.x), "=d"(v.y), "=d"(v.z), "=d"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_u16x4(const uint16_t *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_pair(double *p, double x, double y)
{
    asm volatile("st.global.v2.f64 [%0], {%1, %2};" ::"l"(p), "d"(x), "d"(y) : "memory");
}

__device__ __forceinline__ void flag(int *err)
{
    atomicOr(err, BS_DEVERR_BOUNDS);
}

// ------------------------------------------- bulk async copies (TMA engine)
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arms the barrier for `bytes` and copies [src, src + bytes) into shared
// memory at dst; 16-byte aligned addresses, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Waits for the completion of the barrier's phase of the given parity
// (0 for its first use, then alternating); gives up after a bounded number
// of polls (each poll may suspend the thread briefly) and reports false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    constexpr uint32_t kMaxPolls = 1u << 24;
    for (uint32_t i = 0; i < kMaxPolls; ++i) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(smem_u32(bar)), "r"(parity)
                     : "memory");
        if (done)
            return true;
    }
    return false;
}

// Waits for a bulk staging started by stage_start (barrier phase of the
// given parity): thread 0 polls the barrier (bounded) while the other
// threads wait at the block barrier, so the wait issues almost no
// instructions; a wait that ran out is followed by one more bounded wait
// for the copy still in flight.  Afterwards every thread tests the
// (completed) phase once, which is its own acquire of the copied data.
// Returns the outcome in every thread; after a failed wait the caller
// stops using the barrier (its phase is no longer known).
__device__ __forceinline__ bool stage_wait(bool bulk, uint64_t *bar, uint32_t parity)
{
    __shared__ int s_staged;
    if (threadIdx.x == 0) {
        int ok = 1;
        if (bulk && !mbar_wait(bar, parity)) {
            ok = 0;
            mbar_wait(bar, parity);
        }
        s_staged = ok;
    }
    __syncthreads();
    const bool staged = s_staged != 0;
    if (bulk && staged) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(smem_u32(bar)), "r"(parity)
                     : "memory");
        (void)done;
    }
    __syncthreads();  // s_staged is rewritten by the next wait
    return staged;
}

// Asks the bulk-copy engine to bring [p, p + bytes) into L2 (no data to the
// SM, no completion to wait for).  Only whole 16-byte units inside the
// range are requested, so nothing outside it is touched.
__device__ __forceinline__ void prefetch_l2(const void *p, int64_t bytes)
{
    uintptr_t a = reinterpret_cast<uintptr_t>(p), e = a + static_cast<uintptr_t>(bytes);
    a = (a + 15u) & ~static_cast<uintptr_t>(15);
    e &= ~static_cast<uintptr_t>(15);
    while (a < e) {
        const uint32_t n = static_cast<uint32_t>(e - a < 65536u ? e - a : 65536u);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(n) : "memory");
        a += n;
    }
}

// [lo, hi) clamped into [0, n]; false if empty.
__device__ __forceinline__ bool clamp_range(int64_t &lo, int64_t &hi, int64_t n)
{
    lo = lo < 0 ? 0 : (lo > n ? n : lo);
    hi = hi < lo ? lo : (hi > n ? n : hi);
    return hi > lo;
}

// Writes [src, src + bytes) of shared memory to global memory by the
// bulk-copy engine and waits only until the engine has read the source.
// The caller has made the shared-memory writes visible to the async proxy.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Stages n consecutive doubles into shared memory: by the bulk-copy engine
// when the source is 16-byte aligned and `use_bulk` (an odd last element
// by a thread), else by the threads.  `bar` must be initialised; every
// thread calls it and later calls stage_wait with the returned flag.
__device__ __forceinline__ bool stage_start(double *dst, const double *src, int n, uint64_t *bar,
                                            bool use_bulk = true)
{
    const bool bulk = use_bulk && n >= 2 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
    if (bulk) {
        if (threadIdx.x == 0)
            bulk_load(dst, src, static_cast<uint32_t>(n & ~1) * 8u, bar);
        if ((n & 1) && threadIdx.x == 1)
            dst[n - 1] = src[n - 1];
    }
    return bulk;
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

// Calls put(idx[j], val[j]) once for every j in [j0, j1), in no particular
// order, from all threads of the block.  Where val + j and idx + j can both
// be read two entries at a time (16-byte values, 4-byte index pairs), each
// thread has kP pairs in flight -- twice the entries of the one-at-a-time
// loop (kP = kU) for about the same registers, which is what a latency-
// bound placement needs; otherwise entries are read one at a time.  With
// kQuad, four at a time where both allow it (32-byte values, 8-byte index
// quads; kP/2 quads in flight): half the load instructions, which the
// scatter pass 2 and the fused operator (queue-throttled on global loads)
// gain from and the gather pass 2 (at its register limit) does not.
template <int kP, bool kQuad = false, class F>
__device__ __forceinline__ void stream_entries(const uint16_t *idx, const double *val, int32_t j0,
                                               int32_t j1, F &&put)
{
    if (j0 >= j1)
        return;
    const uintptr_t av = reinterpret_cast<uintptr_t>(val + j0);
    const uintptr_t ai = reinterpret_cast<uintptr_t>(idx + j0);
    const bool quad = kQuad && (av & 7u) == 0 && (ai & 1u) == 0 && ((av >> 3) & 3u) == ((ai >> 1) & 3u);
    const bool paired = (av & 7u) == 0 && (ai & 1u) == 0 && ((av >> 3) & 1u) == ((ai >> 1) & 1u);
    if (quad) {
        // up to three entries first, so that val + j is 32-byte aligned
        const int32_t h = min(static_cast<int32_t>((4u - ((av >> 3) & 3u)) & 3u), j1 - j0);
        if (static_cast<int32_t>(threadIdx.x) < h)
            put(ld_u16(idx + j0 + threadIdx.x), ld_seq(val + j0 + threadIdx.x));
        const int32_t j = j0 + h;
        const int32_t nq = (j1 - j) >> 2;
        const double *vp = val + j;
        const uint16_t *ip = idx + j;
        constexpr int kQ = (kP + 1) / 2;
        for (int32_t q = threadIdx.x; q < nq; q += kQ * kT) {
            Quad v[kQ];
            uint2 p[kQ];
#pragma unroll
            for (int i = 0; i < kQ; ++i) {
                const int32_t qq = q + i * kT;
                v[i] = qq < nq ? ld_quad(vp + 4 * qq) : Quad{0.0, 0.0, 0.0, 0.0};
                p[i] = qq < nq ? ld_u16x4(ip + 4 * qq) : make_uint2(0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < kQ; ++i)
                if (q + i * kT < nq) {
                    put(p[i].x & 0xffffu, v[i].x);
                    put(p[i].x >> 16, v[i].y);
                    put(p[i].y & 0xffffu, v[i].z);
                    put(p[i].y >> 16, v[i].w);
                }
        }
        // the last (j1 - j) mod 4 entries
        const int32_t t0 = j + 4 * nq;
        const int32_t lt = static_cast<int32_t>(threadIdx.x) - 32;
        if (lt >= 0 && lt < j1 - t0)
            put(ld_u16(idx + t0 + lt), ld_seq(val + t0 + lt));
    } else if (paired) {
        int32_t j = j0;
        if ((av >> 3) & 1u) {  // one entry first, so that val + j is 16-byte aligned
            if (threadIdx.x == 0)
                put(ld_u16(idx + j), ld_seq(val + j));
            ++j;
        }
        const int32_t np = (j1 - j) >> 1;
        const double *vp = val + j;
        const uint16_t *ip = idx + j;
        for (int32_t q = threadIdx.x; q < np; q += kP * kT) {
            double2 v[kP];
            uint32_t p[kP];
#pragma unroll
            for (int i = 0; i < kP; ++i) {
                const int32_t qq = q + i * kT;
                v[i] = qq < np ? ld_pair(vp + 2 * qq) : make_double2(0.0, 0.0);
                p[i] = qq < np ? ld_u16x2(ip + 2 * qq) : 0u;
            }
#pragma unroll
            for (int i = 0; i < kP; ++i)
                if (q + i * kT < np) {
                    put(p[i] & 0xffffu, v[i].x);
                    put(p[i] >> 16, v[i].y);
                }
        }
        if (((j1 - j) & 1) && threadIdx.x == 32)
            put(ld_u16(idx + j1 - 1), ld_seq(val + j1 - 1));
    } else {
        for (int32_t j = j0 + threadIdx.x; j < j1; j += kU * kT) {
            uint16_t d[kU];
            double v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int32_t jj = j + u * kT;
                d[u] = jj < j1 ? ld_u16(idx + jj) : 0;
                v[u] = jj < j1 ? ld_seq(val + jj) : 0.0;
            }
#pragma unroll
            for (int u = 0; u < kU; ++u)
                if (j + u * kT < j1)
                    put(d[u], v[u]);
        }
    }
}

// In-place exclusive scan of a[0..n); a[n] receives the total.  All
// threads of the block call it; it ends with a barrier.
template <class T>
__device__ void block_exclusive_scan(T *a, int n)
{
    __shared__ T warp_tot[kT / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (n + kT - 1) / kT;
    const int i0 = threadIdx.x * per;
    T local = 0;
    for (int k = 0; k < per; ++k)
        if (i0 + k < n)
            local += a[i0 + k];
    T v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += y;
    }
    if (lane == 31)
        warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        constexpr int kWarps = kT / 32;  // <= 32
        T w = lane < kWarps ? warp_tot[lane] : T(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const T y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        if (lane < kWarps)
            warp_tot[lane] = w;
    }
    __syncthreads();
    T prefix = (v - local) + (warp > 0 ? warp_tot[warp - 1] : T(0));
    for (int k = 0; k < per; ++k)
        if (i0 + k < n) {
            const T x = a[i0 + k];
            a[i0 + k] = prefix;
            prefix += x;
        }
    if (threadIdx.x == 0)
        a[n] = warp_tot[kT / 32 - 1];
    __syncthreads();
}

// v[0] + v[stride] + ... + v[(n-1) stride], n >= 1, in that order.  The
// row sum of the gather, (+0.0 + v[0]) + v[stride] + ..., is this value
// with -0.0 mapped to +0.0 (plus_zero): a sum started from +0.0 is never
// -0.0 and otherwise equals the same sum started from v[0], so the first
// binary64 addition (scarce on this GPU) is replaced by integer work.
__device__ __forceinline__ double row_sum(const double *v, int n, int stride)
{
    double s = v[0];
    for (int j = 1; j < n; ++j)
        s += v[j * stride];
    return s;
}

// In-place row sums of one row-length group: the R rows of length m sit
// column-major from `base` (entry j of row k at base + j R + k); the rows
// k = t0, t0 + nt, ... of this thread get their sum (in row_sum's order)
// in their first slot.  Four rows per step, so that four independent
// addition chains are in flight (a binary64 addition's latency is tens of
// cycles; one chain at a time leaves the FP64 pipe mostly idle).
__device__ __forceinline__ void group_sums(double *vals, int32_t base, int m, int32_t R, int t0,
                                           int nt)
{
    int32_t k = t0;
    for (; k + 3 * nt < R; k += 4 * nt) {
        double *v = vals + base + k;
        double s0 = v[0], s1 = v[nt], s2 = v[2 * nt], s3 = v[3 * nt];
        for (int j = 1; j < m; ++j) {
            const double *w = v + j * R;
            s0 += w[0];
            s1 += w[nt];
            s2 += w[2 * nt];
            s3 += w[3 * nt];
        }
        v[0] = s0;
        v[nt] = s1;
        v[2 * nt] = s2;
        v[3 * nt] = s3;
    }
    for (; k < R; k += nt)
        vals[base + k] = row_sum(vals + base + k, m, R);
}

__device__ __forceinline__ double plus_zero(double s)
{
    return (__double_as_longlong(s) << 1) == 0 ? 0.0 : s;
}

// A tile's run table in shared memory: runs[b] = (runOff[b] << 32) | ci[b]
// with runOff the exclusive scan of the run lengths and ci that of "run b
// is not empty" (runs[nb] holds both totals).
__device__ __forceinline__ int32_t run_off(int64_t r) { return static_cast<int32_t>(r >> 32); }
__device__ __forceinline__ int32_t run_ci(int64_t r) { return static_cast<int32_t>(r); }

// Largest b in [0, n) with runOff[b] <= k, for 0 <= k < runOff[n]: the
// (non-empty) run holding slot k.
__device__ __forceinline__ int find_run(const int64_t *runs, int n, int32_t k)
{
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (run_off(runs[mid]) <= k)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// The (tile, bucket) run table row of tile `t`, fetched into registers
// (issued before the tile staging so both are in flight together), then
// committed to shared memory as the packed scan `runs` (see run_off) and
// runD[i] = work position of the i-th non-empty run minus its runOff, so
// that slot k of that run goes to work[runD[i] + k].
constexpr int kRunRegs = 4;  // run-table entries per thread held in registers

struct RunFetch {
    int32_t p0[kRunRegs], p1[kRunRegs];
};

__device__ __forceinline__ RunFetch fetch_runs(const int32_t *runStart, int t, int nb)
{
    RunFetch f;
#pragma unroll
    for (int j = 0; j < kRunRegs; ++j) {
        const int b = threadIdx.x + j * kT;
        f.p0[j] = b < nb ? runStart[static_cast<int64_t>(t) * nb + b] : 0;
        f.p1[j] = b < nb ? runStart[static_cast<int64_t>(t + 1) * nb + b] : 0;
    }
    return f;
}

__device__ __forceinline__ bool run_ok(int32_t p0, int32_t p1, int64_t nnz)
{
    return p0 >= 0 && p1 >= p0 && p1 <= nnz;
}

// Returns false (uniformly) on a bad table; its runs are then all empty.
__device__ bool commit_runs(const RunFetch &f, const int32_t *runStart, int t, int nb,
                            int64_t nnz, int64_t *runs, int32_t *runD)
{
    __shared__ int bad_runs;
    if (threadIdx.x == 0)
        bad_runs = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRunRegs; ++j) {
        const int b = threadIdx.x + j * kT;
        if (b < nb) {
            const bool ok = run_ok(f.p0[j], f.p1[j], nnz);
            const int64_t len = ok ? f.p1[j] - f.p0[j] : 0;
            runs[b] = (len << 32) | (len > 0);
            if (!ok)
                bad_runs = 1;
        }
    }
    for (int b = threadIdx.x + kRunRegs * kT; b < nb; b += kT) {
        const int32_t p0 = runStart[static_cast<int64_t>(t) * nb + b];
        const int32_t p1 = runStart[static_cast<int64_t>(t + 1) * nb + b];
        const bool ok = run_ok(p0, p1, nnz);
        const int64_t len = ok ? p1 - p0 : 0;
        runs[b] = (len << 32) | (len > 0);
        if (!ok)
            bad_runs = 1;
    }
    __syncthreads();
    block_exclusive_scan(runs, nb);
#pragma unroll
    for (int j = 0; j < kRunRegs; ++j) {
        const int b = threadIdx.x + j * kT;
        if (b < nb && run_ok(f.p0[j], f.p1[j], nnz) && f.p1[j] > f.p0[j]) {
            const int64_t r = runs[b];
            runD[run_ci(r)] = f.p0[j] - run_off(r);
        }
    }
    for (int b = threadIdx.x + kRunRegs * kT; b < nb; b += kT) {
        const int32_t p0 = runStart[static_cast<int64_t>(t) * nb + b];
        const int32_t p1 = runStart[static_cast<int64_t>(t + 1) * nb + b];
        if (run_ok(p0, p1, nnz) && p1 > p0) {
            const int64_t r = runs[b];
            runD[run_ci(r)] = p0 - run_off(r);
        }
    }
    __syncthreads();
    return bad_runs == 0;
}

// all[i] without a dynamically indexed array (keeps the pointers in
// registers instead of the local-memory stack).
template <int CS>
__device__ __forceinline__ double *pick(double *const *all, int i)
{
    if constexpr (CS == 1)
        return all[0];
    else if constexpr (CS == 2)
        return i ? all[1] : all[0];
    else
        return i < 2 ? (i ? all[1] : all[0]) : (i == 3 ? all[3] : all[2]);
}

// Bit 15 of a pass-1 source offset marks the first slot of a run.
constexpr uint32_t kRunStart = 0x8000u;

// Writes the tile's slots [kbeg, kend) to the work array: slot k of the
// i-th non-empty run goes to work[runD[i] + k], its value taken from the
// cluster's staged tile at offset src[base + k] & 0x7fff (block o / per
// holds offsets [o*per, (o+1)*per)).  Each warp takes one contiguous range
// of slots, 32 (one per lane) at a time, so the src loads and the work
// stores of a warp instruction are contiguous.  A lane's run is the number
// of run starts up to its slot (one ballot and a population count over the
// warp's 32 slots), counted from the run holding the warp's first slot
// (one binary search); the next range's offsets are loaded while the
// current range is written.  Every destination is checked against the
// work array's length, so a corrupted table cannot write outside it.
template <int CS>
__device__ __forceinline__ bool emit_runs(const int64_t *runs, const int32_t *runD, int nb,
                                          int32_t kbeg, int32_t kend, const uint16_t *src,
                                          int64_t base, double *const *tile, int per, int nvals,
                                          double *work, int64_t nwork)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kT / 32;
    const int64_t n = kend - kbeg;
    const int32_t wb = kbeg + static_cast<int32_t>(n * warp / kWarps);
    const int32_t we = kbeg + static_cast<int32_t>(n * (warp + 1) / kWarps);
    if (wb >= we)
        return false;
    const uint32_t le_mask = (2u << lane) - 1u;  // lanes <= this lane
    const int32_t nne = run_ci(runs[nb]);         // non-empty runs (>= 1 here)
    // non-empty runs starting before slot wb, minus one
    const int64_t rb = runs[find_run(runs, nb, wb)];
    int32_t before = run_ci(rb) + (run_off(rb) < wb ? 1 : 0) - 1;
    bool bad = false;
    uint16_t o[kU], on[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int32_t k = wb + 32 * u + lane;
        o[u] = k < we ? ld_u16(src + base + k) : 0;
    }
    for (int32_t c0 = wb; c0 < we; c0 += 32 * kU) {
        const int32_t c1 = c0 + 32 * kU;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t k = c1 + 32 * u + lane;
            on[u] = k < we ? ld_u16(src + base + k) : 0;
        }
        // straight-line over the chunk (no early exit), so that the loads
        // of later groups overlap the stores of earlier ones; slots past
        // `we` carry offset 0 (no run start) and store nothing
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (c0 + 32 * u >= we)  // (warp-uniform) the rest of the last chunk is past the range
                break;
            const int32_t k = c0 + 32 * u + lane;
            const uint32_t raw = o[u];
            const uint32_t starts = __ballot_sync(0xffffffffu, raw & kRunStart);
            const int32_t c = before + __popc(starts & le_mask);
            before += __popc(starts);
            if (k < we) {
                const uint32_t off = raw & (kRunStart - 1u);
                double v = 0.0;
                if (off < static_cast<uint32_t>(nvals)) {
                    const int owner = CS == 1 ? 0 : off / per;
                    v = pick<CS>(tile, owner)[off - owner * per];
                } else {
                    bad = true;
                }
                // 32-bit unsigned arithmetic: positions are below nnz < 2^31,
                // and a corrupted table can only yield d >= nwork (skipped)
                const uint32_t ci = static_cast<uint32_t>(c);
                bad |= ci >= static_cast<uint32_t>(nne);
                const uint32_t d = static_cast<uint32_t>(runD[ci < static_cast<uint32_t>(nne) ? ci : 0u]) +
                                   static_cast<uint32_t>(k);
                if (d < static_cast<uint32_t>(nwork))
                    work[d] = v;
                else
                    bad = true;
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
            o[u] = on[u];
    }
    return bad;
}

// Steps of 32 slots per chunk of the gather runs' writes (gather pass 1 and
// the fused operator): measured best of 2, 3, 4, 6, 8, 12, 16 on the stress
// and large meshes (the scatter's pass 1 keeps kU: 4 was 3 us slower per
// stress scatter).
constexpr int kGatherEmitSteps = 4;

// One chunk of 32 kE slots of emit_runs_lean: lane slots c0 + 32 u + lane,
// offsets o[u]; kTail: only slots below `we` exist (the warp's last chunk).
// Shared-memory reads are clamped into the tile (vmax) and the run table
// (cmax); a value out of range sets the returned flag.
template <bool kTail, int kE>
__device__ __forceinline__ uint32_t emit_chunk(const uint16_t (&o)[kE], int32_t c0, int32_t we,
                                               int32_t &before, uint32_t le_mask, const double *tile,
                                               uint32_t vmax, const int32_t *runD, uint32_t cmax,
                                               double *work, uint32_t nwork)
{
    const int lane = threadIdx.x & 31;
    uint32_t bad = 0;
#pragma unroll
    for (int u = 0; u < kE; ++u) {
        if (kTail && c0 + 32 * u >= we)  // (warp-uniform) past the warp's range
            break;
        const int32_t k = c0 + 32 * u + lane;
        const uint32_t raw = o[u];
        const uint32_t starts = __ballot_sync(0xffffffffu, raw & kRunStart);
        const uint32_t c = static_cast<uint32_t>(before + __popc(starts & le_mask));
        before += __popc(starts);
        const uint32_t off = raw & (kRunStart - 1u);
        const double v = tile[min(off, vmax)];
        const uint32_t d = static_cast<uint32_t>(runD[min(c, cmax)]) + static_cast<uint32_t>(k);
        const bool in = !kTail || k < we;
        bad |= static_cast<uint32_t>(in && (off > vmax || c > cmax || d >= nwork));
        if (in && d < nwork)
            work[d] = v;
    }
    return bad;
}

// emit_runs for one block (cluster 1) with fewer instructions per slot: a
// warp's full chunks of 32 kE slots carry no per-slot range test, and the
// table checks are clamps plus one flag instead of branches.  Same writes,
// same checks.
template <int kE = kU>
__device__ __forceinline__ bool emit_runs_lean(const int64_t *runs, const int32_t *runD, int nb,
                                               int32_t kbeg, int32_t kend, const uint16_t *src,
                                               int64_t base, const double *tile, int nvals,
                                               double *work, int64_t nwork)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kT / 32;
    const int64_t n = kend - kbeg;
    const int32_t wb = kbeg + static_cast<int32_t>(n * warp / kWarps);
    const int32_t we = kbeg + static_cast<int32_t>(n * (warp + 1) / kWarps);
    if (wb >= we)
        return false;
    const int32_t nne = run_ci(runs[nb]);  // non-empty runs
    if (nvals < 1 || nne < 1)
        return true;
    const uint32_t le_mask = (2u << lane) - 1u;
    const int64_t rb = runs[find_run(runs, nb, wb)];
    int32_t before = run_ci(rb) + (run_off(rb) < wb ? 1 : 0) - 1;
    const uint32_t vmax = static_cast<uint32_t>(nvals - 1), cmax = static_cast<uint32_t>(nne - 1);
    const uint32_t nw = static_cast<uint32_t>(nwork);  // nwork <= nnz < 2^31
    const uint16_t *sp = src + base;
    constexpr int32_t kChunk = 32 * kE;
    const int32_t wf = wb + (we - wb) / kChunk * kChunk;  // end of the full chunks
    uint32_t bad = 0;
    uint16_t o[kE];
    if (wb < wf) {
#pragma unroll
        for (int u = 0; u < kE; ++u)
            o[u] = ld_u16(sp + wb + 32 * u + lane);
    }
    for (int32_t c0 = wb; c0 < wf; c0 += kChunk) {
        // the next chunk's offsets (or the tail's) load while this one is written
        const int32_t c1 = c0 + kChunk;
        uint16_t on[kE];
#pragma unroll
        for (int u = 0; u < kE; ++u) {
            const int32_t k = c1 + 32 * u + lane;
            on[u] = k < we ? ld_u16(sp + k) : 0;
        }
        bad |= emit_chunk<false, kE>(o, c0, we, before, le_mask, tile, vmax, runD, cmax, work, nw);
#pragma unroll
        for (int u = 0; u < kE; ++u)
            o[u] = on[u];
    }
    if (wf < we) {
        if (wf == wb) {  // no full chunk: the tail's offsets are not loaded yet
#pragma unroll
            for (int u = 0; u < kE; ++u) {
                const int32_t k = wb + 32 * u + lane;
                o[u] = k < we ? ld_u16(sp + k) : 0;
            }
        }
        bad |= emit_chunk<true, kE>(o, wf, we, before, le_mask, tile, vmax, runD, cmax, work, nw);
    }
    return bad != 0;
}

template <int CS>
__device__ __forceinline__ void cluster_barrier()
{
    if constexpr (CS > 1)
        cg::this_cluster().sync();
    else
        __syncthreads();
}

template <int CS>
__device__ __forceinline__ int cluster_rank()
{
    if constexpr (CS > 1)
        return static_cast<int>(cg::this_cluster().block_rank());
    else
        return 0;
}

// Pointers to the same shared-memory array in every block of the cluster.
template <int CS>
__device__ __forceinline__ void map_cluster(double *mine, double **all)
{
    if constexpr (CS > 1) {
        cg::cluster_group cl = cg::this_cluster();
#pragma unroll
        for (int j = 0; j < CS; ++j)
            all[j] = cl.map_shared_rank(mine, j);
    } else {
        all[0] = mine;
    }
}

// ------------------------------------------- L2 prefetch of a block's next item
// In a persistent grid each block takes items blockIdx, blockIdx + step, ...
// (step = the number of blocks or clusters), so it knows its next tile or
// bucket; one lane asks the bulk-copy engine to bring that item's
// sequential inputs into L2 while the block works on the current one, so
// that the next staging or placement reads L2 instead of waiting on HBM.
// Ranges come from the tables, clamped into the arrays.
__device__ __forceinline__ bool pf_lane() { return threadIdx.x == kT - 32; }

__device__ void pf_scatter_tile(const PlanArgs &a, int t, const double *qG)
{
    const int64_t B = a.s_nbuckets;
    int64_t r0 = a.s_tileRows[t], r1 = a.s_tileRows[t + 1];
    if (clamp_range(r0, r1, a.NG)) {
        prefetch_l2(qG + r0, 8 * (r1 - r0));
        int64_t e0 = a.rowStarts[r0], e1 = a.rowStarts[r1];
        if (clamp_range(e0, e1, a.nnz))
            prefetch_l2(a.s_src + e0, 2 * (e1 - e0));
    }
    prefetch_l2(a.s_runStart + t * B, 8 * B);
}

__device__ void pf_scatter_bucket(const PlanArgs &a, int b, const double *ws)
{
    int64_t j0 = a.s_runStart[b];
    int64_t j1 = a.s_runStart[static_cast<int64_t>(a.s_ntiles) * a.s_nbuckets + b];
    if (clamp_range(j0, j1, a.nnz)) {
        prefetch_l2(ws + j0, 8 * (j1 - j0));
        prefetch_l2(a.s_dst + j0, 2 * (j1 - j0));
    }
}

__device__ void pf_gather_tile(const PlanArgs &a, int u, const double *qL)
{
    const int64_t C = a.g_nbuckets;
    int64_t l0 = static_cast<int64_t>(u) * a.g_tile_len, l1 = l0 + a.g_tile_len;
    if (clamp_range(l0, l1, a.NL))
        prefetch_l2(qL + l0, 8 * (l1 - l0));
    int64_t s0 = a.g_tileSlot[u], s1 = a.g_tileSlot[u + 1];
    if (clamp_range(s0, s1, a.nnz))
        prefetch_l2(a.g_src + s0, 2 * (s1 - s0));
    prefetch_l2(a.g_runStart + u * C, 8 * C);
}

__device__ void pf_gather_bucket(const PlanArgs &a, int c, const double *wg)
{
    int64_t b0 = a.g_subRows[c], b1 = a.g_subRows[c + 1];
    if (!clamp_range(b0, b1, a.NG))
        return;
    prefetch_l2(a.g_rowPos + b0, 2 * (b1 - b0));
    int64_t e0 = a.rowStarts[b0], e1 = a.rowStarts[b1];
    if (clamp_range(e0, e1, a.nnz)) {
        prefetch_l2(wg + e0, 8 * (e1 - e0));
        prefetch_l2(a.g_pos + e0, 2 * (e1 - e0));
    }
}

// Block-uniform "a bulk staging wait ran out": the barrier's phase is then
// unknown, so the block stops using bulk copies for the rest of the launch.
struct StageState {
    uint32_t parity = 0;
    bool broken = false;
};

__device__ __forceinline__ bool stage_done(StageState &st, bool bulk, uint64_t *bar)
{
    const bool staged = stage_wait(bulk, bar, st.parity);
    if (bulk)
        st.parity ^= 1u;
    if (!staged)
        st.broken = true;
    return staged;
}

// --------------------------------------------------------------- scatter
// One cluster per tile of CS * s_tile_rows global rows; block r stages rows
// [r * s_tile_rows, (r+1) * s_tile_rows) of it and emits 1/CS of the slots.
// A grid with fewer clusters than tiles loops over tiles (persistent).
template <int CS>
__global__ void __launch_bounds__(kT, 1) scatter_tile_kernel(PlanArgs a, const double *__restrict__ qG)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *vals = reinterpret_cast<double *>(smem);
    int64_t *runs = reinterpret_cast<int64_t *>(vals + a.s_tile_rows);
    int32_t *runD = reinterpret_cast<int32_t *>(runs + a.s_nbuckets + 1);
    __shared__ uint64_t bar;
    if (threadIdx.x == 0)
        mbar_init(&bar);
    __syncthreads();
    const int r = cluster_rank<CS>();
    const int step = static_cast<int>(gridDim.x) / CS;
    double *tile[CS];
    map_cluster<CS>(vals, tile);
    StageState st;
    for (int t = static_cast<int>(blockIdx.x) / CS; t < a.s_ntiles; t += step) {
        // The plan's tiles are the row ranges [t TR, (t+1) TR) clipped to
        // N_G, so the staging starts without waiting for a table;
        // s_tileRows and the CSR entry range are loaded meanwhile and
        // checked before use.
        const int64_t TR = static_cast<int64_t>(CS) * a.s_tile_rows;
        const int32_t r0 = static_cast<int32_t>(min(t * TR, a.NG));
        const int32_t r1 = static_cast<int32_t>(min((t + 1) * TR, a.NG));
        const int32_t nrows = r1 - r0;
        const int32_t e0 = a.rowStarts[r0], e1 = a.rowStarts[r1];
        if (pf_lane()) {  // the run writes' source offsets, read after the staging
            int64_t p0 = e0, p1 = e1;
            if (clamp_range(p0, p1, a.nnz))
                prefetch_l2(a.s_src + p0, 2 * (p1 - p0));
        }
        bool ok = a.s_tileRows[t] == r0 && a.s_tileRows[t + 1] == r1 && !st.broken;
        const int32_t m0 = min(r * a.s_tile_rows, nrows);
        const int32_t m1 = min((r + 1) * a.s_tile_rows, nrows);
        const bool bulk = stage_start(vals, qG + r0 + m0, m1 - m0, &bar, !st.broken);
        ok = ok && e0 >= 0 && e1 >= e0 && e1 <= a.nnz;
        const RunFetch rf = fetch_runs(a.s_runStart, t, a.s_nbuckets);
        if (!bulk)
            stage(vals, qG + r0 + m0, m1 - m0);
        ok = commit_runs(rf, a.s_runStart, t, a.s_nbuckets, a.nnz, runs, runD) && ok &&
             run_off(runs[a.s_nbuckets]) == e1 - e0;
        ok = stage_done(st, bulk, &bar) && ok;
        if (a.pf_next && pf_lane() && t + step < a.s_ntiles)
            pf_scatter_tile(a, t + step, qG);
        cluster_barrier<CS>();  // every block's slice is staged
        if (ok) {
            const int32_t total = e1 - e0;
            const int32_t kb = static_cast<int32_t>(static_cast<int64_t>(total) * r / CS);
            const int32_t ke = static_cast<int32_t>(static_cast<int64_t>(total) * (r + 1) / CS);
            const bool bad = CS == 1
                                 ? emit_runs_lean(runs, runD, a.s_nbuckets, kb, ke, a.s_src, e0, vals, nrows,
                                                  a.work, a.nnz)
                                 : emit_runs<CS>(runs, runD, a.s_nbuckets, kb, ke, a.s_src, e0, tile,
                                                 a.s_tile_rows, nrows, a.work, a.nnz);
            if (bad)
                flag(a.err);
        } else if (threadIdx.x == 0) {
            flag(a.err);
        }
        cluster_barrier<CS>();  // peers may still read this block's slice
    }
}

// One cluster per bucket of CS * s_bucket_len locals; block r holds locals
// [r * s_bucket_len, (r+1) * s_bucket_len) of it and places 1/CS of the
// bucket's work entries (into any block of the cluster).  A grid with
// fewer clusters than buckets loops over buckets (persistent).
template <int CS>
__global__ void __launch_bounds__(kT, 1) scatter_bucket_kernel(PlanArgs a, double *__restrict__ qL)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *out = reinterpret_cast<double *>(smem);
    const int r = cluster_rank<CS>();
    const int step = static_cast<int>(gridDim.x) / CS;
    double *dst[CS];
    map_cluster<CS>(out, dst);
    for (int b = static_cast<int>(blockIdx.x) / CS; b < a.s_nbuckets; b += step) {
        if (a.pf_next && pf_lane() && b + step < a.s_nbuckets)
            pf_scatter_bucket(a, b + step, a.work);
        const int32_t per = a.s_bucket_len;
        const int64_t l0 = static_cast<int64_t>(b) * CS * per;
        const int64_t rest = a.NL - l0;
        const int32_t len =
            static_cast<int32_t>(rest < static_cast<int64_t>(CS) * per ? rest : CS * per);
        const int32_t mine = max(0, min(per, len - r * per));
        const int32_t j0 = a.s_runStart[b];
        const int32_t j1 = a.s_runStart[static_cast<int64_t>(a.s_ntiles) * a.s_nbuckets + b];
        if (a.pf_s2 && pf_lane()) {
            int64_t p0 = j0 + 2048, p1 = j1;  // past what the first loads take
            if (clamp_range(p0, p1, a.nnz)) {
                prefetch_l2(a.work + p0, 8 * (p1 - p0));
                prefetch_l2(a.s_dst + p0, 2 * (p1 - p0));
            }
        }
        const bool ok = len > 0 && j0 >= 0 && j1 >= j0 && j1 <= a.nnz && j1 - j0 <= len;
        // pre-zeroed for masked locals; a bucket with as many entries as
        // locals has none (every local has exactly one entry), and every
        // slot is placed
        if (!(ok && j1 - j0 == len))
            for (int32_t i = threadIdx.x; i < mine; i += kT)
                out[i] = 0.0;
        cluster_barrier<CS>();  // every block's slice is zeroed
        bool bad = !ok;
        if (ok) {
            const int32_t n = j1 - j0;
            const int32_t jb = j0 + static_cast<int32_t>(static_cast<int64_t>(n) * r / CS);
            const int32_t je = j0 + static_cast<int32_t>(static_cast<int64_t>(n) * (r + 1) / CS);
            stream_entries<CS == 1 ? kU : 6, true>(a.s_dst, a.work, jb, je, [&](uint32_t d, double v) {
                if (d < static_cast<uint32_t>(len)) {
                    const int owner = CS == 1 ? 0 : d / per;
                    pick<CS>(dst, owner)[d - owner * per] = v;
                } else {
                    bad = true;
                }
            });
        }
        if constexpr (CS == 1)  // the placements are read next by the bulk-copy engine
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        cluster_barrier<CS>();  // every placement has landed
        const int64_t q0 = l0 + static_cast<int64_t>(r) * per;
        if (CS == 1 && mine >= 2 && (reinterpret_cast<uintptr_t>(qL + q0) & 15u) == 0) {
            if (threadIdx.x == 0)
                bulk_store(qL + q0, out, static_cast<uint32_t>(mine & ~1) * 8u);
            if ((mine & 1) && threadIdx.x == 32)
                qL[q0 + mine - 1] = out[mine - 1];
        } else {
            for (int32_t i = threadIdx.x; i < mine; i += kT)
                qL[q0 + i] = out[i];
        }
        if (bad && (threadIdx.x == 0 || ok))
            flag(a.err);
        // the bulk store has read `out` (thread 0 waited for it) and the
        // peers are done with this slice before it is zeroed again
        cluster_barrier<CS>();
    }
}

// ---------------------------------------------------------------- gather
// One cluster per tile of CS * g_tile_len locals; a grid with fewer
// clusters than tiles loops over tiles (persistent).
template <int CS, int kE = kGatherEmitSteps>
__global__ void __launch_bounds__(kT, 1) gather_tile_kernel(PlanArgs a, const double *__restrict__ qL)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *vals = reinterpret_cast<double *>(smem);
    int64_t *runs = reinterpret_cast<int64_t *>(vals + a.g_tile_len);
    int32_t *runD = reinterpret_cast<int32_t *>(runs + a.g_nbuckets + 1);
    __shared__ uint64_t bar;
    if (threadIdx.x == 0)
        mbar_init(&bar);
    __syncthreads();
    const int r = cluster_rank<CS>();
    const int step = static_cast<int>(gridDim.x) / CS;
    double *tile[CS];
    map_cluster<CS>(vals, tile);
    StageState st;
    for (int u = static_cast<int>(blockIdx.x) / CS; u < a.g_ntiles; u += step) {
        const int32_t per = a.g_tile_len;
        const int64_t l0 = static_cast<int64_t>(u) * CS * per;
        const int64_t rest = a.NL - l0;
        const int32_t len =
            static_cast<int32_t>(rest < static_cast<int64_t>(CS) * per ? rest : CS * per);
        const int32_t s0 = a.g_tileSlot[u], s1 = a.g_tileSlot[u + 1];
        if (pf_lane()) {  // the run writes' source offsets, read after the staging
            int64_t p0 = s0, p1 = s1;
            if (clamp_range(p0, p1, a.nnz))
                prefetch_l2(a.g_src + p0, 2 * (p1 - p0));
        }
        bool ok = len > 0 && s0 >= 0 && s1 >= s0 && s1 <= a.nnz && s1 - s0 <= len && !st.broken;
        const int32_t m0 = ok ? min(r * per, len) : 0, m1 = ok ? min((r + 1) * per, len) : 0;
        const bool bulk = stage_start(vals, qL + l0 + m0, m1 - m0, &bar, !st.broken);
        const RunFetch rf = fetch_runs(a.g_runStart, u, a.g_nbuckets);
        if (!bulk)
            stage(vals, qL + l0 + m0, m1 - m0);
        ok = commit_runs(rf, a.g_runStart, u, a.g_nbuckets, a.nnz, runs, runD) && ok &&
             run_off(runs[a.g_nbuckets]) == s1 - s0;
        ok = stage_done(st, bulk, &bar) && ok;
        if (a.pf_next && pf_lane() && u + step < a.g_ntiles)
            pf_gather_tile(a, u + step, qL);
        cluster_barrier<CS>();
        if (ok) {
            const int32_t total = s1 - s0;
            const int32_t kb = static_cast<int32_t>(static_cast<int64_t>(total) * r / CS);
            const int32_t ke = static_cast<int32_t>(static_cast<int64_t>(total) * (r + 1) / CS);
            const bool bad = CS == 1
                                 ? emit_runs_lean<kE>(runs, runD, a.g_nbuckets, kb, ke, a.g_src, s0, vals, len,
                                                  a.work, a.nnz)
                                 : emit_runs<CS>(runs, runD, a.g_nbuckets, kb, ke, a.g_src, s0, tile, per,
                                                 len, a.work, a.nnz);
            if (bad)
                flag(a.err);
        } else if (threadIdx.x == 0) {
            flag(a.err);
        }
        cluster_barrier<CS>();
    }
}

// One cluster per bucket = CS consecutive sub-buckets of rows; block r
// holds sub-bucket r, its values staged grouped by row length; it places
// 1/CS of the bucket's work entries into the owning block, then sums its
// rows group by group (a warp's lanes all sum rows of the same length) and
// writes its rows of q_G in order.  A grid with fewer clusters than
// buckets loops over buckets (persistent).
template <int CS>
__global__ void __launch_bounds__(kT, 1) gather_bucket_kernel(PlanArgs a, double *__restrict__ qG)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *vals = reinterpret_cast<double *>(smem);
    int32_t *grp = reinterpret_cast<int32_t *>(vals + a.g_bucket_entries_max);  // [mmax+1]
    __shared__ int32_t grpRows[kMaxRow + 1];  // rows of each length
    __shared__ int grp_bad;
    const int r = cluster_rank<CS>();
    const int step = static_cast<int>(gridDim.x) / CS;
    double *dst[CS];
    map_cluster<CS>(vals, dst);
    const int MM = a.g_mmax;
    for (int c = static_cast<int>(blockIdx.x) / CS; c < a.g_nbuckets; c += step) {
        if (a.pf_next && pf_lane() && c + step < a.g_nbuckets)
            pf_gather_bucket(a, c + step, a.work);
        const int64_t sb = static_cast<int64_t>(c) * CS + r;
        // Independent loads first: the bucket's work range, this block's
        // rows and its group table.
        const int32_t j0 = a.g_runStart[c];
        const int32_t j1 = a.g_runStart[static_cast<int64_t>(a.g_ntiles) * a.g_nbuckets + c];
        const int32_t r0 = a.g_subRows[sb], r1 = a.g_subRows[sb + 1];
        const int32_t nrows = r1 - r0;
        bool ok = MM >= 1 && MM <= kMaxRow && r0 >= 0 && nrows >= 0 && r1 <= a.NG;
        if (MM >= 1 && MM <= kMaxRow && threadIdx.x <= MM)
            grp[threadIdx.x] = a.g_groupStart[sb * (MM + 1) + threadIdx.x];
        // entry offsets of the CS sub-buckets relative to the bucket start
        int32_t sub[CS + 1];
        int32_t E0;
        bool csr_ok = true;  // the plan agrees with the CSR (checked late)
        if constexpr (CS == 1) {
            // the bucket's work range is its CSR entry range: no dependent
            // load before the placement; rowStarts is compared after it
            E0 = j0;
            sub[0] = 0;
            sub[1] = j1 - j0;
            ok = ok && sub[1] <= a.g_bucket_entries_max;
            const int32_t s0 = ok ? a.rowStarts[r0] : 0, s1 = ok ? a.rowStarts[r1] : 0;
            csr_ok = s0 == j0 && s1 == j1;
        } else {
            const int32_t b0 = a.g_subRows[static_cast<int64_t>(c) * CS];
            ok = ok && b0 >= 0 && b0 <= a.NG;
            E0 = ok ? a.rowStarts[b0] : 0;
#pragma unroll
            for (int j = 0; j <= CS; ++j) {
                const int32_t row = a.g_subRows[static_cast<int64_t>(c) * CS + j];
                ok = ok && row >= b0 && row <= a.NG;
                sub[j] = ok ? a.rowStarts[row] - E0 : 0;
                if (j > 0)
                    ok = ok && sub[j] >= sub[j - 1] && sub[j] - sub[j - 1] <= a.g_bucket_entries_max;
            }
            ok = ok && j0 == E0 && j1 == E0 + sub[CS];
        }
        int32_t mine0 = sub[0], mine1 = sub[1];
#pragma unroll
        for (int w = 1; w < CS; ++w)
            if (r == w) {
                mine0 = sub[w];
                mine1 = sub[w + 1];
            }
        const int32_t ne = sub[CS], mine = mine1 - mine0;
        ok = ok && E0 >= 0 && ne >= 0 && E0 + ne <= a.nnz;
        if (threadIdx.x == 0)
            grp_bad = 0;
        cluster_barrier<CS>();  // all blocks resident; grp staged
        if (ok && threadIdx.x == 0) {
            // rows of length m: (grp[m] - grp[m-1]) / m
            int bad = grp[0] != 0 || grp[MM] != mine;
            int32_t acc = 0;
            for (int m = 1; m <= MM; ++m) {
                const int32_t len = grp[m] - grp[m - 1];
                bad |= len < 0 || len % m != 0;
                grpRows[m] = len / m;
                acc += len / m;
            }
            bad |= acc > nrows;
            grp_bad = bad;
        }
        bool bad = false;
        if (ok) {
            const int32_t jb = static_cast<int32_t>(static_cast<int64_t>(ne) * r / CS);
            const int32_t je = static_cast<int32_t>(static_cast<int64_t>(ne) * (r + 1) / CS);
            stream_entries<CS == 1 ? kU : 6>(a.g_pos + E0, a.work + E0, jb, je,
                                             [&](uint32_t p, double v) {
                if (p < static_cast<uint32_t>(ne)) {
                    int owner = 0;
                    int32_t base = sub[0];
#pragma unroll
                    for (int w = 1; w < CS; ++w) {
                        owner += p >= static_cast<uint32_t>(sub[w]);
                        base = p >= static_cast<uint32_t>(sub[w]) ? sub[w] : base;
                    }
                    pick<CS>(dst, owner)[p - base] = v;
                } else {
                    bad = true;
                }
            });
        }
        // the first rows' staged positions, in flight during the row sums
        constexpr int kRP = 16;
        uint16_t rp[kRP];
#pragma unroll
        for (int q = 0; q < kRP; ++q) {
            const int32_t k = threadIdx.x + q * kT;
            rp[q] = ok && k < nrows ? ld_u16(a.g_rowPos + r0 + k) : 0;
        }
        cluster_barrier<CS>();  // every placement has landed; grpRows ready
        const bool go = ok && grp_bad == 0 && csr_ok;
        if (go) {
            // sums group by group, in place into each row's first slot; a
            // group is column-major, so the lanes of a warp read
            // consecutive words (a one-entry row is its own sum)
            for (int m = 2; m <= MM; ++m)
                group_sums(vals, grp[m - 1], m, grpRows[m], threadIdx.x, kT);
        }
        __syncthreads();
        if (go) {
            // q_G[row] = the row's sum, +0.0 for a row without entries (0xFFFF)
#pragma unroll
            for (int q = 0; q < kRP; ++q) {
                const int32_t k = threadIdx.x + q * kT;
                if (k < nrows) {
                    double v = 0.0;
                    if (rp[q] != 0xFFFF) {
                        if (rp[q] < mine)
                            v = plus_zero(vals[rp[q]]);
                        else
                            bad = true;
                    }
                    qG[r0 + k] = v;
                }
            }
            for (int32_t k0 = kRP * kT + threadIdx.x; k0 < nrows; k0 += kU * kT) {
                uint16_t p[kU];
#pragma unroll
                for (int q = 0; q < kU; ++q)
                    p[q] = k0 + q * kT < nrows ? ld_u16(a.g_rowPos + r0 + k0 + q * kT) : 0;
#pragma unroll
                for (int q = 0; q < kU; ++q)
                    if (k0 + q * kT < nrows) {
                        double v = 0.0;
                        if (p[q] != 0xFFFF) {
                            if (p[q] < mine)
                                v = plus_zero(vals[p[q]]);
                            else
                                bad = true;
                        }
                        qG[r0 + k0 + q * kT] = v;
                    }
            }
        }
        if (bad || (!go && threadIdx.x == 0))
            flag(a.err);
        cluster_barrier<CS>();  // vals, grp and grpRows are rewritten next
    }
}

// ------------------------------------------- gather pass 2 with a TMEM buffer
// The bucket kernel above holds one bucket in shared memory, so each SM
// runs its phases back to back: place (read the work range from HBM, ~8 us
// on the stress mesh), sum (binary64, ~3.4 us), write q_G (~4 us), and HBM
// idles while the SM sums.  Here the SM's tensor memory (TMEM: 128 lanes x
// 512 columns of 32 bits, 256 KB, otherwise unused by this library) holds
// the NEXT bucket's work entries and positions: warps 16..31 stream them
// from HBM into TMEM while warps 0..15 sum and write the current bucket,
// and the placement then reads TMEM instead of waiting on HBM.  Persistent:
// one block per SM, buckets blockIdx.x, blockIdx.x + gridDim.x, ...  The
// row sums and q_G writes run on fewer warps than in the kernel above and
// slow down somewhat; on the stress mesh a gather call still gains ~6%.
//
// TMEM layout of a bucket's entries j < ne: entry j sits in lane j % 128 of
// 128-entry block j / 128; blocks are grouped by 8.  Group g's values take
// columns 16 g .. 16 g + 15 (block 8 g + k: columns 16 g + 2 k and + 1, the
// low and high words); its 16-bit positions take columns pc + 4 g .. + 3
// (column pc + 4 g + i: blocks 8 g + 2 i in the low half, 8 g + 2 i + 1 in
// the high half), entries past ne carry position 0xFFFF.  A warp reaches
// the 32 lanes of its quarter (warp index mod 4) only, so lane 32 q + t of
// every block is loaded, stored and read by lane t of warps in quarter q.
constexpr int kTmGroupEntries = 1024; // 8 blocks of 128 entries
constexpr int kTmCols = 512;

__device__ __forceinline__ void tm_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tm_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Block barrier that also orders the threads' TMEM accesses around it.
__device__ __forceinline__ void tm_sync()
{
    tm_fence_before();
    __syncthreads();
    tm_fence_after();
}

__device__ __forceinline__ void tm_st16(uint32_t addr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, "
                 "%9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(addr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
                 "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tm_st4(uint32_t addr, const uint32_t (&r)[4])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ void tm_ld16(uint32_t addr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
                 "%10, %11, %12, %13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void tm_ld4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Work range [j0, j1) of gather bucket c (cluster 1), if the tables hold a
// valid one that fits the staging (the checks both the loaders and the
// placing threads apply).
__device__ __forceinline__ bool tm_bucket_range(const PlanArgs &a, int c, int32_t &j0, int32_t &ne)
{
    j0 = a.g_runStart[c];
    const int32_t j1 = a.g_runStart[static_cast<int64_t>(a.g_ntiles) * a.g_nbuckets + c];
    ne = j1 - j0;
    return j0 >= 0 && j1 >= j0 && j1 <= a.nnz && ne <= a.g_bucket_entries_max;
}

// Loader warp (quarter q, index i of n in its quarter): entries and
// positions of [w, w + ne) into TMEM, groups i, i + n, ...
__device__ __forceinline__ void tm_load(uint32_t lane_addr, int pc, const double *w,
                                        const uint16_t *pos, int32_t ne, int q, int i, int n)
{
    const int lane = threadIdx.x & 31;
    const int ng = (ne + kTmGroupEntries - 1) / kTmGroupEntries;
    for (int g = i; g < ng; g += n) {
        double d[8];
        uint32_t p[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int32_t j = (g * 8 + k) * 128 + q * 32 + lane;
            d[k] = j < ne ? ld_seq(w + j) : 0.0;
            p[k] = j < ne ? static_cast<uint32_t>(ld_u16(pos + j)) : 0xFFFFu;
        }
        uint32_t v[16], pk[4];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            v[2 * k] = static_cast<uint32_t>(__double2loint(d[k]));
            v[2 * k + 1] = static_cast<uint32_t>(__double2hiint(d[k]));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            pk[k] = p[2 * k] | (p[2 * k + 1] << 16);
        tm_st16(lane_addr + 16u * g, v);
        tm_st4(lane_addr + pc + 4u * g, pk);
    }
    tm_wait_st();
}

// Placing warp (quarter q, index i of n): vals[pos[j]] = w[j] for the
// bucket's entries in TMEM, groups i, i + n, ...; returns true on a
// position outside [0, ne) (skipped).
__device__ __forceinline__ bool tm_place(uint32_t lane_addr, int pc, double *vals, int32_t ne, int q,
                                         int i, int n)
{
    const int lane = threadIdx.x & 31;
    const int ng = (ne + kTmGroupEntries - 1) / kTmGroupEntries;
    bool bad = false;
    for (int g = i; g < ng; g += n) {
        uint32_t v[16], pk[4];
        tm_ld16(lane_addr + 16u * g, v);
        tm_ld4(lane_addr + pc + 4u * g, pk);
        tm_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int32_t j = (g * 8 + k) * 128 + q * 32 + lane;
            const uint32_t pos = (pk[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
            if (j < ne) {
                if (pos < static_cast<uint32_t>(ne))
                    vals[pos] = __hiloint2double(static_cast<int>(v[2 * k + 1]), static_cast<int>(v[2 * k]));
                else
                    bad = true;
            }
        }
    }
    return bad;
}

// kTmWorkers warps (a multiple of 4) sum and write; the others load.
constexpr int kTmWorkersDefault = 20;
template <int kTmWorkers>
__global__ void __launch_bounds__(kT, 1) gather_bucket_tm_kernel(PlanArgs a, double *__restrict__ qG,
                                                                 int pc)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *vals = reinterpret_cast<double *>(smem);
    int32_t *grp = reinterpret_cast<int32_t *>(vals + a.g_bucket_entries_max);  // [mmax+1]
    __shared__ int32_t grpRows[kMaxRow + 1];
    __shared__ int grp_bad;
    __shared__ uint32_t s_taddr;
    const int warp = threadIdx.x >> 5, q = warp & 3;
    const bool worker = warp < kTmWorkers;
    const int step = static_cast<int>(gridDim.x);
    const int MM = a.g_mmax;
    constexpr int kW = kTmWorkers * 32;  // worker threads
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(&s_taddr))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tm_sync();
    const uint32_t lane_addr = s_taddr + (static_cast<uint32_t>(q * 32) << 16);
    int c = static_cast<int>(blockIdx.x);
    if (!worker && c < a.g_nbuckets) {  // the first bucket
        int32_t j0, ne;
        if (tm_bucket_range(a, c, j0, ne))
            tm_load(lane_addr, pc, a.work + j0, a.g_pos + j0, ne, q, (warp - kTmWorkers) >> 2,
                    (32 - kTmWorkers) / 4);
    }
    tm_sync();
    for (; c < a.g_nbuckets; c += step) {
        // this bucket's entries are in TMEM
        int32_t j0, ne;
        const bool range_ok = tm_bucket_range(a, c, j0, ne);
        const int32_t r0 = a.g_subRows[c], r1 = a.g_subRows[c + 1];
        const int32_t nrows = r1 - r0;
        bool ok = range_ok && MM >= 1 && MM <= kMaxRow && r0 >= 0 && nrows >= 0 && r1 <= a.NG;
        if (MM >= 1 && MM <= kMaxRow && threadIdx.x <= MM)
            grp[threadIdx.x] = a.g_groupStart[static_cast<int64_t>(c) * (MM + 1) + threadIdx.x];
        const int32_t s0 = ok ? a.rowStarts[r0] : 0, s1 = ok ? a.rowStarts[r1] : 0;
        const bool csr_ok = s0 == j0 && s1 == j0 + ne;  // the work range is the CSR range
        if (threadIdx.x == 0)
            grp_bad = 0;
        __syncthreads();  // grp staged
        if (ok && threadIdx.x == 0) {
            int bad = grp[0] != 0 || grp[MM] != ne;
            int32_t acc = 0;
            for (int m = 1; m <= MM; ++m) {
                const int32_t len = grp[m] - grp[m - 1];
                bad |= len < 0 || len % m != 0;
                grpRows[m] = len / m;
                acc += len / m;
            }
            bad |= acc > nrows;
            grp_bad = bad;
        }
        bool bad = ok ? tm_place(lane_addr, pc, vals, ne, q, warp >> 2, 8) : false;
        // The rows' staged positions, in flight during the sums: worker i
        // holds rows rb + 2 (i + k kW) + {0, 1}, k < kRP (rb = r0 rounded
        // down to even), their positions read two at a time and their
        // values stored two at a time where both rows are in the bucket and
        // the arrays allow; rows past 2 kRP kW of the bucket are read as they
        // are written.
        constexpr int kRP = 11;
        uint32_t rp[kRP];
        const int32_t rb = r0 & ~1;
        const bool pairs = (reinterpret_cast<uintptr_t>(a.g_rowPos) & 3u) == 0 &&
                           (reinterpret_cast<uintptr_t>(qG) & 15u) == 0;
        if (worker) {
#pragma unroll
            for (int k = 0; k < kRP; ++k) {
                const int32_t row = rb + 2 * (static_cast<int32_t>(threadIdx.x) + k * kW);
                const bool in0 = ok && row >= r0 && row < r1, in1 = ok && row + 1 >= r0 && row + 1 < r1;
                if (pairs && in0 && in1)
                    rp[k] = ld_u16x2(a.g_rowPos + row);
                else
                    rp[k] = (in0 ? static_cast<uint32_t>(ld_u16(a.g_rowPos + row)) : 0xFFFFu) |
                             ((in1 ? static_cast<uint32_t>(ld_u16(a.g_rowPos + row + 1)) : 0xFFFFu) << 16);
            }
        }
        tm_sync();  // placements landed, grpRows ready; TMEM is free
        if (!worker) {
            const int cn = c + step;
            int32_t jn, nn;
            if (cn < a.g_nbuckets && tm_bucket_range(a, cn, jn, nn))
                tm_load(lane_addr, pc, a.work + jn, a.g_pos + jn, nn, q, (warp - kTmWorkers) >> 2,
                        (32 - kTmWorkers) / 4);
        } else {
            const bool go = ok && grp_bad == 0 && csr_ok;
            if (go) {
                for (int m = 2; m <= MM; ++m)
                    group_sums(vals, grp[m - 1], m, grpRows[m], threadIdx.x, kW);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kW) : "memory");  // workers: sums done
            if (go) {
                // a row's value: its sum, +0.0 for an empty row (0xFFFF)
                auto value = [&](uint32_t p) {
                    double v = 0.0;
                    if (p != 0xFFFFu) {
                        if (p < static_cast<uint32_t>(ne))
                            v = plus_zero(vals[p]);
                        else
                            bad = true;
                    }
                    return v;
                };
#pragma unroll
                for (int k = 0; k < kRP; ++k) {
                    const int32_t row = rb + 2 * (static_cast<int32_t>(threadIdx.x) + k * kW);
                    const bool in0 = row >= r0 && row < r1, in1 = row + 1 >= r0 && row + 1 < r1;
                    const double v0 = in0 ? value(rp[k] & 0xFFFFu) : 0.0;
                    const double v1 = in1 ? value(rp[k] >> 16) : 0.0;
                    if (pairs && in0 && in1) {
                        st_pair(qG + row, v0, v1);
                    } else {
                        if (in0)
                            qG[row] = v0;
                        if (in1)
                            qG[row + 1] = v1;
                    }
                }
                // rows past the paired ones (a bucket of more than 2 kRP kW rows)
                for (int32_t row = rb + 2 * kRP * kW + static_cast<int32_t>(threadIdx.x); row < r1; row += kW)
                    if (row >= r0)
                        qG[row] = value(ld_u16(a.g_rowPos + row));
            }
            if (!go && threadIdx.x == 0)
                bad = true;
        }
        if (bad)
            flag(a.err);
        tm_sync();  // the next bucket is in TMEM; vals, grp are free
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(s_taddr),
                     "n"(kTmCols)
                     : "memory");
}

// ------------------------------------------- fused Z^T diag(d) Z (pass 2 + 1)
// One block per local range [u TL, (u+1) TL), which is at once scatter
// bucket u and gather tile u (the plan has s_bucket_len == g_tile_len and
// one block per cluster).  It places scatter bucket u's runs (read from
// `ws`) in shared memory -- that is q_L = Z x on the range, masked locals
// +0.0 --, multiplies by d_L (skipped for dL == nullptr: the identity local
// operator), and emits gather tile u's runs into `wg` directly, so q_L
// never reaches HBM.  A grid with fewer blocks than ranges loops over them.
__global__ void __launch_bounds__(kT, 1)
    fused_diag_kernel(PlanArgs a, const double *__restrict__ ws, const double *__restrict__ dL,
                      double *__restrict__ wg)
{
    extern __shared__ __align__(16) unsigned char smem[];
    double *vals = reinterpret_cast<double *>(smem);
    int64_t *runs = reinterpret_cast<int64_t *>(vals + a.g_tile_len);
    int32_t *runD = reinterpret_cast<int32_t *>(runs + a.g_nbuckets + 1);
    const int step = static_cast<int>(gridDim.x);
    for (int u = static_cast<int>(blockIdx.x); u < a.g_ntiles; u += step) {
        if (a.pf_next && pf_lane() && u + step < a.g_ntiles) {
            const int v = u + step;
            pf_scatter_bucket(a, v, ws);
            if (dL) {
                int64_t d0 = static_cast<int64_t>(v) * a.g_tile_len, d1 = d0 + a.g_tile_len;
                if (clamp_range(d0, d1, a.NL))
                    prefetch_l2(dL + d0, 8 * (d1 - d0));
            }
            int64_t s0 = a.g_tileSlot[v], s1 = a.g_tileSlot[v + 1];
            if (clamp_range(s0, s1, a.nnz))
                prefetch_l2(a.g_src + s0, 2 * (s1 - s0));
            prefetch_l2(a.g_runStart + static_cast<int64_t>(v) * a.g_nbuckets, 8ll * a.g_nbuckets);
        }
        const int64_t l0 = static_cast<int64_t>(u) * a.g_tile_len;
        const int32_t len = static_cast<int32_t>(a.NL - l0 < a.g_tile_len ? a.NL - l0 : a.g_tile_len);
        const int32_t j0 = a.s_runStart[u];
        const int32_t j1 = a.s_runStart[static_cast<int64_t>(a.s_ntiles) * a.s_nbuckets + u];
        if (a.pf_s2 && pf_lane()) {  // as in the scatter's pass 2: the range's later entries into L2
            int64_t p0 = j0 + 2048, p1 = j1;
            if (clamp_range(p0, p1, a.nnz)) {
                prefetch_l2(ws + p0, 8 * (p1 - p0));
                prefetch_l2(a.s_dst + p0, 2 * (p1 - p0));
            }
        }
        const int32_t s0 = a.g_tileSlot[u], s1 = a.g_tileSlot[u + 1];
        bool ok = len > 0 && j0 >= 0 && j1 >= j0 && j1 <= a.nnz && j1 - j0 <= len && s0 >= 0 &&
                  s1 >= s0 && s1 <= a.nnz && s1 - s0 <= len;
        if (!(ok && j1 - j0 == len))  // (no masked local: every slot is placed)
            for (int32_t i = threadIdx.x; i < len; i += kT)
                vals[i] = 0.0;
        const RunFetch rf = fetch_runs(a.g_runStart, u, a.g_nbuckets);
        __syncthreads();  // zeroed
        bool bad = false;
        if (ok) {
            stream_entries<6, true>(a.s_dst, ws, j0, j1, [&](uint32_t d, double v) {
                if (d < static_cast<uint32_t>(len))
                    vals[d] = v;
                else
                    bad = true;
            });
        }
        // (commit_runs begins with a barrier: the placements are complete after it)
        ok = commit_runs(rf, a.g_runStart, u, a.g_nbuckets, a.nnz, runs, runD) && ok &&
             run_off(runs[a.g_nbuckets]) == s1 - s0;
        if (ok && dL) {
            for (int32_t i0 = threadIdx.x; i0 < len; i0 += kU * kT) {
                double w[kU];
#pragma unroll
                for (int q = 0; q < kU; ++q)
                    w[q] = i0 + q * kT < len ? ld_seq(dL + l0 + i0 + q * kT) : 0.0;
#pragma unroll
                for (int q = 0; q < kU; ++q)
                    if (i0 + q * kT < len)
                        vals[i0 + q * kT] = mul_rn(w[q], vals[i0 + q * kT], a.mzero);
            }
        }
        __syncthreads();  // scaled tile ready
        if (ok) {
            if (emit_runs_lean<kGatherEmitSteps>(runs, runD, a.g_nbuckets, 0, s1 - s0, a.g_src, s0, vals, len,
                                                 wg, a.nnz))
                bad = true;
        }
        if (bad || (!ok && threadIdx.x == 0))
            flag(a.err);
        __syncthreads();  // vals and the run tables are rewritten next
    }
}

int64_t smem_s1(const bs_plan_dev *p) { return 8ll * p->s_tile_rows + 8ll * (p->s_nbuckets + 1) + 4ll * p->s_nbuckets; }
int64_t smem_s2(const bs_plan_dev *p) { return 8ll * p->s_bucket_len; }
int64_t smem_g1(const bs_plan_dev *p) { return 8ll * p->g_tile_len + 8ll * (p->g_nbuckets + 1) + 4ll * p->g_nbuckets; }
int64_t smem_g2(const bs_plan_dev *p) { return 8ll * p->g_bucket_entries_max + 4ll * (kMaxRow + 1); }

constexpr int64_t kSmemMax = 232448;

// Launches `kernel` over `items` tiles or buckets: one cluster of `cs`
// blocks per item, or, with the context's persistent setting, at most one
// cluster per `cs` SMs, each looping over its items.
template <class... KArgs, class... Args>
int launch(bs_ctx *ctx, const char *name, void (*kernel)(KArgs...), int cs, int64_t items,
           int64_t smem, cudaStream_t s, Args... args)
{
    int64_t clusters = items;
    if (ctx->tune.persist) {
        const int64_t cap = ctx->sms / cs > 0 ? ctx->sms / cs : 1;
        clusters = items < cap ? items : cap;
    }
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess)
        return bs_set_error(ctx, BS_ECUDA, "%s: cudaFuncSetAttribute: %s", name,
                            cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs), 1, 1);
    cfg.blockDim = dim3(kT, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cs > 1 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess)
        return bs_set_error(ctx, BS_ECUDA, "launch of %s: %s", name, cudaGetErrorString(e));
    return BS_OK;
}

int check_plan(bs_ctx *ctx, const char *name, const bs_gs_dev *t, const void *qL, const void *qG)
{
    const bs_plan_dev *p = t->plan;
    if (!t->rowStarts)
        return bs_set_error(ctx, BS_EINVAL, "%s: the plan needs rowStarts", name);
    if (p->cluster != 1 && p->cluster != 2 && p->cluster != 4)
        return bs_set_error(ctx, BS_EINVAL, "%s: plan cluster size must be 1, 2 or 4", name);
    if (p->s_ntiles < 1 || p->s_nbuckets < 1 || p->s_tile_rows < 1 || p->s_bucket_len < 1 ||
        p->g_ntiles < 1 || p->g_nbuckets < 1 || p->g_tile_len < 1 || p->g_bucket_entries_max < 1 ||
        p->g_bucket_rows_max < 1)
        return bs_set_error(ctx, BS_EINVAL, "%s: bad plan sizes", name);
    const int64_t cs = p->cluster;
    if (cs * p->s_tile_rows > 32768 || cs * p->s_bucket_len > 65536 ||
        cs * p->g_tile_len > 32768 || cs * p->g_bucket_entries_max > 65535)
        return bs_set_error(ctx, BS_EINVAL, "%s: plan offsets exceed their 15 or 16 bits", name);
    if (cs * p->s_nbuckets * p->s_bucket_len < t->NL || cs * p->g_ntiles * p->g_tile_len < t->NL ||
        cs * p->s_ntiles * p->s_tile_rows < t->NG)
        return bs_set_error(ctx, BS_EINVAL, "%s: plan does not cover the mesh", name);
    if (smem_s1(p) > kSmemMax || smem_s2(p) > kSmemMax || smem_g1(p) > kSmemMax ||
        smem_g2(p) > kSmemMax)
        return bs_set_error(ctx, BS_EINVAL, "%s: plan needs too much shared memory", name);
    if (p->g_mmax < 1 || p->g_mmax > kMaxRow)
        return bs_set_error(ctx, BS_EINVAL, "%s: plan row length bound outside [1, %d]", name,
                            kMaxRow);
    if (!p->s_tileRows || !p->s_runStart || !p->g_subRows || !p->g_tileSlot ||
        !p->g_runStart || !p->work || !p->g_groupStart || !p->g_rowPos ||
        (t->nnz > 0 && (!p->s_src || !p->s_dst || !p->g_src || !p->g_pos)))
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
    a.g_mmax = p->g_mmax;
    a.rowStarts = t->rowStarts;
    a.s_tileRows = p->s_tileRows;
    a.s_runStart = p->s_runStart;
    a.s_src = p->s_src;
    a.s_dst = p->s_dst;
    a.g_subRows = p->g_subRows;
    a.g_tileSlot = p->g_tileSlot;
    a.g_runStart = p->g_runStart;
    a.g_src = p->g_src;
    a.g_pos = p->g_pos;
    a.g_groupStart = p->g_groupStart;
    a.g_rowPos = p->g_rowPos;
    a.work = p->work;
    a.err = ctx->dev_err;
    a.pf_next = ctx->tune.persist && ctx->tune.l2_prefetch;
    a.mzero = -0.0;
    // only where the work array is well beyond L2: measured -7 us per stress
    // scatter (453 MB of work entries), +1.5 us on a 134 MB one
    a.pf_s2 = 8 * t->nnz > 2ll * ctx->l2_bytes;
    return a;
}

template <int CS>
int scatter_cs(bs_ctx *ctx, const PlanArgs &a, const bs_plan_dev *p, const double *qG, double *qL,
               cudaStream_t s)
{
    if (int st = launch(ctx, "scatter_tile_kernel", scatter_tile_kernel<CS>, CS, p->s_ntiles,
                        smem_s1(p), s, a, qG))
        return st;
    return launch(ctx, "scatter_bucket_kernel", scatter_bucket_kernel<CS>, CS, p->s_nbuckets,
                  smem_s2(p), s, a, qL);
}

// TMEM column where the staged positions start (values take 16 columns per
// group of 1024 entries, positions 4), or -1 if a bucket does not fit.
int tm_pos_col(const bs_plan_dev *p)
{
    const int64_t ng = (p->g_bucket_entries_max + kTmGroupEntries - 1) / kTmGroupEntries;
    return 20 * ng <= kTmCols ? static_cast<int>(16 * ng) : -1;
}

// Gather pass 2: the TMEM-buffered persistent kernel (cluster 1, a bucket
// that fits TMEM, the context's setting), else one block per bucket.
template <int CS>
int gather_pass2(bs_ctx *ctx, const PlanArgs &a, const bs_plan_dev *p, double *qG, cudaStream_t s)
{
    const int pc = tm_pos_col(p);
    if (CS == 1 && ctx->tune.tmem && pc >= 0) {
        // 20 summing/writing warps and 12 loading ones: measured fastest of
        // 16/16 (the loads hide, the sums and writes slow), 20/12, 24/8 (the
        // loads outlast the sums and writes)
        void (*k)(PlanArgs, double *, int) = gather_bucket_tm_kernel<kTmWorkersDefault>;
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem_g2(p)));
        if (e != cudaSuccess)
            return bs_set_error(ctx, BS_ECUDA, "gather_bucket_tm_kernel: cudaFuncSetAttribute: %s",
                                cudaGetErrorString(e));
        const int grid = p->g_nbuckets < ctx->sms ? p->g_nbuckets : ctx->sms;
        k<<<grid, kT, static_cast<size_t>(smem_g2(p)), s>>>(a, qG, pc);
        BS_LAUNCH_CHECK(ctx, "gather_bucket_tm_kernel");
        return BS_OK;
    }
    return launch(ctx, "gather_bucket_kernel", gather_bucket_kernel<CS>, CS, p->g_nbuckets,
                  smem_g2(p), s, a, qG);
}

template <int CS>
int gather_cs(bs_ctx *ctx, const PlanArgs &a, const bs_plan_dev *p, const double *qL, double *qG,
              cudaStream_t s)
{
    if (int st = launch(ctx, "gather_tile_kernel", gather_tile_kernel<CS>, CS, p->g_ntiles,
                        smem_g1(p), s, a, qL))
        return st;
    return gather_pass2<CS>(ctx, a, p, qG, s);
}

} // namespace

int bs_scatter_planned(bs_ctx *ctx, const bs_gs_dev *t, const double *qG, double *qL,
                       cudaStream_t s)
{
    if (int st = check_plan(ctx, "bs_scatter", t, qL, qG))
        return st;
    const bs_plan_dev *p = t->plan;
    const PlanArgs a = make_args(ctx, t);
    switch (p->cluster) {
    case 1: return scatter_cs<1>(ctx, a, p, qG, qL, s);
    case 2: return scatter_cs<2>(ctx, a, p, qG, qL, s);
    default: return scatter_cs<4>(ctx, a, p, qG, qL, s);
    }
}

int bs_gather_planned(bs_ctx *ctx, const bs_gs_dev *t, const double *qL, double *qG,
                      cudaStream_t s)
{
    if (int st = check_plan(ctx, "bs_gather", t, qL, qG))
        return st;
    const bs_plan_dev *p = t->plan;
    const PlanArgs a = make_args(ctx, t);
    switch (p->cluster) {
    case 1: return gather_cs<1>(ctx, a, p, qL, qG, s);
    case 2: return gather_cs<2>(ctx, a, p, qL, qG, s);
    default: return gather_cs<4>(ctx, a, p, qL, qG, s);
    }
}

int bs_apply_diag_planned(bs_ctx *ctx, const bs_gs_dev *t, const double *xG, const double *dL,
                          double *yG, cudaStream_t s)
{
    if (int st = check_plan(ctx, "bs_apply_diag", t, dL, xG))
        return st;
    const bs_plan_dev *p = t->plan;
    if (p->cluster != 1 || p->s_bucket_len != p->g_tile_len || p->s_nbuckets != p->g_ntiles)
        return bs_set_error(ctx, BS_EINVAL,
                            "bs_apply_diag: the plan needs cluster 1 and scatter buckets equal to "
                            "gather tiles (s_bucket_len == g_tile_len)");
    if (p->work_len < 2 * t->nnz)
        return bs_set_error(ctx, BS_EINVAL, "bs_apply_diag: work buffer shorter than 2 nnz");
    if (bs_overlap(p->work, 8 * p->work_len, dL, 8 * t->NL) ||
        bs_overlap(p->work, 8 * p->work_len, yG, 8 * t->NG))
        return bs_set_error(ctx, BS_EINVAL, "bs_apply_diag: work buffer overlaps dL or yG");
    PlanArgs a = make_args(ctx, t);
    double *ws = p->work, *wg = p->work + t->nnz;
    if (int st = launch(ctx, "scatter_tile_kernel", scatter_tile_kernel<1>, 1, p->s_ntiles,
                        smem_s1(p), s, a, xG))
        return st;
    if (int st = launch(ctx, "fused_diag_kernel", fused_diag_kernel, 1, p->g_ntiles, smem_g1(p), s,
                        a, static_cast<const double *>(ws), dL, wg))
        return st;
    a.work = wg;
    return gather_pass2<1>(ctx, a, p, yG, s);
}
