// bs_vec.cu -- BS1-BS5: copy, AXPY, norm, inner product, fused CG update.
//
// "Portable high-order finite element kernels I: Streaming Operations",
// Benchmark Streaming test list and the CG vector operations.  All five are
// HBM streams with at most three fused multiply-adds per element, so the
// kernels are built for bytes in flight, not arithmetic:
//
//  * persistent grid of (SMs x blocks-per-SM) blocks of 256 threads, grid
//    stride over 32-byte vectors (ld/st.global.v4.f64, sm_100+), UNROLL
//    independent vectors per operand in flight per thread;
//  * loads skip L1 (L1::no_allocate) and ask L2 for 256-byte prefetch;
//    stores are streaming (.cs: evict first), so a kernel's written lines
//    leave L2 while it runs instead of during the next kernel;
//  * a misaligned head (< 4 elements) and the ragged tail are done by the
//    first threads of the grid with scalar accesses;
//  * reductions (BS3-BS5) are one launch: each block reduces its threads'
//    fixed element sets by warp shuffles and a shared-memory step, writes
//    one partial, and the last block to finish (completion counter, no
//    waiting) sums the partials in a fixed tree.  The element -> thread
//    map depends only on (grid, n, alignment), so results are bitwise
//    reproducible run to run.  The pages' version is two kernels (a partial
//    reduction to Nblocks values, then a second reduction) with a shuffle
//    finish of the last warp.
#include <cuda_runtime.h>


#include "bs_internal.h"

namespace {

constexpr int kThreads = 256;

template <int V>
struct Vec {
    double v[V];
};

template <int V>
__device__ __forceinline__ Vec<V> ld_stream(const double *p);

template <>
__device__ __forceinline__ Vec<4> ld_stream<4>(const double *p)
{
    Vec<4> r;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.f64 {%0,%1,%2,%3}, [%4];"
                 : "=d"(r.v[0]), "=d"(r.v[1]), "=d"(r.v[2]), "=d"(r.v[3])
                 : "l"(p));
    return r;
}

template <>
__device__ __forceinline__ Vec<2> ld_stream<2>(const double *p)
{
    Vec<2> r;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v2.f64 {%0,%1}, [%2];"
                 : "=d"(r.v[0]), "=d"(r.v[1])
                 : "l"(p));
    return r;
}

template <>
__device__ __forceinline__ Vec<1> ld_stream<1>(const double *p)
{
    Vec<1> r;
    asm volatile("ld.global.L1::no_allocate.L2::256B.f64 %0, [%1];" : "=d"(r.v[0]) : "l"(p));
    return r;
}

template <int V>
__device__ __forceinline__ void st_stream(double *p, const Vec<V> &r);

template <>
__device__ __forceinline__ void st_stream<4>(double *p, const Vec<4> &r)
{
    asm volatile("st.global.cs.v4.f64 [%0], {%1,%2,%3,%4};" ::"l"(p), "d"(r.v[0]),
                 "d"(r.v[1]), "d"(r.v[2]), "d"(r.v[3])
                 : "memory");
}

template <>
__device__ __forceinline__ void st_stream<2>(double *p, const Vec<2> &r)
{
    asm volatile("st.global.cs.v2.f64 [%0], {%1,%2};" ::"l"(p), "d"(r.v[0]),
                 "d"(r.v[1])
                 : "memory");
}

template <>
__device__ __forceinline__ void st_stream<1>(double *p, const Vec<1> &r)
{
    asm volatile("st.global.cs.f64 [%0], %1;" ::"l"(p), "d"(r.v[0]) : "memory");
}

// Elements [0, h) and [h + nv V, h + nv V + t) are scalars; element index
// of scalar slot k (k < h + t).
__device__ __forceinline__ int64_t scalar_index(int64_t k, int64_t h, int64_t nv, int V)
{
    return k < h ? k : h + nv * V + (k - h);
}

struct RedOut {
    double *partials;
    unsigned int *counter;
    double *out;
};

__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide sum; the result is valid in thread 0.  Fixed order.
__device__ __forceinline__ double block_sum(double v, double *sh)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0)
        sh[w] = v;
    __syncthreads();
    if (w == 0) {
        v = lane < kThreads / 32 ? sh[lane] : 0.0;
        v = warp_sum(v);
    }
    return v;
}

// Writes this block's partial; the last block to arrive sums all partials
// in index order and writes the result, then re-arms the counter.  A grid
// of one block writes its sum directly (as 0.0 + sum: the same bits the
// finisher's sum from +0.0 gives), saving the fence, the counter round trip
// and the second block sum -- the launch-latency floor of small reductions.
__device__ __forceinline__ void finish_reduction(double v, const RedOut &o)
{
    __shared__ double sh[kThreads / 32];
    __shared__ unsigned int ticket;
    v = block_sum(v, sh);
    if (gridDim.x == 1) {
        if (threadIdx.x == 0)
            *o.out = 0.0 + v;
        return;
    }
    if (threadIdx.x == 0) {
        o.partials[blockIdx.x] = v;
        __threadfence();
        ticket = atomicAdd(o.counter, 1u);
    }
    __syncthreads();
    if (ticket != gridDim.x - 1)
        return;
    __threadfence();
    double s = 0.0;
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += kThreads)
        s += __ldcg(o.partials + i);
    s = block_sum(s, sh);
    if (threadIdx.x == 0) {
        *o.out = s;
        *o.counter = 0u;
    }
}

// ------------------------------------------- sums of squares off the FP64 pipe
// GB300 runs binary64 fma/add at ~1.6 per clock per SM, so a sum of
// squares with one fma per element is bound by the FP64 pipe below HBM
// speed.  SqAcc forms x^2 and sums it on the FP32 and integer pipes:
//   |x| = xh + xl + dx with xh the leading 24 significant bits (a float,
//   exact), xl the next 23 bits and dx the last 6 bits, dropped:
//   0 <= dx < 2^-46 |x|; 2 xl is formed exactly as the float difference
//   2^k (1 + f) - 2^k (Sterbenz) from integer operations only (on this
//   part int<->float conversions are as scarce as FP64 math);
//   x^2 ~= xh^2 + 2 xh xl, xh^2 exact as p + e (TwoProduct by fmaf), q =
//   fma(xh, 2 xl, e) rounded once; p is added to a float-float sum (s, c)
//   by Fast2Sum with the larger of s, p first (both are >= 0: exact), q
//   and the addition's error to c.  Every chunk of at most 8 elements is
//   flushed: (s, c) move into a binary64 total through an exact
//   float->double conversion on the integer pipe.
// Worst case, for a chunk with exact sum S of squares (all terms >= 0):
//   dropped bits dx and the left-out xl^2: x^2 underestimated by
//   <= 2^-45 x^2 + 2^-46 x^2; q's rounding: <= 2^-24 * 1.25 * 2^-22 x^2;
//   c: every term t_j = err_j + q_j has |err_j| <= 2^-24 S and
//   sum |q_j| <= 1.25 * 2^-22 S, so |c| <= (k 2^-24 + 1.25 * 2^-22) S =
//   3.25 * 2^-22 S for k = 8, and its k + k float roundings add
//   <= 2^-24 (1 + k) * 3.25 * 2^-22 S = 29.25 * 2^-46 S;
//   in all < 2.1 * 2^-45 S + 29.25 * 2^-46 S < 4.8e-13 S, plus the binary64
//   flushes and the fixed reduction tree (2^-53 per addition).  So the
//   total is within 5e-13 relative of the exact sum of squares.  |x|
//   outside [2^-40, 2^41) (subnormal, tiny, huge, inf, NaN) goes through a
//   separate binary64 fma sum instead.
constexpr uint32_t kSqExpLo = 1023 - 40, kSqExpHi = 1023 + 40;

__device__ __forceinline__ double float_to_double_exact(float f)
{
    const uint32_t b = __float_as_uint(f);
    const uint32_t mag = b & 0x7FFFFFFFu;
    if ((mag >> 23) == 0)  // zero or subnormal: far below the running sum
        return 0.0;
    const uint32_t hi = (b & 0x80000000u) | ((mag >> 3) + ((1023u - 127u) << 20));
    return __hiloint2double(static_cast<int>(hi), static_cast<int>(mag << 29));
}

struct SqAcc {
    float s, c;   // float-float partial sum of the current chunk
    double d;     // flushed chunks
    double slow;  // out-of-range terms

    __device__ __forceinline__ void init()
    {
        s = 0.f;
        c = 0.f;
        d = 0.0;
        slow = 0.0;
    }

    // Adds x^2 if |x| is in the fast range or x is 0; otherwise only marks
    // the lane (`pending`): the caller re-walks its elements with add_slow
    // afterwards.  No binary64 math on this path -- an issued fma holds the
    // FP64 pipe for the whole warp even when predicated off.
    __device__ __forceinline__ void add(double x, bool &pending)
    {
        const uint32_t hw = static_cast<uint32_t>(__double2hiint(x)) & 0x7FFFFFFFu;
        const uint32_t lw = static_cast<uint32_t>(__double2loint(x));
        const uint32_t E = hw >> 20;
        const bool fast = E - kSqExpLo <= kSqExpHi - kSqExpLo;
        pending |= !fast && (hw | lw) != 0;
        if (fast) {
            const uint32_t t = hw - ((1023u - 127u) << 20);
            const float xh = __uint_as_float(__funnelshift_l(lw, t, 3));
            // 2 xl: bits 6..28 of the fraction as the mantissa f of a float
            // 2^k (1 + f), minus 2^k, k = e - 22 (e: x's exponent); exact
            const uint32_t one = (E - (1023u + 22u - 127u)) << 23;
            const float xl2 = __fsub_rn(__uint_as_float(one | ((lw & 0x1FFFFFFFu) >> 6)),
                                        __uint_as_float(one));
            const float p = __fmul_rn(xh, xh);
            float q = __fmaf_rn(xh, xh, -p);  // exact: xh^2 = p + q
            q = __fmaf_rn(xh, xl2, q);        // + 2 xh xl
            const float a = fmaxf(s, p), b = fminf(s, p);
            const float sn = __fadd_rn(a, b);
            const float err = __fsub_rn(b, __fsub_rn(sn, a));  // exact (a >= b >= 0)
            s = sn;
            c = __fadd_rn(c, __fadd_rn(err, q));
        }
    }

    // The second walk: x^2 of the out-of-range values only, in binary64.
    __device__ __forceinline__ void add_slow(double x)
    {
        const uint32_t hw = static_cast<uint32_t>(__double2hiint(x)) & 0x7FFFFFFFu;
        const uint32_t lw = static_cast<uint32_t>(__double2loint(x));
        const uint32_t E = hw >> 20;
        if (!(E - kSqExpLo <= kSqExpHi - kSqExpLo) && (hw | lw) != 0)
            slow = __fma_rn(x, x, slow);
    }

    __device__ __forceinline__ void flush()
    {
        d = __dadd_rn(d, float_to_double_exact(s));
        d = __dadd_rn(d, float_to_double_exact(c));
        s = 0.f;
        c = 0.f;
    }

    __device__ __forceinline__ double total()
    {
        flush();
        return __dadd_rn(d, slow);
    }
};

// ---------------------------------------------------------------- BS1 copy
template <int V, int UNROLL>
__global__ void __launch_bounds__(kThreads) copy_kernel(const double *__restrict__ x,
                                                        double *__restrict__ y, int64_t h,
                                                        int64_t nv, int64_t t)
{
    const int64_t gid = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const double *xv = x + h;
    double *yv = y + h;
    for (int64_t b = gid; b < nv; b += stride * UNROLL) {
        Vec<V> r[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < nv)
                r[u] = ld_stream<V>(xv + (b + u * stride) * V);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < nv)
                st_stream<V>(yv + (b + u * stride) * V, r[u]);
    }
    if (gid < h + t) {
        const int64_t i = scalar_index(gid, h, nv, V);
        y[i] = x[i];
    }
}

// num / den, or 0 where den is 0: a device-side CG coefficient (rr / pAp or
// rr_new / rr) whose denominator vanishes only once the iteration has met
// an exact solution, where a zero step keeps it.
__device__ __forceinline__ double dev_quotient(const double *num, const double *den)
{
    const double d = den[0];
    return d != 0.0 ? __ddiv_rn(num[0], d) : 0.0;
}

// ---------------------------------------------------------------- BS2 AXPY
// beta = beta_num[0] / beta_den[0] (dev_quotient) when beta_num is given.
template <int V, int UNROLL, bool BETA1>
__global__ void __launch_bounds__(kThreads) axpy_kernel(double alpha, const double *x, double beta,
                                                        double *y, int64_t h, int64_t nv,
                                                        int64_t t, const double *beta_num,
                                                        const double *beta_den, double mzero)
{
    if (!BETA1 && beta_num) {
        __shared__ double s_beta;
        if (threadIdx.x == 0)
            s_beta = dev_quotient(beta_num, beta_den);
        __syncthreads();
        beta = s_beta;
    }
    const int64_t gid = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const double *xv = x + h;
    double *yv = y + h;
    for (int64_t b = gid; b < nv; b += stride * UNROLL) {
        Vec<V> a[UNROLL], c[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < nv) {
                a[u] = ld_stream<V>(xv + (b + u * stride) * V);
                c[u] = ld_stream<V>(yv + (b + u * stride) * V);
            }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < nv) {
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const double by = BETA1 ? c[u].v[k] : mul_rn(beta, c[u].v[k], mzero);
                    c[u].v[k] = __fma_rn(alpha, a[u].v[k], by);
                }
                st_stream<V>(yv + (b + u * stride) * V, c[u]);
            }
    }
    if (gid < h + t) {
        const int64_t i = scalar_index(gid, h, nv, V);
        const double by = BETA1 ? y[i] : mul_rn(beta, y[i], mzero);
        y[i] = __fma_rn(alpha, x[i], by);
    }
}

// ----------------------------------------------------- BS3 norm, BS4 dot
// DOT == false: sum x_i^2 (y unused).  DOT == true: sum x_i y_i.
template <int V, int UNROLL, bool DOT>
__global__ void __launch_bounds__(kThreads) dot_kernel(const double *__restrict__ x,
                                                       const double *__restrict__ y, int64_t h,
                                                       int64_t nv, int64_t t, RedOut o)
{
    const int64_t gid = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const double *xv = x + h;
    const double *yv = y + h;
    double acc[V];
    SqAcc sq;
    bool pending = false;
#pragma unroll
    for (int k = 0; k < V; ++k)
        acc[k] = 0.0;
    sq.init();
    for (int64_t b = gid; b < nv; b += stride * UNROLL) {
        Vec<V> a[UNROLL], c[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < nv) {
                a[u] = ld_stream<V>(xv + (b + u * stride) * V);
                if (DOT)
                    c[u] = ld_stream<V>(yv + (b + u * stride) * V);
            }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (b + u * stride < nv) {
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    if (DOT)
                        acc[k] = __fma_rn(a[u].v[k], c[u].v[k], acc[k]);
                    else
                        sq.add(a[u].v[k], pending);
                }
            }
            // chunks of at most 8 squares (the accumulator's error bound)
            if (!DOT && ((u + 1) * V) % 8 == 0)
                sq.flush();
        }
        if (!DOT && (UNROLL * V) % 8 != 0)
            sq.flush();
    }
    if (gid < h + t) {
        const int64_t i = scalar_index(gid, h, nv, V);
        if (DOT)
            acc[0] = __fma_rn(x[i], y[i], acc[0]);
        else
            sq.add(x[i], pending);
    }
    if (!DOT && pending) {  // this thread met values outside the fast range
        for (int64_t b = gid; b < nv; b += stride)
            for (int k = 0; k < V; ++k)
                sq.add_slow(xv[b * V + k]);
        if (gid < h + t)
            sq.add_slow(x[scalar_index(gid, h, nv, V)]);
    }
    double s;
    if (DOT) {
        s = acc[0];
#pragma unroll
        for (int k = 1; k < V; ++k)
            s += acc[k];
    } else {
        s = sq.total();
    }
    finish_reduction(s, o);
}

// ------------------------------------------------------ BS5 fused CG update
template <int V, int UNROLL, bool RED>
__global__ void __launch_bounds__(kThreads)
    cg_kernel(const double *__restrict__ alpha_num, const double *__restrict__ alpha_den,
              double alpha_host, const double *__restrict__ p, const double *__restrict__ Ap,
              double *__restrict__ x, double *__restrict__ r, int64_t h, int64_t nv, int64_t t,
              RedOut o)
{
    __shared__ double s_alpha;
    double alpha = alpha_host;
    if (alpha_num) {
        if (threadIdx.x == 0)
            s_alpha = dev_quotient(alpha_num, alpha_den);
        __syncthreads();
        alpha = s_alpha;
    }
    const double nalpha = -alpha;
    const int64_t gid = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    SqAcc sq;
    sq.init();
    bool pending = false;
    int chunk = 0;
    for (int64_t b = gid; b < nv; b += stride * UNROLL) {
        Vec<V> vp[UNROLL], va[UNROLL], vx[UNROLL], vr[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < nv) {
                const int64_t e = h + (b + u * stride) * V;
                vp[u] = ld_stream<V>(p + e);
                va[u] = ld_stream<V>(Ap + e);
                vx[u] = ld_stream<V>(x + e);
                vr[u] = ld_stream<V>(r + e);
            }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            if (b + u * stride < nv) {
                const int64_t e = h + (b + u * stride) * V;
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    vx[u].v[k] = __fma_rn(alpha, vp[u].v[k], vx[u].v[k]);
                    vr[u].v[k] = __fma_rn(nalpha, va[u].v[k], vr[u].v[k]);
                    if (RED)
                        sq.add(vr[u].v[k], pending);
                }
                st_stream<V>(x + e, vx[u]);
                st_stream<V>(r + e, vr[u]);
            }
        // flush the float-float chunk every 8 elements
        if (RED && (chunk += UNROLL * V) >= 8) {
            sq.flush();
            chunk = 0;
        }
    }
    if (gid < h + t) {
        const int64_t i = scalar_index(gid, h, nv, V);
        x[i] = __fma_rn(alpha, p[i], x[i]);
        const double ri = __fma_rn(nalpha, Ap[i], r[i]);
        r[i] = ri;
        if (RED)
            sq.add(ri, pending);
    }
    if (RED) {
        if (pending) {  // re-walk this thread's updated r for out-of-range values
            for (int64_t b = gid; b < nv; b += stride)
                for (int k = 0; k < V; ++k)
                    sq.add_slow(r[h + b * V + k]);
            if (gid < h + t)
                sq.add_slow(r[scalar_index(gid, h, nv, V)]);
        }
        finish_reduction(sq.total(), o);
    }
}

// ------------------------------------------------------------- host side

// How a length-n operation over the given operands is split into a scalar
// head, 8V-byte vectors and a scalar tail.
struct Plan {
    int V;
    int64_t h, nv, t;
};

Plan make_plan(int64_t n, int vmax, const void *const *ptrs, int np)
{
    for (int V = vmax; V >= 2; V >>= 1) {
        const uintptr_t bytes = 8u * V;
        const uintptr_t m0 = reinterpret_cast<uintptr_t>(ptrs[0]) % bytes;
        bool same = true;
        for (int i = 1; i < np; ++i)
            same = same && reinterpret_cast<uintptr_t>(ptrs[i]) % bytes == m0;
        if (!same)
            continue;
        int64_t h = static_cast<int64_t>((bytes - m0) % bytes) / 8;
        if (h > n)
            h = n;
        const int64_t nv = (n - h) / V;
        return Plan{V, h, nv, n - h - nv * V};
    }
    return Plan{1, 0, n, 0};
}

bool aligned8(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 7u) == 0;
}

int grid_for(const bs_ctx *ctx, int blocks_per_sm, int64_t work_items, int cap)
{
    int64_t g = static_cast<int64_t>(ctx->sms) * blocks_per_sm;
    const int64_t need = (work_items + kThreads - 1) / kThreads;
    if (need < g)
        g = need;
    if (g > cap)
        g = cap;
    return g < 1 ? 1 : static_cast<int>(g);
}

constexpr int kStreamUnroll = 2;
constexpr int kReduceUnroll = 2;
constexpr int kNormUnroll = 4;  // the norm computes ~25 instructions per element
constexpr int kCgUnroll = 1;

template <int V>
void launch_copy(int grid, cudaStream_t s, const double *x, double *y, const Plan &pl)
{
    copy_kernel<V, kStreamUnroll><<<grid, kThreads, 0, s>>>(x, y, pl.h, pl.nv, pl.t);
}

template <int V>
void launch_axpy(int grid, cudaStream_t s, double a, const double *x, double b, double *y,
                 const Plan &pl, const double *bnum, const double *bden)
{
    if (b == 1.0 && !bnum)
        axpy_kernel<V, kStreamUnroll, true><<<grid, kThreads, 0, s>>>(a, x, b, y, pl.h, pl.nv, pl.t,
                                                                      nullptr, nullptr, -0.0);
    else
        axpy_kernel<V, kStreamUnroll, false><<<grid, kThreads, 0, s>>>(a, x, b, y, pl.h, pl.nv,
                                                                       pl.t, bnum, bden, -0.0);
}

template <int V, bool DOT>
void launch_dot(int grid, cudaStream_t s, const double *x, const double *y, const Plan &pl,
                const RedOut &o)
{
    dot_kernel<V, DOT ? kReduceUnroll : kNormUnroll, DOT><<<grid, kThreads, 0, s>>>(
        x, y, pl.h, pl.nv, pl.t, o);
}

template <int V>
void launch_cg(int grid, cudaStream_t s, const double *num, const double *den, double alpha,
               const double *p, const double *Ap, double *x, double *r, const Plan &pl,
               const RedOut &o, bool red)
{
    if (red)
        cg_kernel<V, kCgUnroll, true><<<grid, kThreads, 0, s>>>(num, den, alpha, p, Ap, x, r, pl.h,
                                                                pl.nv, pl.t, o);
    else
        cg_kernel<V, kCgUnroll, false><<<grid, kThreads, 0, s>>>(num, den, alpha, p, Ap, x, r,
                                                                 pl.h, pl.nv, pl.t, o);
}

int reduce_grid(const bs_ctx *ctx, const Plan &pl, int unroll)
{
    return grid_for(ctx, ctx->tune.reduce_blocks_per_sm, (pl.nv + unroll - 1) / unroll,
                    kMaxReduceBlocks);
}

} // namespace

extern "C" int bs_copy(bs_ctx *ctx, int64_t n, const double *x, double *y, void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (n < 0 || (n > 0 && (!x || !y)))
        return bs_set_error(ctx, BS_EINVAL, "bs_copy: bad length or NULL pointer");
    if (n == 0)
        return BS_OK;
    if (!aligned8(x) || !aligned8(y))
        return bs_set_error(ctx, BS_EINVAL, "bs_copy: pointers must be 8-byte aligned");
    if (x != y && bs_overlap(x, 8 * n, y, 8 * n))
        return bs_set_error(ctx, BS_EINVAL, "bs_copy: x and y overlap");
    if (int st = bs_check_device(ctx))
        return st;
    if (x == y)
        return BS_OK;
    const void *ps[2] = {x, y};
    const Plan pl = make_plan(n, ctx->tune.vec_width, ps, 2);
    const int grid = grid_for(ctx, ctx->tune.stream_blocks_per_sm, (pl.nv + 1) / 2, 1 << 30);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (pl.V) {
    case 4: launch_copy<4>(grid, s, x, y, pl); break;
    case 2: launch_copy<2>(grid, s, x, y, pl); break;
    default: launch_copy<1>(grid, s, x, y, pl); break;
    }
    BS_LAUNCH_CHECK(ctx, "copy_kernel");
    return BS_OK;
}

static int axpy_common(bs_ctx *ctx, const char *name, int64_t n, double alpha, const double *x,
                       double beta, const double *bnum, const double *bden, double *y,
                       void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (n < 0 || (n > 0 && (!x || !y)))
        return bs_set_error(ctx, BS_EINVAL, "%s: bad length or NULL pointer", name);
    if (n == 0)
        return BS_OK;
    if (!aligned8(x) || !aligned8(y) || (bnum && (!aligned8(bnum) || !aligned8(bden))))
        return bs_set_error(ctx, BS_EINVAL, "%s: pointers must be 8-byte aligned", name);
    if (x != y && bs_overlap(x, 8 * n, y, 8 * n))
        return bs_set_error(ctx, BS_EINVAL, "%s: x and y overlap", name);
    if (bnum && (bs_overlap(bnum, 8, y, 8 * n) || bs_overlap(bden, 8, y, 8 * n)))
        return bs_set_error(ctx, BS_EINVAL, "%s: beta scalars overlap y", name);
    if (int st = bs_check_device(ctx))
        return st;
    const void *ps[2] = {x, y};
    const Plan pl = make_plan(n, ctx->tune.vec_width, ps, 2);
    const int grid = grid_for(ctx, ctx->tune.stream_blocks_per_sm, (pl.nv + 1) / 2, 1 << 30);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (pl.V) {
    case 4: launch_axpy<4>(grid, s, alpha, x, beta, y, pl, bnum, bden); break;
    case 2: launch_axpy<2>(grid, s, alpha, x, beta, y, pl, bnum, bden); break;
    default: launch_axpy<1>(grid, s, alpha, x, beta, y, pl, bnum, bden); break;
    }
    BS_LAUNCH_CHECK(ctx, "axpy_kernel");
    return BS_OK;
}

extern "C" int bs_axpy(bs_ctx *ctx, int64_t n, double alpha, const double *x, double beta,
                       double *y, void *stream)
{
    return axpy_common(ctx, "bs_axpy", n, alpha, x, beta, nullptr, nullptr, y, stream);
}

extern "C" int bs_axpy_dev(bs_ctx *ctx, int64_t n, double alpha, const double *x,
                           const double *beta_num_dev, const double *beta_den_dev, double *y,
                           void *stream)
{
    if (ctx && (!beta_num_dev || !beta_den_dev))
        return bs_set_error(ctx, BS_EINVAL, "bs_axpy_dev: NULL beta scalar");
    return axpy_common(ctx, "bs_axpy_dev", n, alpha, x, 0.0, beta_num_dev, beta_den_dev, y,
                       stream);
}

static int dot_common(bs_ctx *ctx, const char *name, int64_t n, const double *x, const double *y,
                      double *out, void *stream, bool dot)
{
    if (!ctx)
        return BS_EINVAL;
    if (n < 0 || !out || (n > 0 && (!x || (dot && !y))))
        return bs_set_error(ctx, BS_EINVAL, "%s: bad length or NULL pointer", name);
    if (!aligned8(out) || (n > 0 && (!aligned8(x) || (dot && !aligned8(y)))))
        return bs_set_error(ctx, BS_EINVAL, "%s: pointers must be 8-byte aligned", name);
    if (int st = bs_check_device(ctx))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n == 0) {
        BS_CUDA_TRY(ctx, cudaMemsetAsync(out, 0, sizeof(double), s));
        return BS_OK;
    }
    const void *ps[2] = {x, dot ? y : x};
    const Plan pl = make_plan(n, ctx->tune.vec_width, ps, 2);
    const int grid = reduce_grid(ctx, pl, dot ? kReduceUnroll : kNormUnroll);
    const RedOut o{ctx->partials, ctx->counter, out};
    if (dot) {
        switch (pl.V) {
        case 4: launch_dot<4, true>(grid, s, x, y, pl, o); break;
        case 2: launch_dot<2, true>(grid, s, x, y, pl, o); break;
        default: launch_dot<1, true>(grid, s, x, y, pl, o); break;
        }
    } else {
        switch (pl.V) {
        case 4: launch_dot<4, false>(grid, s, x, x, pl, o); break;
        case 2: launch_dot<2, false>(grid, s, x, x, pl, o); break;
        default: launch_dot<1, false>(grid, s, x, x, pl, o); break;
        }
    }
    BS_LAUNCH_CHECK(ctx, name);
    return BS_OK;
}

extern "C" int bs_norm(bs_ctx *ctx, int64_t n, const double *x, double *out_dev, void *stream)
{
    return dot_common(ctx, "bs_norm", n, x, nullptr, out_dev, stream, false);
}

extern "C" int bs_dot(bs_ctx *ctx, int64_t n, const double *x, const double *y, double *out_dev,
                      void *stream)
{
    return dot_common(ctx, "bs_dot", n, x, y, out_dev, stream, true);
}

extern "C" int bs_cg_update(bs_ctx *ctx, int64_t n, const double *alpha_num_dev,
                            const double *alpha_den_dev, double alpha, const double *p,
                            const double *Ap, double *x, double *r, double *rdotr_dev,
                            void *stream)
{
    if (!ctx)
        return BS_EINVAL;
    if (n < 0 || (n > 0 && (!p || !Ap || !x || !r)))
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_update: bad length or NULL pointer");
    if ((alpha_num_dev == nullptr) != (alpha_den_dev == nullptr))
        return bs_set_error(ctx, BS_EINVAL,
                            "bs_cg_update: give both alpha_num_dev and alpha_den_dev or neither");
    if ((rdotr_dev && !aligned8(rdotr_dev)) || (alpha_num_dev && !aligned8(alpha_num_dev)) ||
        (alpha_den_dev && !aligned8(alpha_den_dev)) ||
        (n > 0 && (!aligned8(p) || !aligned8(Ap) || !aligned8(x) || !aligned8(r))))
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_update: pointers must be 8-byte aligned");
    const int64_t nb = 8 * n;
    if (bs_overlap(x, nb, r, nb) || bs_overlap(x, nb, p, nb) || bs_overlap(x, nb, Ap, nb) ||
        bs_overlap(r, nb, p, nb) || bs_overlap(r, nb, Ap, nb))
        return bs_set_error(ctx, BS_EINVAL, "bs_cg_update: x and r must not overlap x, r, p, Ap");
    if (int st = bs_check_device(ctx))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (rdotr_dev)
            BS_CUDA_TRY(ctx, cudaMemsetAsync(rdotr_dev, 0, sizeof(double), s));
        return BS_OK;
    }
    const void *ps[4] = {p, Ap, x, r};
    const Plan pl = make_plan(n, ctx->tune.vec_width, ps, 4);
    const int grid = reduce_grid(ctx, pl, kCgUnroll);
    const RedOut o{ctx->partials, ctx->counter, rdotr_dev};
    const bool red = rdotr_dev != nullptr;
    switch (pl.V) {
    case 4: launch_cg<4>(grid, s, alpha_num_dev, alpha_den_dev, alpha, p, Ap, x, r, pl, o, red); break;
    case 2: launch_cg<2>(grid, s, alpha_num_dev, alpha_den_dev, alpha, p, Ap, x, r, pl, o, red); break;
    default: launch_cg<1>(grid, s, alpha_num_dev, alpha_den_dev, alpha, p, Ap, x, r, pl, o, red); break;
    }
    BS_LAUNCH_CHECK(ctx, "cg_kernel");
    return BS_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free inner product.
//
// Some callers cannot call cudaMalloc: code that runs inside a device-memory
// allocator's own hooks (where allocating would recurse into the allocator),
// or an embedding runtime that owns every device allocation and forbids
// others.  They cannot create a bs_ctx either, since a context allocates its
// reduction workspace.  bs_dot_noalloc runs the same BS4 kernel as bs_dot
// but keeps the per-block partial sums and the completion counter in the
// fixed array below, which every GPU that loads this library holds until
// the process exits.
namespace {
constexpr int kNoAllocMaxBlocks = 1024;  // partial sums the array can hold
constexpr size_t kNoAllocCounterOffset = kNoAllocMaxBlocks * sizeof(double);
constexpr size_t kNoAllocScratchBytes = kNoAllocCounterOffset + 256;
constexpr int kNoAllocBlocksPerSm = 4;
} // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of the scratch array on the current device and that
// device's SM count.  The address is looked up on every call (a host-side
// lookup once the module is loaded, no allocation): a cached address could
// outlive the context that the array lives in (cudaDeviceReset, a new
// primary context), and a kernel given it would write to unmapped memory.
int noalloc_setup(unsigned char **scratch, int *sms)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return BS_ECUDA;
    }
    void *p = nullptr;
    int n_sms = 0;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p ||
        cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n_sms < 1) {
        cudaGetLastError();  // this call's own error (none was pending on entry)
        return BS_ECUDA;
    }
    *scratch = static_cast<unsigned char *>(p);
    *sms = n_sms;
    return BS_OK;
}

} // namespace

extern "C" int bs_dot_noalloc(int64_t n, const double *x, const double *y, double *out_dev,
                              void *stream)
{
    if (n < 0 || !out_dev || (n > 0 && (!x || !y)))
        return BS_EINVAL;
    if (!aligned8(out_dev) || (n > 0 && (!aligned8(x) || !aligned8(y))))
        return BS_EINVAL;
    // An error left pending by the caller's earlier work stays theirs: report
    // it, launch nothing and do not clear it.  Past this point any error the
    // runtime reports is this call's own.
    if (cudaPeekAtLastError() != cudaSuccess)
        return BS_ECUDA;
    int sms = 0;
    unsigned char *scratch = nullptr;
    if (int st = noalloc_setup(&scratch, &sms))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (cudaMemsetAsync(out_dev, 0, sizeof(double), s) == cudaSuccess)
            return BS_OK;
        cudaGetLastError();
        return BS_ECUDA;
    }
    const void *ps[2] = {x, y};
    const Plan pl = make_plan(n, 4, ps, 2);
    const int64_t need = ((pl.nv + kReduceUnroll - 1) / kReduceUnroll + kThreads - 1) / kThreads;
    int64_t grid = static_cast<int64_t>(sms) * kNoAllocBlocksPerSm;
    if (need < grid)
        grid = need < 1 ? 1 : need;
    if (grid > kNoAllocMaxBlocks)
        return BS_EINVAL;  // the device wants more partial sums than the array holds
    unsigned int *counter = reinterpret_cast<unsigned int *>(scratch + kNoAllocCounterOffset);
    // The array keeps the previous call's contents; the counter must start at 0.
    if (cudaMemsetAsync(counter, 0, sizeof(unsigned int), s) != cudaSuccess) {
        cudaGetLastError();
        return BS_ECUDA;
    }
    const RedOut o{reinterpret_cast<double *>(scratch), counter, out_dev};
    switch (pl.V) {
    case 4: launch_dot<4, true>(static_cast<int>(grid), s, x, y, pl, o); break;
    case 2: launch_dot<2, true>(static_cast<int>(grid), s, x, y, pl, o); break;
    default: launch_dot<1, true>(static_cast<int>(grid), s, x, y, pl, o); break;
    }
    return cudaGetLastError() == cudaSuccess ? BS_OK : BS_ECUDA;
}
