// bs_internal.h -- shared definitions of the libbs.so translation units.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "bs.h"

// Reduction workspace capacity: one partial sum per block of a reduction.
constexpr int kMaxReduceBlocks = 4096;

// Launch-shape knobs of a context.  Defaults are the tuned values for
// GB300; BS_TUNE_* environment variables override them at context creation
// (used by the tuning sweeps; never needed for correctness).
struct bs_tune {
    int stream_blocks_per_sm;  // BS1/BS2 grid = SMs x this
    int reduce_blocks_per_sm;  // BS3-BS5 grid = SMs x this (capped by kMaxReduceBlocks)
    int scatter_blocks_per_sm; // BS7 grid = SMs x this
    int vec_width;             // widest vector in doubles: 4 (32 B), 2 (16 B) or 1
    int persist;               // two-pass kernels: 1 one block (cluster) per SM looping over
                               // tiles/buckets, 0 one block per tile/bucket
    int l2_prefetch;           // persistent two-pass kernels: 1 prefetch each block's next
                               // tile/bucket into L2 while it works on the current one
    int tmem;                  // gather pass 2 stages the next bucket in TMEM (1, default:
                               // measured faster) or holds one bucket at a time (0)
    int small_onepass;         // 1: one-pass gather/scatter for L2-sized vectors even with a
                               // plan (bs_gather / bs_scatter); 0: always the plan
};

// Below these sizes of the randomly read vector the one-pass kernels beat
// the two-pass plan on GB300 (random reads that stay in L2 run ~3.7x faster
// than from HBM, and a two-pass call pays two launches and its phases):
// scatter reads q_G, gather reads q_L.  Measured: scatter 23 against 42 us
// at q_G = 22 MB, gather 9 against 29 us at q_L = 0.3 MB but 61 against
// 56 us at q_L = 33 MB.
constexpr int64_t kOnePassScatterBytes = BS_ONEPASS_SCATTER_BYTES;
constexpr int64_t kOnePassGatherBytes = BS_ONEPASS_GATHER_BYTES;

struct bs_ctx {
    int device;
    int sms;
    int l2_bytes;
    bs_tune tune;
    double *partials;      // [kMaxReduceBlocks] device
    unsigned int *counter; // [1] device, zero between launches
    int *dev_err;          // [1] device, 0 = ok, else BS_DEVERR_* bits
    char msg[512];
};

// Bits of the device error flag.
constexpr int BS_DEVERR_BOUNDS = 1;
constexpr int BS_DEVERR_TIMEOUT = 2;  // a bounded device-side wait gave up

int bs_set_error(bs_ctx *ctx, int status, const char *fmt, ...);

// Returns BS_OK if the calling thread's current device is the context's.
// With launching (every call that launches work), an injected "launch"
// fault (bs_fault) makes it report BS_ECUDA instead, so nothing launches.
int bs_check_device(bs_ctx *ctx, bool launching = true);

#ifdef __CUDACC__
// a * b as the fused multiply-add a * b + mzero with mzero = -0 passed in at
// run time (a constant -0 lets the compiler turn it back into a multiply):
// adding -0 changes no rounded product (a zero product keeps its sign), so
// the result is bit for bit that of a multiplication, and on GB300 the FP64
// pipe retires fused multiply-adds faster than multiplications.
__device__ __forceinline__ double mul_rn(double a, double b, double mzero)
{
    double r;
    asm("fma.rn.f64 %0, %1, %2, %3;" : "=d"(r) : "d"(a), "d"(b), "d"(mzero));
    return r;
}
#endif

#define BS_CUDA_TRY(ctx, call)                                                                   \
    do {                                                                                         \
        cudaError_t e_ = (call);                                                                 \
        if (e_ != cudaSuccess)                                                                   \
            return bs_set_error((ctx), BS_ECUDA, "%s: %s", #call, cudaGetErrorString(e_));      \
    } while (0)

#define BS_LAUNCH_CHECK(ctx, what)                                                               \
    do {                                                                                         \
        cudaError_t e_ = cudaGetLastError();                                                     \
        if (e_ != cudaSuccess)                                                                   \
            return bs_set_error((ctx), BS_ECUDA, "launch of %s: %s", (what),                     \
                                cudaGetErrorString(e_));                                         \
    } while (0)

// Two-pass tiled gather/scatter (bs_gs2.cu); t->plan is non-NULL and the
// common arguments are already validated.
int bs_scatter_planned(bs_ctx *ctx, const bs_gs_dev *t, const double *qG, double *qL,
                       cudaStream_t s);
int bs_gather_planned(bs_ctx *ctx, const bs_gs_dev *t, const double *qL, double *qG,
                      cudaStream_t s);
int bs_apply_diag_planned(bs_ctx *ctx, const bs_gs_dev *t, const double *xG, const double *dL,
                          double *yG, cudaStream_t s);

// Do the byte ranges [a, a+na) and [b, b+nb) overlap?
inline bool bs_overlap(const void *a, int64_t na, const void *b, int64_t nb)
{
    auto pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && pa < pb + static_cast<uintptr_t>(nb) &&
           pb < pa + static_cast<uintptr_t>(na);
}
