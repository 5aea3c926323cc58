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
    int l2_prefetch;           // two-pass kernels: 0 none (default: measured fastest),
                               // 1 own inputs, 2 also the inputs of the block one wave ahead
};

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
