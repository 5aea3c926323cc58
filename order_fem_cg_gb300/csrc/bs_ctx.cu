// bs_ctx.cu -- contexts, error reporting, device status.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <new>

#include "bs_internal.h"
#include "bs_mesh_impl.h"

int bs_set_error(bs_ctx *ctx, int status, const char *fmt, ...)
{
    if (ctx) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(ctx->msg, sizeof(ctx->msg), fmt, ap);
        va_end(ap);
    }
    return status;
}

bool bs_fault(const char *what)
{
    const char *s = std::getenv("BS_FAULT");
    if (!s || !*what)
        return false;
    const size_t n = std::strlen(what);
    while (*s) {
        const char *e = std::strchr(s, ',');
        const size_t len = e ? static_cast<size_t>(e - s) : std::strlen(s);
        if (len == n && std::strncmp(s, what, n) == 0)
            return true;
        if (!e)
            break;
        s = e + 1;
    }
    return false;
}

int bs_check_device(bs_ctx *ctx, bool launching)
{
    if (launching && bs_fault("launch"))
        return bs_set_error(ctx, BS_ECUDA, "injected launch failure (BS_FAULT=launch)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return bs_set_error(ctx, BS_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev != ctx->device)
        return bs_set_error(ctx, BS_EINVAL, "current device %d is not the context's device %d",
                            dev, ctx->device);
    return BS_OK;
}

extern "C" const char *bs_strerror(int status)
{
    switch (status) {
    case BS_OK: return "ok";
    case BS_EINVAL: return "invalid argument";
    case BS_ECUDA: return "CUDA error";
    case BS_ENOMEM: return "out of memory";
    case BS_EBOUNDS: return "index table entry out of range";
    case BS_EALIGN: return "misaligned pointer";
    case BS_ETIMEOUT: return "a device-side wait timed out";
    default: return "unknown status";
    }
}

extern "C" const char *bs_last_error(const bs_ctx *ctx)
{
    return ctx ? ctx->msg : "no context";
}

static int env_int(const char *name, int dflt, int lo, int hi)
{
    const char *s = std::getenv(name);
    if (!s || !*s)
        return dflt;
    int v = std::atoi(s);
    return v < lo ? lo : (v > hi ? hi : v);
}

extern "C" int bs_ctx_create(int device, bs_ctx **out)
{
    if (!out)
        return BS_EINVAL;
    *out = nullptr;
    if (bs_fault("alloc"))
        return BS_ENOMEM;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
        cudaGetLastError();
        return BS_EINVAL;
    }
    bs_ctx *ctx = new (std::nothrow) bs_ctx();
    if (!ctx)
        return BS_ENOMEM;
    ctx->device = device;
    int prev = 0;
    cudaGetDevice(&prev);
    int st = BS_OK;
    do {
        if (cudaSetDevice(device) != cudaSuccess) { st = BS_ECUDA; break; }
        if (cudaDeviceGetAttribute(&ctx->sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
            cudaDeviceGetAttribute(&ctx->l2_bytes, cudaDevAttrL2CacheSize, device) != cudaSuccess) {
            st = BS_ECUDA;
            break;
        }
        ctx->tune.stream_blocks_per_sm = env_int("BS_TUNE_STREAM_BPS", 4, 1, 32);
        ctx->tune.reduce_blocks_per_sm = env_int("BS_TUNE_REDUCE_BPS", 4, 1, 32);
        ctx->tune.scatter_blocks_per_sm = env_int("BS_TUNE_SCATTER_BPS", 8, 1, 32);
        ctx->tune.vec_width = env_int("BS_TUNE_VEC", 4, 1, 4);
        ctx->tune.persist = env_int("BS_TUNE_PERSIST", 0, 0, 1);
        ctx->tune.l2_prefetch = env_int("BS_TUNE_L2PF", 1, 0, 1);
        ctx->tune.small_onepass = env_int("BS_TUNE_ONEPASS", 1, 0, 1);
        ctx->tune.tmem = env_int("BS_TUNE_TMEM", 1, 0, 1);
        if (ctx->tune.vec_width == 3)
            ctx->tune.vec_width = 2;
        if (cudaMalloc(&ctx->partials, kMaxReduceBlocks * sizeof(double)) != cudaSuccess ||
            cudaMalloc(&ctx->counter, 256) != cudaSuccess ||
            cudaMalloc(&ctx->dev_err, 256) != cudaSuccess) {
            st = BS_ENOMEM;
            break;
        }
        if (cudaMemset(ctx->counter, 0, 256) != cudaSuccess ||
            cudaMemset(ctx->dev_err, 0, 256) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            st = BS_ECUDA;
            break;
        }
    } while (0);
    cudaGetLastError();
    cudaSetDevice(prev);
    if (st != BS_OK) {
        bs_ctx_destroy(ctx);
        return st;
    }
    *out = ctx;
    return BS_OK;
}

extern "C" int bs_ctx_destroy(bs_ctx *ctx)
{
    if (!ctx)
        return BS_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(ctx->device);
    if (ctx->partials) cudaFree(ctx->partials);
    if (ctx->counter) cudaFree(ctx->counter);
    if (ctx->dev_err) cudaFree(ctx->dev_err);
    cudaGetLastError();
    cudaSetDevice(prev);
    delete ctx;
    return BS_OK;
}

extern "C" int bs_ctx_num_sms(const bs_ctx *ctx)
{
    return ctx ? ctx->sms : 0;
}

extern "C" int bs_ctx_device_status(bs_ctx *ctx, void *stream, int *out_status)
{
    if (!ctx || !out_status)
        return BS_EINVAL;
    if (int st = bs_check_device(ctx, false))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int flag = 0;
    BS_CUDA_TRY(ctx, cudaMemcpyAsync(&flag, ctx->dev_err, sizeof(int), cudaMemcpyDeviceToHost, s));
    BS_CUDA_TRY(ctx, cudaMemsetAsync(ctx->dev_err, 0, sizeof(int), s));
    BS_CUDA_TRY(ctx, cudaStreamSynchronize(s));
    *out_status = (flag & BS_DEVERR_TIMEOUT) ? BS_ETIMEOUT : flag ? BS_EBOUNDS : BS_OK;
    if (flag & BS_DEVERR_TIMEOUT)
        bs_set_error(ctx, BS_ETIMEOUT, "a grid barrier of a cooperative kernel gave up waiting");
    else if (flag)
        bs_set_error(ctx, BS_EBOUNDS, "a gather/scatter kernel met an out-of-range table entry");
    return BS_OK;
}
