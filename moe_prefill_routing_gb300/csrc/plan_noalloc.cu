// moe_plan_noalloc: the routing plan with its scratch (status word + per-block
// expert counts) in a fixed device array of this library instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
// It launches the same kernels as moe_plan.
#include "../../include/moe_prefill.h"
#include "internal.h"

#include <cuda_runtime.h>

#include <climits>
#include <mutex>

namespace {

constexpr size_t kHeaderBytes = 256;  // status word when the caller passes none

// Scratch shared by every moe_plan_noalloc call on a device.  In host code
// this name only stands for the array; its device address comes from
// cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_plan_scratch[MOE_PLAN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of g_plan_scratch on the current device, looked up once per
// device (with that device current).
cudaError_t scratch_address(unsigned char **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_plan_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_scratch_addr[dev]);
    return cudaSuccess;
}

inline bool aligned4(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 3) == 0;
}

}  // namespace

extern "C" int moe_plan_noalloc(const int32_t *ids, const float *w, int T, int k, int E, int tm,
                                int32_t *offsets, int32_t *counts, int32_t *srt_tok,
                                float *srt_w, int32_t *pos, int32_t *tile_expert, int64_t cap,
                                uint32_t *status, moe_stream_t stream)
{
    if (T < 0 || k < 1 || k > MOE_MAX_TOPK || E < 1 || E > MOE_MAX_EXPERTS ||
        int64_t(T) * k > INT_MAX || tm < 1 || tm > MOE_MAX_TM)
        return MOE_ERR_SHAPE;
    if (!offsets || !counts || !srt_tok || !srt_w || !tile_expert ||
        (T > 0 && (!ids || !w || !pos)))
        return MOE_ERR_NULL;
    if (cap < moe_capacity(T, k, E, tm) || cap > INT_MAX)
        return MOE_ERR_CAPACITY;
    if (int64_t(moe::plan_count_rows(int64_t(T) * k)) * E > MOE_PLAN_NOALLOC_MAX_COUNTS)
        return MOE_ERR_WORKSPACE;
    if (!aligned4(ids) || !aligned4(w) || !aligned4(offsets) || !aligned4(counts) ||
        !aligned4(srt_tok) || !aligned4(srt_w) || !aligned4(pos) || !aligned4(tile_expert) ||
        !aligned4(status))
        return MOE_ERR_ALIGN;
    unsigned char *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return MOE_ERR_CUDA;
    uint32_t *st = status ? status : reinterpret_cast<uint32_t *>(scratch);
    const cudaError_t e = moe::launch_plan(
        ids, w, T, k, E, tm, offsets, counts, srt_tok, srt_w, pos, tile_expert, cap, st,
        reinterpret_cast<int32_t *>(scratch + kHeaderBytes), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
