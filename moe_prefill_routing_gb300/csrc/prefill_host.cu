// A prompt processed as a sequence of prefill chunks straight from host
// memory: each chunk's x, ids and w are copied in, the layer runs, and y is
// copied back.  "Round 4 Track C: Prefill MoE Plan ...", Table 2.1, runs the
// layer on chunks of a prompt, and "#372 Prompt path ..." measures prompts
// of 2K-32K tokens; neither page moves data between host and device, so
// the overlap below is this library's own: two copy streams and two sets of
// device staging buffers let chunk c+1's host-to-device copies and chunk
// c-1's device-to-host copy run on the copy engines while chunk c's layer
// runs on the caller's stream.
#include "../../include/moe_prefill.h"
#include "internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kMaxDevices = 64;

struct CopyStreams {
    cudaStream_t h2d = nullptr;
    cudaStream_t d2h = nullptr;
};

std::mutex g_streams_mu;
CopyStreams g_streams[kMaxDevices];

// The two copy streams of the current device, created on first use and kept
// for the life of the process.
cudaError_t copy_streams(CopyStreams &out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_streams_mu);
    CopyStreams &cs = g_streams[dev];
    if (!cs.h2d) {
        cudaStream_t a = nullptr, b = nullptr;
        e = cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            if (a)
                cudaStreamDestroy(a);
            return e;
        }
        cs.h2d = a;
        cs.d2h = b;
    }
    out = cs;
    return cudaSuccess;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Byte offsets inside the workspace: the layer's workspace, then two sets
// of staging buffers (x, ids, w, y).
struct HostLayout {
    size_t layer, x, ids, w, y, set, total;
};

bool host_layout(int T, int d, int E, int k, int f, int tm, HostLayout &L)
{
    const size_t layer = moe_workspace_bytes(T, d, E, k, f, tm);
    if (layer == 0)
        return false;
    L.layer = align256(layer);
    L.x = 0;
    L.ids = L.x + align256(size_t(T) * d * 2);
    L.w = L.ids + align256(size_t(T) * k * 4);
    L.y = L.w + align256(size_t(T) * k * 4);
    L.set = L.y + align256(size_t(T) * d * 2);
    L.total = L.layer + 2 * L.set;
    return true;
}

// Events of one call, released when it returns; work already enqueued on
// them is unaffected.
struct CallEvents {
    static constexpr int kCount = 7;
    cudaEvent_t ev[kCount] = {};
    cudaError_t create()
    {
        for (int i = 0; i < kCount; ++i) {
            const cudaError_t e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
            if (e != cudaSuccess)
                return e;
        }
        return cudaSuccess;
    }
    ~CallEvents()
    {
        for (int i = 0; i < kCount; ++i)
            if (ev[i])
                cudaEventDestroy(ev[i]);
    }
};

}  // namespace
}  // namespace moe

extern "C" {

size_t moe_prefill_host_workspace_bytes(int T, int d, int E, int k, int f, int tm)
{
    moe::HostLayout L;
    return moe::host_layout(T, d, E, k, f, tm, L) ? L.total : 0;
}

int moe_prefill_forward_host(int n_chunks, const void *const *x_h, const int32_t *const *ids_h,
                             const float *const *w_h, void *const *y_h, const void *Wg,
                             const void *Wu, const void *Wd, const float *sg, const float *su,
                             const float *sd, int act_e4m3, int T, int d, int E, int k, int f,
                             int tm, void *ws, size_t ws_bytes, moe_stream_t stream)
{
    if (n_chunks < 0)
        return MOE_ERR_SHAPE;
    moe::HostLayout L;
    // the shape rules of moe_layer_forward, checked before anything is enqueued
    if (tm < 16 || tm % 16 != 0 || d <= 0 || f <= 0 || d % 64 != 0 || f % 64 != 0 ||
        !moe::host_layout(T, d, E, k, f, tm, L))
        return MOE_ERR_SHAPE;
    if (!Wg || !Wu || !Wd || !ws || (n_chunks > 0 && (!x_h || !ids_h || !w_h || !y_h)) ||
        (sg && (!su || !sd)) || (act_e4m3 && !sg))
        return MOE_ERR_NULL;
    for (int c = 0; T > 0 && c < n_chunks; ++c)
        if (!x_h[c] || !ids_h[c] || !w_h[c] || !y_h[c])
            return MOE_ERR_NULL;
    if (ws_bytes < L.total)
        return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0 ||
        ((reinterpret_cast<uintptr_t>(Wg) | reinterpret_cast<uintptr_t>(Wu) |
          reinterpret_cast<uintptr_t>(Wd)) & 15) != 0)
        return MOE_ERR_ALIGN;
    if (n_chunks == 0 || T == 0)
        return MOE_OK;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    moe::CopyStreams cs;
    moe::CallEvents evs;
    cudaError_t e = moe::copy_streams(cs);
    if (e == cudaSuccess)
        e = evs.create();
    if (e != cudaSuccess)
        return MOE_ERR_CUDA;
    cudaEvent_t start = evs.ev[0], *in = evs.ev + 1, *out = evs.ev + 3, *back = evs.ev + 5;

    uint8_t *base = static_cast<uint8_t *>(ws);
    void *layer_ws = base;
    const size_t xb = size_t(T) * d * 2, ikb = size_t(T) * k * 4;
    // the copy streams start after everything already on the caller's stream
    e = cudaEventRecord(start, s);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(cs.h2d, start, 0);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(cs.d2h, start, 0);
    for (int c = 0; e == cudaSuccess && c < n_chunks; ++c) {
        const int b = c & 1;
        uint8_t *set = base + L.layer + size_t(b) * L.set;
        void *x = set + L.x, *y = set + L.y;
        int32_t *ids = reinterpret_cast<int32_t *>(set + L.ids);
        float *w = reinterpret_cast<float *>(set + L.w);
        // inputs: staging set b is free once chunk c-2's layer has run
        if (c >= 2)
            e = cudaStreamWaitEvent(cs.h2d, out[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(x, x_h[c], xb, cudaMemcpyHostToDevice, cs.h2d);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ids, ids_h[c], ikb, cudaMemcpyHostToDevice, cs.h2d);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(w, w_h[c], ikb, cudaMemcpyHostToDevice, cs.h2d);
        if (e == cudaSuccess)
            e = cudaEventRecord(in[b], cs.h2d);
        // the layer: after its inputs land and after chunk c-2's y has left
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(s, in[b], 0);
        if (e == cudaSuccess && c >= 2)
            e = cudaStreamWaitEvent(s, back[b], 0);
        if (e != cudaSuccess)
            break;
        const uint8_t *qg = static_cast<const uint8_t *>(Wg), *qu = static_cast<const uint8_t *>(Wu),
                      *qd = static_cast<const uint8_t *>(Wd);
        const int rc =
            act_e4m3 ? moe_layer_forward_f8(x, ids, w, qg, sg, qu, su, qd, sd, T, d, E, k, f, tm,
                                            y, layer_ws, L.layer, stream)
            : sg     ? moe_layer_forward_e4m3(x, ids, w, qg, sg, qu, su, qd, sd, T, d, E, k, f, tm,
                                              y, layer_ws, L.layer, stream)
                     : moe_layer_forward(x, ids, w, Wg, Wu, Wd, T, d, E, k, f, tm, y, layer_ws,
                                         L.layer, stream);
        if (rc != MOE_OK)
            return rc;
        e = cudaEventRecord(out[b], s);
        // the result
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(cs.d2h, out[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(y_h[c], y, xb, cudaMemcpyDeviceToHost, cs.d2h);
        if (e == cudaSuccess)
            e = cudaEventRecord(back[b], cs.d2h);
    }
    // join: the caller's stream completes after the last copy back
    for (int b = 0; e == cudaSuccess && b < 2 && b < n_chunks; ++b)
        e = cudaStreamWaitEvent(s, back[b], 0);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
