// The C ABI: argument checks, workspace layout and the launch sequence.
// Every check happens on the host before anything is enqueued.
#include "../../include/moe_prefill.h"
#include "internal.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>

namespace moe {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<bool> g_smem_set[kMaxDevices][kSlotCount];

}  // namespace

int device_sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 1;
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v > 0)
        return v;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t ensure_smem_limit(const void *kernel, int slot, size_t bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached && g_smem_set[dev][slot].load(std::memory_order_acquire))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e == cudaSuccess && cached)
        g_smem_set[dev][slot].store(true, std::memory_order_release);
    return e;
}

}  // namespace moe

namespace {

inline bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline size_t align256(size_t b)
{
    return (b + 255) & ~size_t(255);
}

inline bool base_sizes_ok(int T, int k, int E)
{
    return T >= 0 && k >= 1 && k <= MOE_MAX_TOPK && E >= 1 && E <= MOE_MAX_EXPERTS &&
           int64_t(T) * k <= INT_MAX;
}

inline int cuda_rc(cudaError_t e)
{
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline cudaStream_t as_stream(moe_stream_t s)
{
    return reinterpret_cast<cudaStream_t>(s);
}

int layout(int T, int d, int E, int k, int f, int tm, size_t *out)
{
    if (!base_sizes_ok(T, k, E) || tm < 1 || tm > MOE_MAX_TM || d < 0 || f < 0)
        return MOE_ERR_SHAPE;
    const int64_t cap = moe_capacity(T, k, E, tm);
    if (cap < 0 || cap > INT_MAX)
        return MOE_ERR_CAPACITY;
    const int64_t n = int64_t(T) * k;
    const size_t sizes[MOE_WS_TOTAL] = {
        256,                                             // status word
        size_t(moe::plan_count_rows(n)) * E * 4,       // per-block expert counts / bases
        size_t(E + 1) * 4,                               // offsets
        size_t(E) * 4,                                   // counts
        size_t(cap) * 4,                                 // srt_tok
        size_t(cap) * 4,                                 // srt_w
        size_t(n) * 4,                                   // pos
        size_t(cap / tm + 1) * 4,                        // tile_expert
        // xs; with E4M3 activations it holds the E4M3 rows and their
        // exponents, later those of H
        std::max(size_t(cap) * d * 2, align256(size_t(cap) * f) + size_t(cap) * 4),
        size_t(cap) * f * 2,                             // H
        size_t(cap) * d * 2,                             // Ys
    };
    size_t off = 0;
    for (int i = 0; i < MOE_WS_TOTAL; ++i) {
        out[i] = off;
        off += align256(sizes[i]);
    }
    out[MOE_WS_TOTAL] = off;
    return MOE_OK;
}

}  // namespace

extern "C" {

int64_t moe_capacity(int T, int k, int E, int tm)
{
    if (!base_sizes_ok(T, k, E) || tm < 1 || tm > MOE_MAX_TM)
        return -1;
    const int64_t n = int64_t(T) * k;
    return n + std::min<int64_t>(E, n) * (tm - 1);
}

size_t moe_plan_workspace_bytes(int T, int k, int E)
{
    if (!base_sizes_ok(T, k, E))
        return 0;
    return 256 + align256(size_t(moe::plan_count_rows(int64_t(T) * k)) * E * 4);
}

int moe_plan(const int32_t *ids, const float *w, int T, int k, int E, int tm, int32_t *offsets,
             int32_t *counts, int32_t *srt_tok, float *srt_w, int32_t *pos,
             int32_t *tile_expert, int64_t cap, void *ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!base_sizes_ok(T, k, E) || tm < 1 || tm > MOE_MAX_TM)
        return MOE_ERR_SHAPE;
    if (!offsets || !counts || !srt_tok || !srt_w || !tile_expert || !ws ||
        (T > 0 && (!ids || !w || !pos)))
        return MOE_ERR_NULL;
    if (cap < moe_capacity(T, k, E, tm) || cap > INT_MAX)
        return MOE_ERR_CAPACITY;
    if (ws_bytes < moe_plan_workspace_bytes(T, k, E))
        return MOE_ERR_WORKSPACE;
    if (!aligned(ids, 4) || !aligned(w, 4) || !aligned(offsets, 4) || !aligned(counts, 4) ||
        !aligned(srt_tok, 4) || !aligned(srt_w, 4) || !aligned(pos, 4) ||
        !aligned(tile_expert, 4) || !aligned(ws, 256))
        return MOE_ERR_ALIGN;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    return cuda_rc(moe::launch_plan(ids, w, T, k, E, tm, offsets, counts, srt_tok, srt_w, pos,
                                    tile_expert, cap, reinterpret_cast<uint32_t *>(wsb),
                                    reinterpret_cast<int32_t *>(wsb + 256), as_stream(stream)));
}

int moe_gather(const void *x, int dtype, int T, int d, const int32_t *srt_tok,
               const int32_t *offsets, int E, int64_t cap, void *xs, moe_stream_t stream)
{
    if (dtype != MOE_DT_BF16 && dtype != MOE_DT_F16)
        return MOE_ERR_DTYPE;
    if (T < 0 || d <= 0 || d % 8 != 0 || E < 1 || E > MOE_MAX_EXPERTS)
        return MOE_ERR_SHAPE;
    if (cap < 0 || cap > INT_MAX)
        return MOE_ERR_CAPACITY;
    if (!srt_tok || !offsets || !xs || (T > 0 && !x))
        return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(xs, 16) || !aligned(srt_tok, 4) || !aligned(offsets, 4))
        return MOE_ERR_ALIGN;
    if (cap == 0)
        return MOE_OK;
    return cuda_rc(moe::launch_gather(x, T, d, srt_tok, offsets, E, cap, xs, as_stream(stream)));
}

static int ffn_checks(const void *a, const void *b, const void *c, const int32_t *offsets,
                      int E, int d, int f, int64_t cap, const void *out)
{
    if (E < 1 || E > MOE_MAX_EXPERTS || d <= 0 || f <= 0 || d % 64 != 0 || f % 64 != 0)
        return MOE_ERR_SHAPE;
    if (cap < 0 || cap > INT_MAX)
        return MOE_ERR_CAPACITY;
    if (!a || !b || !c || !offsets || !out)
        return MOE_ERR_NULL;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 16) || !aligned(out, 16) ||
        !aligned(offsets, 4))
        return MOE_ERR_ALIGN;
    return MOE_OK;
}

int moe_ffn_gate_up(const void *xs, const void *Wg, const void *Wu, const int32_t *offsets,
                    int E, int d, int f, int64_t cap, void *H, uint32_t *status,
                    moe_stream_t stream)
{
    const int rc = ffn_checks(xs, Wg, Wu, offsets, E, d, f, cap, H);
    if (rc != MOE_OK || cap == 0)
        return rc;
    if (!aligned(status, 4))
        return MOE_ERR_ALIGN;
    return cuda_rc(moe::launch_ffn_gate_up(xs, Wg, Wu, offsets, E, d, f, cap, H, status,
                                           as_stream(stream)));
}

int moe_ffn_gate_up_rows(const void *x, int T, const int32_t *srt_tok, const void *Wg,
                         const void *Wu, const int32_t *offsets, int E, int d, int f, int64_t cap,
                         void *H, uint32_t *status, moe_stream_t stream)
{
    int rc = ffn_checks(x, Wg, Wu, offsets, E, d, f, cap, H);
    if (rc != MOE_OK)
        return rc;
    if (T < 0)
        return MOE_ERR_SHAPE;
    if (!srt_tok)
        return MOE_ERR_NULL;
    if (!aligned(status, 4) || !aligned(srt_tok, 4))
        return MOE_ERR_ALIGN;
    if (cap == 0 || T == 0)
        return MOE_OK;
    return cuda_rc(moe::launch_ffn_gate_up_rows(x, T, srt_tok, Wg, Wu, offsets, E, d, f, cap, H,
                                                status, as_stream(stream)));
}

int moe_ffn_down(const void *H, const void *Wd, const int32_t *offsets, const float *srt_w,
                 int E, int d, int f, int64_t cap, void *Ys, uint32_t *status,
                 moe_stream_t stream)
{
    const int rc = ffn_checks(H, Wd, srt_w, offsets, E, d, f, cap, Ys);
    if (rc != MOE_OK || cap == 0)
        return rc;
    if (!aligned(status, 4))
        return MOE_ERR_ALIGN;
    return cuda_rc(moe::launch_ffn_down(H, Wd, offsets, srt_w, E, d, f, cap, Ys, status,
                                        as_stream(stream)));
}

int moe_expert_ffn(const void *xs, const void *Wg, const void *Wu, const void *Wd,
                   const int32_t *offsets, const float *srt_w, int E, int d, int f,
                   int64_t cap, void *H, void *Ys, uint32_t *status, moe_stream_t stream)
{
    int rc = ffn_checks(xs, Wg, Wu, offsets, E, d, f, cap, H);
    if (rc == MOE_OK)
        rc = ffn_checks(H, Wd, srt_w, offsets, E, d, f, cap, Ys);
    if (rc != MOE_OK)
        return rc;
    rc = moe_ffn_gate_up(xs, Wg, Wu, offsets, E, d, f, cap, H, status, stream);
    if (rc != MOE_OK)
        return rc;
    return moe_ffn_down(H, Wd, offsets, srt_w, E, d, f, cap, Ys, status, stream);
}

int moe_combine(const void *Ys, const int32_t *pos, int T, int k, int d, void *y,
                moe_stream_t stream)
{
    if (T < 0 || k < 1 || k > MOE_MAX_TOPK || d <= 0 || d % 8 != 0 || int64_t(T) * k > INT_MAX)
        return MOE_ERR_SHAPE;
    if (T == 0)
        return MOE_OK;
    if (!Ys || !pos || !y)
        return MOE_ERR_NULL;
    if (!aligned(Ys, 16) || !aligned(y, 16) || !aligned(pos, 4))
        return MOE_ERR_ALIGN;
    return cuda_rc(moe::launch_combine(Ys, pos, T, k, d, y, as_stream(stream)));
}

size_t moe_workspace_bytes(int T, int d, int E, int k, int f, int tm)
{
    size_t out[MOE_WS_FIELDS];
    return layout(T, d, E, k, f, tm, out) == MOE_OK ? out[MOE_WS_TOTAL] : 0;
}

int moe_workspace_layout(int T, int d, int E, int k, int f, int tm, size_t *out)
{
    if (!out)
        return MOE_ERR_NULL;
    return layout(T, d, E, k, f, tm, out);
}

// The expert weights of a layer: bf16, or E4M3 codes with per-feature scales
// (act_e4m3: Wg, Wu K-major and the gate/up rows in E4M3 too), or MXFP4
// codes with per-block scale exponents (xg, xu, xd).
struct LayerWeights {
    const void *Wg, *Wu, *Wd;
    const float *sg, *su, *sd;  // E4M3 scales; null otherwise
    bool act_e4m3;
    const uint8_t *xg = nullptr, *xu = nullptr, *xd = nullptr;  // MXFP4 scale exponents
};

static int layer_forward(const void *x, const int32_t *ids, const float *w,
                         const LayerWeights &W, int T, int d, int E, int k, int f, int tm, void *y,
                         void *ws, size_t ws_bytes, moe_stream_t stream)
{
    const bool e4m3 = W.sg != nullptr, mx4 = W.xg != nullptr;
    if (!base_sizes_ok(T, k, E) || tm < 16 || tm > MOE_MAX_TM || tm % 16 != 0 || d <= 0 ||
        f <= 0 || d % 64 != 0 || f % 64 != 0)
        return MOE_ERR_SHAPE;
    if (!W.Wg || !W.Wu || !W.Wd || !ws || (T > 0 && (!x || !ids || !w || !y)) ||
        (e4m3 && (!W.su || !W.sd)) || (mx4 && (!W.xu || !W.xd)))
        return MOE_ERR_NULL;
    size_t L[MOE_WS_FIELDS];
    int rc = layout(T, d, E, k, f, tm, L);
    if (rc != MOE_OK)
        return rc;
    if (ws_bytes < L[MOE_WS_TOTAL])
        return MOE_ERR_WORKSPACE;
    if (!aligned(ws, 256) || !aligned(x, 16) || !aligned(y, 16) || !aligned(W.Wg, 16) ||
        !aligned(W.Wu, 16) || !aligned(W.Wd, 16) || !aligned(ids, 4) || !aligned(w, 4) ||
        !aligned(W.sg, 4) || !aligned(W.su, 4) || !aligned(W.sd, 4) || !aligned(W.xg, 16) ||
        !aligned(W.xu, 16) || !aligned(W.xd, 16))
        return MOE_ERR_ALIGN;
    if (T == 0)
        return MOE_OK;
    uint8_t *b = static_cast<uint8_t *>(ws);
    const int64_t cap = moe_capacity(T, k, E, tm);
    uint32_t *status = reinterpret_cast<uint32_t *>(b + L[MOE_WS_STATUS]);
    int32_t *offsets = reinterpret_cast<int32_t *>(b + L[MOE_WS_OFFSETS]);
    int32_t *pos = reinterpret_cast<int32_t *>(b + L[MOE_WS_POS]);
    int32_t *srt_tok = reinterpret_cast<int32_t *>(b + L[MOE_WS_SRT_TOK]);
    float *srt_w = reinterpret_cast<float *>(b + L[MOE_WS_SRT_W]);
    void *xs = b + L[MOE_WS_XS];
    void *H = b + L[MOE_WS_H];
    void *Ys = b + L[MOE_WS_YS];
    cudaStream_t s = as_stream(stream);
    cudaError_t e = moe::launch_plan(
        ids, w, T, k, E, tm, offsets, reinterpret_cast<int32_t *>(b + L[MOE_WS_COUNTS]), srt_tok,
        srt_w, pos, reinterpret_cast<int32_t *>(b + L[MOE_WS_TILE_EXPERT]), cap, status,
        reinterpret_cast<int32_t *>(b + L[MOE_WS_BCNT]), s);
    // E4M3 rows share the xs region: codes [cap, d], then the row exponents
    uint8_t *xs8 = static_cast<uint8_t *>(xs);
    int32_t *xexp = reinterpret_cast<int32_t *>(xs8 + ((size_t(cap) * d + 255) & ~size_t(255)));
    // with E4M3 rows each token is quantized once, into the Ys field (free
    // until down runs), and its codes are then gathered as bytes
    uint8_t *tok8 = static_cast<uint8_t *>(Ys);
    int32_t *texp = reinterpret_cast<int32_t *>(tok8 + ((size_t(T) * d + 255) & ~size_t(255)));
    if (e == cudaSuccess && W.act_e4m3)
        e = moe::launch_quant_tokens_e4m3(x, T, d, tok8, texp, s);
    if (e == cudaSuccess)
        e = W.act_e4m3 ? moe::launch_gather_codes(tok8, texp, T, d, srt_tok, offsets, E, cap, xs8,
                                                  xexp, s)
                       : moe::launch_gather(x, T, d, srt_tok, offsets, E, cap, xs, s);
    const uint8_t *qg = static_cast<const uint8_t *>(W.Wg), *qu = static_cast<const uint8_t *>(W.Wu);
    if (e == cudaSuccess)
        e = W.act_e4m3 ? moe::launch_ffn_gate_up_native(xs8, xexp, qg, W.sg, qu, W.su, offsets, E,
                                                        d, f, cap, H, status, s)
            : mx4      ? moe::launch_ffn_gate_up_mxfp4(xs, qg, W.xg, qu, W.xu, offsets, E, d, f,
                                                       cap, H, status, s)
            : e4m3     ? moe::launch_ffn_gate_up_e4m3(xs, qg, W.sg, qu, W.su, offsets, E, d, f, cap,
                                                      H, status, s)
                       : moe::launch_ffn_gate_up(xs, W.Wg, W.Wu, offsets, E, d, f, cap, H, status,
                                                 s);
    // E4M3 activations: H's rows become E4M3 rows in the xs field (free once
    // gate/up has run), then down runs on them
    uint8_t *h8 = xs8;
    int32_t *hexp = reinterpret_cast<int32_t *>(h8 + ((size_t(cap) * f + 255) & ~size_t(255)));
    if (e == cudaSuccess && W.act_e4m3)
        e = moe::launch_rows_e4m3(H, f, offsets, E, cap, h8, hexp, s);
    const uint8_t *qd = static_cast<const uint8_t *>(W.Wd);
    if (e == cudaSuccess)
        e = W.act_e4m3 ? moe::launch_ffn_down_native(h8, hexp, qd, W.sd, offsets, srt_w, E, d, f,
                                                     cap, Ys, status, s)
            : mx4      ? moe::launch_ffn_down_mxfp4(H, qd, W.xd, offsets, srt_w, E, d, f, cap, Ys,
                                                    status, s)
            : e4m3     ? moe::launch_ffn_down_e4m3(H, qd, W.sd, offsets, srt_w, E, d, f, cap, Ys,
                                                   status, s)
                       : moe::launch_ffn_down(H, W.Wd, offsets, srt_w, E, d, f, cap, Ys, status,
                                              s);
    if (e == cudaSuccess)
        e = moe::launch_combine(Ys, pos, T, k, d, y, s);
    return cuda_rc(e);
}

int moe_layer_forward(const void *x, const int32_t *ids, const float *w, const void *Wg,
                      const void *Wu, const void *Wd, int T, int d, int E, int k, int f, int tm,
                      void *y, void *ws, size_t ws_bytes, moe_stream_t stream)
{
    const LayerWeights W{Wg, Wu, Wd, nullptr, nullptr, nullptr, false};
    return layer_forward(x, ids, w, W, T, d, E, k, f, tm, y, ws, ws_bytes, stream);
}

int moe_layer_forward_e4m3(const void *x, const int32_t *ids, const float *w, const uint8_t *Wg,
                           const float *sg, const uint8_t *Wu, const float *su,
                           const uint8_t *Wd, const float *sd, int T, int d, int E, int k, int f,
                           int tm, void *y, void *ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!sg)
        return MOE_ERR_NULL;
    const LayerWeights W{Wg, Wu, Wd, sg, su, sd, false};
    return layer_forward(x, ids, w, W, T, d, E, k, f, tm, y, ws, ws_bytes, stream);
}

int moe_layer_forward_f8(const void *x, const int32_t *ids, const float *w, const uint8_t *Wg,
                         const float *sg, const uint8_t *Wu, const float *su, const uint8_t *Wd,
                         const float *sd, int T, int d, int E, int k, int f, int tm, void *y,
                         void *ws, size_t ws_bytes, moe_stream_t stream)
{
    if (!sg)
        return MOE_ERR_NULL;
    const LayerWeights W{Wg, Wu, Wd, sg, su, sd, true};
    return layer_forward(x, ids, w, W, T, d, E, k, f, tm, y, ws, ws_bytes, stream);
}

int moe_layer_forward_mxfp4(const void *x, const int32_t *ids, const float *w,
                            const uint8_t *Wg, const uint8_t *xg, const uint8_t *Wu,
                            const uint8_t *xu, const uint8_t *Wd, const uint8_t *xd, int T, int d,
                            int E, int k, int f, int tm, void *y, void *ws, size_t ws_bytes,
                            moe_stream_t stream)
{
    if (!xg)
        return MOE_ERR_NULL;
    LayerWeights W{Wg, Wu, Wd, nullptr, nullptr, nullptr, false};
    W.xg = xg;
    W.xu = xu;
    W.xd = xd;
    return layer_forward(x, ids, w, W, T, d, E, k, f, tm, y, ws, ws_bytes, stream);
}

int moe_quantize_mxfp4(const void *W, int E, int K, int M, uint8_t *codes, uint8_t *scales,
                       moe_stream_t stream)
{
    if (E < 1 || E > MOE_MAX_EXPERTS || K < 32 || M < 2 || K % 32 != 0 || M % 2 != 0)
        return MOE_ERR_SHAPE;
    if (!W || !codes || !scales)
        return MOE_ERR_NULL;
    if (!aligned(W, 4) || !aligned(codes, 16))
        return MOE_ERR_ALIGN;
    return cuda_rc(moe::launch_quantize_mxfp4(W, E, K, M, codes, scales, as_stream(stream)));
}

int moe_ffn_gate_up_mxfp4(const void *xs, const uint8_t *Wg, const uint8_t *xg, const uint8_t *Wu,
                          const uint8_t *xu, const int32_t *offsets, int E, int d, int f,
                          int64_t cap, void *H, uint32_t *status, moe_stream_t stream)
{
    int rc = ffn_checks(xs, Wg, Wu, offsets, E, d, f, cap, H);
    if (rc == MOE_OK && (!xg || !xu))
        rc = MOE_ERR_NULL;
    if (rc == MOE_OK && (!aligned(xg, 16) || !aligned(xu, 16) || !aligned(status, 4)))
        rc = MOE_ERR_ALIGN;
    if (rc != MOE_OK || cap == 0)
        return rc;
    return cuda_rc(moe::launch_ffn_gate_up_mxfp4(xs, Wg, xg, Wu, xu, offsets, E, d, f, cap, H,
                                                 status, as_stream(stream)));
}

int moe_ffn_down_mxfp4(const void *H, const uint8_t *Wd, const uint8_t *xd, const int32_t *offsets,
                       const float *srt_w, int E, int d, int f, int64_t cap, void *Ys,
                       uint32_t *status, moe_stream_t stream)
{
    int rc = ffn_checks(H, Wd, srt_w, offsets, E, d, f, cap, Ys);
    if (rc == MOE_OK && !xd)
        rc = MOE_ERR_NULL;
    if (rc == MOE_OK && (!aligned(xd, 16) || !aligned(status, 4)))
        rc = MOE_ERR_ALIGN;
    if (rc != MOE_OK || cap == 0)
        return rc;
    return cuda_rc(moe::launch_ffn_down_mxfp4(H, Wd, xd, offsets, srt_w, E, d, f, cap, Ys, status,
                                              as_stream(stream)));
}

int moe_quantize_e4m3(const void *W, int E, int K, int M, uint8_t *q, float *scale, int kmajor,
                      moe_stream_t stream)
{
    if (E < 1 || E > MOE_MAX_EXPERTS || K < 1 || M < 1 || (kmajor && (K % 64 || M % 64)))
        return MOE_ERR_SHAPE;
    if (!W || !q || !scale)
        return MOE_ERR_NULL;
    if (!aligned(W, 2) || !aligned(scale, 4))
        return MOE_ERR_ALIGN;
    return cuda_rc(moe::launch_quantize_e4m3(W, E, K, M, q, scale, kmajor != 0,
                                             as_stream(stream)));
}

int moe_gather_e4m3(const void *x, int T, int d, const int32_t *srt_tok, const int32_t *offsets,
                    int E, int64_t cap, uint8_t *xs8, int32_t *xexp, moe_stream_t stream)
{
    if (T < 0 || d <= 0 || d % 16 != 0 || E < 1 || E > MOE_MAX_EXPERTS)
        return MOE_ERR_SHAPE;
    if (cap < 0 || cap > INT_MAX)
        return MOE_ERR_CAPACITY;
    if (!srt_tok || !offsets || !xs8 || !xexp || (T > 0 && !x))
        return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(xs8, 16) || !aligned(xexp, 4) || !aligned(srt_tok, 4) ||
        !aligned(offsets, 4))
        return MOE_ERR_ALIGN;
    if (cap == 0)
        return MOE_OK;
    return cuda_rc(moe::launch_gather_e4m3(x, T, d, srt_tok, offsets, E, cap, xs8, xexp,
                                           as_stream(stream)));
}

int moe_ffn_gate_up_f8(const uint8_t *xs8, const int32_t *xexp, const uint8_t *Wg,
                       const float *sg, const uint8_t *Wu, const float *su,
                       const int32_t *offsets, int E, int d, int f, int64_t cap, void *H,
                       uint32_t *status, moe_stream_t stream)
{
    int rc = ffn_checks(xs8, Wg, Wu, offsets, E, d, f, cap, H);
    if (rc == MOE_OK && (!sg || !su || !xexp))
        rc = MOE_ERR_NULL;
    if (rc == MOE_OK &&
        (!aligned(sg, 4) || !aligned(su, 4) || !aligned(xexp, 4) || !aligned(status, 4)))
        rc = MOE_ERR_ALIGN;
    if (rc != MOE_OK || cap == 0)
        return rc;
    return cuda_rc(moe::launch_ffn_gate_up_native(xs8, xexp, Wg, sg, Wu, su, offsets, E, d, f, cap,
                                                  H, status, as_stream(stream)));
}

int moe_rows_e4m3(const void *H, int f, const int32_t *offsets, int E, int64_t cap, uint8_t *H8,
                  int32_t *hexp, moe_stream_t stream)
{
    if (f <= 0 || f % 16 != 0 || E < 1 || E > MOE_MAX_EXPERTS)
        return MOE_ERR_SHAPE;
    if (cap < 0 || cap > INT_MAX)
        return MOE_ERR_CAPACITY;
    if (!H || !offsets || !H8 || !hexp)
        return MOE_ERR_NULL;
    if (!aligned(H, 16) || !aligned(H8, 16) || !aligned(hexp, 4) || !aligned(offsets, 4))
        return MOE_ERR_ALIGN;
    if (cap == 0)
        return MOE_OK;
    return cuda_rc(moe::launch_rows_e4m3(H, f, offsets, E, cap, H8, hexp, as_stream(stream)));
}

int moe_ffn_down_f8(const uint8_t *H8, const int32_t *hexp, const uint8_t *Wd, const float *sd,
                    const int32_t *offsets, const float *srt_w, int E, int d, int f, int64_t cap,
                    void *Ys, uint32_t *status, moe_stream_t stream)
{
    int rc = ffn_checks(H8, Wd, srt_w, offsets, E, d, f, cap, Ys);
    if (rc == MOE_OK && (!sd || !hexp))
        rc = MOE_ERR_NULL;
    if (rc == MOE_OK && (!aligned(sd, 4) || !aligned(hexp, 4) || !aligned(status, 4)))
        rc = MOE_ERR_ALIGN;
    if (rc != MOE_OK || cap == 0)
        return rc;
    return cuda_rc(moe::launch_ffn_down_native(H8, hexp, Wd, sd, offsets, srt_w, E, d, f, cap, Ys,
                                               status, as_stream(stream)));
}

int moe_ffn_gate_up_e4m3(const void *xs, const uint8_t *Wg, const float *sg, const uint8_t *Wu,
                         const float *su, const int32_t *offsets, int E, int d, int f,
                         int64_t cap, void *H, uint32_t *status, moe_stream_t stream)
{
    int rc = ffn_checks(xs, Wg, Wu, offsets, E, d, f, cap, H);
    if (rc == MOE_OK && (!sg || !su))
        rc = MOE_ERR_NULL;
    if (rc == MOE_OK && (!aligned(sg, 4) || !aligned(su, 4) || !aligned(status, 4)))
        rc = MOE_ERR_ALIGN;
    if (rc != MOE_OK || cap == 0)
        return rc;
    return cuda_rc(moe::launch_ffn_gate_up_e4m3(xs, Wg, sg, Wu, su, offsets, E, d, f, cap, H,
                                                status, as_stream(stream)));
}

int moe_ffn_down_e4m3(const void *H, const uint8_t *Wd, const float *sd, const int32_t *offsets,
                      const float *srt_w, int E, int d, int f, int64_t cap, void *Ys,
                      uint32_t *status, moe_stream_t stream)
{
    int rc = ffn_checks(H, Wd, srt_w, offsets, E, d, f, cap, Ys);
    if (rc == MOE_OK && !sd)
        rc = MOE_ERR_NULL;
    if (rc == MOE_OK && (!aligned(sd, 4) || !aligned(status, 4)))
        rc = MOE_ERR_ALIGN;
    if (rc != MOE_OK || cap == 0)
        return rc;
    return cuda_rc(moe::launch_ffn_down_e4m3(H, Wd, sd, offsets, srt_w, E, d, f, cap, Ys, status,
                                             as_stream(stream)));
}

int moe_selftest_wait_limit(const void *xs, const void *Wg, const void *Wu,
                            const int32_t *offsets, int E, int d, int f, int64_t cap, void *H,
                            uint32_t *status, int cta, moe_stream_t stream)
{
    const int rc = ffn_checks(xs, Wg, Wu, offsets, E, d, f, cap, H);
    if (rc != MOE_OK)
        return rc;
    if (!status)
        return MOE_ERR_NULL;
    if (!aligned(status, 4))
        return MOE_ERR_ALIGN;
    if (cta < 0 || cap == 0)
        return MOE_ERR_SHAPE;
    return cuda_rc(moe::launch_ffn_gate_up(xs, Wg, Wu, offsets, E, d, f, cap, H, status,
                                           as_stream(stream), cta));
}

int moe_read_status(const void *ws, moe_stream_t stream, uint32_t *status)
{
    if (!ws || !status)
        return MOE_ERR_NULL;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return cuda_rc(cudaStreamSynchronize(s));
}

const char *moe_status_str(int code)
{
    switch (code) {
    case MOE_OK:
        return "ok";
    case MOE_ERR_NULL:
        return "a required pointer is NULL";
    case MOE_ERR_SHAPE:
        return "a size is outside its documented range";
    case MOE_ERR_CAPACITY:
        return "capacity smaller than moe_capacity(T, k, E, tm) or above INT_MAX";
    case MOE_ERR_WORKSPACE:
        return "workspace smaller than required";
    case MOE_ERR_ALIGN:
        return "a pointer is not aligned as required";
    case MOE_ERR_CUDA:
        return "a CUDA call or kernel launch failed";
    case MOE_ERR_DTYPE:
        return "unsupported dtype";
    default:
        return "unknown return code";
    }
}

}  // extern "C"
