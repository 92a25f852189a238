// Row kernels: the gather of token rows into expert-sorted order and the
// slot-ordered combine.  Both are HBM-bound copies/reductions of whole
// 16-byte-aligned rows, so they move 128-bit vectors with every lane of a
// warp on consecutive vectors of one row (the combine stages its slot rows
// in shared memory with cp.async first); grids are a multiple of the SM
// count and loop over rows.
//
// Gather: "Round 4 Track C: Prefill MoE Plan ... & Epilogue / Gather Audit",
// section 1 item 4 (rows read as 16-bit values with vector loads and stored
// unchanged, bit for bit).  Combine: "Batched resident MoE experts on Apple
// Silicon: a flat parallel expert pass", section 3 (the same per-token top-k
// summation order).
#include "../../include/moe_prefill.h"
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <atomic>

namespace moe {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kRowWarps = 8;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kCtasPerSm = 8;

__device__ __forceinline__ uint4 ldg_nc(const uint4 *p)
{
    return __ldg(p);
}

// xs[r] = x[srt_tok[r]] for r < R_pad (= offsets[E]); zero rows where srt_tok = -1.
// With side_out, also side_out[r] = side_in[srt_tok[r]] (0 for -1 rows): the
// per-token exponents that go with E4M3 token rows.
__global__ void __launch_bounds__(kRowThreads)
    k_gather(const uint4 *__restrict__ x, int T, int dvec, const int32_t *__restrict__ srt_tok,
             const int32_t *__restrict__ offsets, int E, int64_t cap, uint4 *__restrict__ xs,
             const int32_t *__restrict__ side_in, int32_t *__restrict__ side_out)
{
    pdl_wait();
    const int64_t R = min(int64_t(offsets[E]), cap);
    const int lane = threadIdx.x & 31;
    const int64_t nw = int64_t(gridDim.x) * kRowWarps;
    for (int64_t r = int64_t(blockIdx.x) * kRowWarps + (threadIdx.x >> 5); r < R; r += nw) {
        const int t = srt_tok[r];
        uint4 *dst = xs + r * dvec;
        if (side_out && lane == 0)
            side_out[r] = t >= 0 && t < T ? side_in[t] : 0;
        if (t >= 0 && t < T) {
            const uint4 *src = x + int64_t(t) * dvec;
            int c = lane;
            for (; c + 96 < dvec; c += 128) {
                const uint4 a = ldg_nc(src + c), b = ldg_nc(src + c + 32);
                const uint4 e = ldg_nc(src + c + 64), g = ldg_nc(src + c + 96);
                dst[c] = a;
                dst[c + 32] = b;
                dst[c + 64] = e;
                dst[c + 96] = g;
            }
            for (; c < dvec; c += 32)
                dst[c] = ldg_nc(src + c);
        } else {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int c = lane; c < dvec; c += 32)
                dst[c] = z;
        }
    }
    pdl_launch_dependents();
}

// The gather with E4M3 rows for the gate/up GEMM on E4M3 operands: each
// row's codes are its bf16 values times 2^-e, e the smallest integer with
// max |row| <= 448 * 2^e (0 for zero rows and -1 rows), to the nearest E4M3
// value; xexp[r] = e.  Power-of-two scaling is exact, so this is one
// multiply and one conversion per value.  Two passes over the source row
// (the largest magnitude, then the codes); the second pass reads it from L1.
// With srt_tok = null, row r is x[r] itself (the rows of H for the down
// projection on E4M3 operands).
// nrows >= 0 fixes the row count instead of offsets[E] (the token rows of x).
__global__ void __launch_bounds__(kRowThreads)
    k_gather_e4m3(const uint4 *__restrict__ x, int T, int dvec,
                  const int32_t *__restrict__ srt_tok, const int32_t *__restrict__ offsets,
                  int E, int64_t cap, uint2 *__restrict__ xs8, int32_t *__restrict__ xexp,
                  int64_t nrows)
{
    pdl_wait();
    const int64_t R = nrows >= 0 ? nrows : min(int64_t(offsets[E]), cap);
    const int lane = threadIdx.x & 31;
    const int64_t nw = int64_t(gridDim.x) * kRowWarps;
    for (int64_t r = int64_t(blockIdx.x) * kRowWarps + (threadIdx.x >> 5); r < R; r += nw) {
        const int t = srt_tok ? srt_tok[r] : int(r);
        uint2 *dst = xs8 + r * dvec;
        if (t < 0 || t >= T) {
            for (int c = lane; c < dvec; c += 32)
                dst[c] = make_uint2(0u, 0u);
            if (lane == 0)
                xexp[r] = 0;
            continue;
        }
        const uint4 *src = x + int64_t(t) * dvec;
        uint32_t amax_bits = 0;  // bf16 magnitudes order like their bit patterns
        for (int c = lane; c < dvec; c += 32) {
            const uint4 v = ldg_nc(src + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                amax_bits = max(amax_bits, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, o));
        const float amax = __uint_as_float(amax_bits << 16);
        int e = 0;
        if (amax > 0.0f) {
            e = ilogbf(amax) - 8;  // amax in [448 * 2^(e-1), 2 * 448 * 2^e)
            if (amax > ldexpf(448.0f, e))
                ++e;
        }
        const bool plain = e >= -127 && e <= 126;  // 2^-e a normal fp32
        const float mul = plain ? __uint_as_float(uint32_t(127 - e) << 23) : 0.0f;
        for (int c = lane; c < dvec; c += 32) {
            const uint4 v = ldg_nc(src + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t out[2] = {0u, 0u};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xffff0000u);
                a = plain ? a * mul : ldexpf(a, -e);
                b = plain ? b * mul : ldexpf(b, -e);
                const uint32_t pair =
                    __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
                out[i >> 1] |= pair << (16 * (i & 1));
            }
            dst[c] = make_uint2(out[0], out[1]);
        }
        if (lane == 0)
            xexp[r] = e;
    }
    pdl_launch_dependents();
}

__device__ __forceinline__ void add_bf16x8(float *acc, const uint4 v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16);
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float *acc)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]));
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1]));
        w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}



// Combine with the slot rows staged in shared memory: one warp per (token,
// 512-byte segment), each lane on one 16-byte column; the segment's slot
// rows are copied in groups of kCombSlots with cp.async (16 bytes a lane,
// no registers held while they travel), double-buffered so that the next
// group (of this task or the warp's next task) is in flight while this one
// is added.  Each lane reads back only what it copied itself.  Sum order:
// slot 0, 1, ..., k - 1 in fp32 from zero, one bf16 rounding.
constexpr int kCombWarps = 4;
constexpr int kCombSlots = 4;
constexpr int kCombSmem = kCombWarps * 2 * kCombSlots * 32 * 16;

__device__ __forceinline__ void cp_async16(const void *sdst, const void *gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(sdst))),
                 "l"(gsrc)
                 : "memory");
}

__global__ void __launch_bounds__(kCombWarps * 32)
    k_combine(const uint4 *__restrict__ Ys, const int32_t *__restrict__ pos, int T, int k,
              int dvec, uint4 *__restrict__ y)
{
    extern __shared__ __align__(16) uint4 csm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4 *buf = csm + warp * (2 * kCombSlots * 32);  // [2][kCombSlots][32]
    pdl_wait();
    const int nseg = (dvec + 31) / 32;
    const int ngrp = (k + kCombSlots - 1) / kCombSlots;
    const int64_t ntask = int64_t(T) * nseg;
    const int64_t nw = int64_t(gridDim.x) * kCombWarps;
    int64_t task = int64_t(blockIdx.x) * kCombWarps + warp;
    // copy group gg of task tk into buffer b; returns the mask of its non-skipped slots
    auto issue = [&](int64_t tk, int gg, int b) -> uint32_t {
        const int64_t t = tk / nseg;
        const int c = int(tk - t * nseg) * 32 + lane;
        const int j0 = gg * kCombSlots;
        const int jn = min(kCombSlots, k - j0);
        const int pl = lane < jn ? pos[t * k + j0 + lane] : -1;
        uint32_t m = 0;
#pragma unroll
        for (int s = 0; s < kCombSlots; ++s) {
            const int p = __shfl_sync(kFull, pl, s);
            if (s < jn && p >= 0) {
                m |= 1u << s;
                if (c < dvec)
                    cp_async16(buf + (b * kCombSlots + s) * 32 + lane, Ys + int64_t(p) * dvec + c);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        return m;
    };
    if (task < ntask) {
        int g = 0, b = 0;
        uint32_t mcur = issue(task, 0, 0);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = 0.0f;
        while (true) {
            int64_t ntk = task;
            int ng = g + 1;
            if (ng == ngrp) {
                ng = 0;
                ntk = task + nw;
            }
            const bool more = ntk < ntask;
            uint32_t mnext = 0;
            if (more) {
                mnext = issue(ntk, ng, b ^ 1);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
#pragma unroll
            for (int s = 0; s < kCombSlots; ++s)
                if ((mcur >> s) & 1u)
                    add_bf16x8(acc, buf[(b * kCombSlots + s) * 32 + lane]);
            if (g == ngrp - 1) {
                const int64_t t = task / nseg;
                const int c = int(task - t * nseg) * 32 + lane;
                if (c < dvec)
                    y[t * dvec + c] = pack_bf16x8(acc);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i] = 0.0f;
            }
            if (!more)
                break;
            task = ntk;
            g = ng;
            b ^= 1;
            mcur = mnext;
        }
    }
    pdl_launch_dependents();
}

// Resident combine CTAs per SM on this device (registers decide), once per device.
int combine_ctas_per_sm()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 1;
    const int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0)
        return v;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_combine, kCombWarps * 32, kCombSmem) !=
            cudaSuccess ||
        n <= 0) {
        cudaGetLastError();  // a failed query is not the caller's error
        n = 1;
    }
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace

cudaError_t launch_gather(const void *x, int T, int d, const int32_t *srt_tok,
                          const int32_t *offsets, int E, int64_t cap, void *xs,
                          cudaStream_t stream)
{
    const int dvec = d / 8;
    const int64_t want = (cap + kRowWarps - 1) / kRowWarps;
    const int64_t cap_grid = int64_t(device_sm_count()) * kCtasPerSm;
    const int grid = int(want < 1 ? 1 : (want < cap_grid ? want : cap_grid));
    return launch_pdl(k_gather, dim3(grid), dim3(kRowThreads), 0, stream,
                      static_cast<const uint4 *>(x), T, dvec, srt_tok, offsets, E, cap,
                      static_cast<uint4 *>(xs), static_cast<const int32_t *>(nullptr),
                      static_cast<int32_t *>(nullptr));
}

cudaError_t launch_quant_tokens_e4m3(const void *x, int T, int d, uint8_t *x8, int32_t *texp,
                                     cudaStream_t stream)
{
    const int64_t want = (int64_t(T) + kRowWarps - 1) / kRowWarps;
    const int64_t cap_grid = int64_t(device_sm_count()) * kCtasPerSm;
    const int grid = int(want < 1 ? 1 : (want < cap_grid ? want : cap_grid));
    return launch_pdl(k_gather_e4m3, dim3(grid), dim3(kRowThreads), 0, stream,
                      static_cast<const uint4 *>(x), T, d / 8,
                      static_cast<const int32_t *>(nullptr), static_cast<const int32_t *>(nullptr),
                      0, int64_t(T), reinterpret_cast<uint2 *>(x8), texp, int64_t(T));
}

cudaError_t launch_gather_codes(const uint8_t *x8, const int32_t *texp, int T, int d,
                                const int32_t *srt_tok, const int32_t *offsets, int E,
                                int64_t cap, uint8_t *xs8, int32_t *xexp, cudaStream_t stream)
{
    const int dvec = d / 16;
    const int64_t want = (cap + kRowWarps - 1) / kRowWarps;
    const int64_t cap_grid = int64_t(device_sm_count()) * kCtasPerSm;
    const int grid = int(want < 1 ? 1 : (want < cap_grid ? want : cap_grid));
    return launch_pdl(k_gather, dim3(grid), dim3(kRowThreads), 0, stream,
                      reinterpret_cast<const uint4 *>(x8), T, dvec, srt_tok, offsets, E, cap,
                      reinterpret_cast<uint4 *>(xs8), texp, xexp);
}

cudaError_t launch_gather_e4m3(const void *x, int T, int d, const int32_t *srt_tok,
                               const int32_t *offsets, int E, int64_t cap, uint8_t *xs8,
                               int32_t *xexp, cudaStream_t stream)
{
    const int dvec = d / 8;
    const int64_t want = (cap + kRowWarps - 1) / kRowWarps;
    const int64_t cap_grid = int64_t(device_sm_count()) * kCtasPerSm;
    const int grid = int(want < 1 ? 1 : (want < cap_grid ? want : cap_grid));
    return launch_pdl(k_gather_e4m3, dim3(grid), dim3(kRowThreads), 0, stream,
                      static_cast<const uint4 *>(x), T, dvec, srt_tok, offsets, E, cap,
                      reinterpret_cast<uint2 *>(xs8), xexp, int64_t(-1));
}

cudaError_t launch_rows_e4m3(const void *H, int f, const int32_t *offsets, int E, int64_t cap,
                             uint8_t *H8, int32_t *hexp, cudaStream_t stream)
{
    const int dvec = f / 8;
    const int64_t want = (cap + kRowWarps - 1) / kRowWarps;
    const int64_t cap_grid = int64_t(device_sm_count()) * kCtasPerSm;
    const int grid = int(want < 1 ? 1 : (want < cap_grid ? want : cap_grid));
    return launch_pdl(k_gather_e4m3, dim3(grid), dim3(kRowThreads), 0, stream,
                      static_cast<const uint4 *>(H), int(cap), dvec,
                      static_cast<const int32_t *>(nullptr), offsets, E, cap,
                      reinterpret_cast<uint2 *>(H8), hexp, int64_t(-1));
}

cudaError_t launch_combine(const void *Ys, const int32_t *pos, int T, int k, int d, void *y,
                           cudaStream_t stream)
{
    const int dvec = d / 8;
    const int64_t ntask = int64_t(T) * ((dvec + 31) / 32);
    const int64_t want = (ntask + kCombWarps - 1) / kCombWarps;
    const int64_t cap_grid = int64_t(device_sm_count()) * combine_ctas_per_sm();
    const int grid = int(want < 1 ? 1 : (want < cap_grid ? want : cap_grid));
    return launch_pdl(k_combine, dim3(grid), dim3(kCombWarps * 32), size_t(kCombSmem), stream,
                      static_cast<const uint4 *>(Ys), pos, T, k, dvec, static_cast<uint4 *>(y));
}

}  // namespace moe
