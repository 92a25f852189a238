// Routing plan: per-block expert histogram with in-block ranks -> single-CTA
// padded scan with the tail-row fill -> parallel place.
//
// "Round 4 Track C: Prefill MoE Plan (mm_clear + mm_hist + mm_scan + mm_place)
// & Epilogue / Gather Audit", section 1:
//  - item 1: the histogram writes every (block, expert) count, so nothing has
//    to be cleared; the scan, which already knows each expert's first row,
//    count and padded size, writes the -1 tail rows itself;
//  - item 2: the rank of an entry among the earlier entries of its block
//    with the same expert is found without a serial per-thread loop.  Here
//    the histogram kernel finds it while counting: inside a warp,
//    __match_any_sync groups the lanes holding the same expert and popc of
//    the lower peers is the rank; across the block's warps, each warp's
//    per-expert count (shared memory, one byte per expert per warp) is added
//    for the warps before it.  No counter can overflow and nothing depends
//    on top-k.  The place kernel is then a parallel scatter: row = block
//    base of the expert + rank.
//  - item 3: one CTA for the whole histogram+scan was slower than a multi-CTA
//    histogram plus a one-CTA scan; the same split is kept.
#include "../../include/moe_prefill.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kHistThreads = 512;   // 16 warps: one 512-entry sub-block per pass
constexpr int kHistWarps = kHistThreads / 32;
constexpr int kScanThreads = 1024;
constexpr int kPlaceThreads = 256;
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kRankSkipped = -1;  // id -1
constexpr int kRankBadId = -2;    // id outside [-1, E)

// Block b of B flat entries.  For each entry: pos[i] = its rank among the
// earlier entries of the block with the same expert (or -1 / -2 for a
// skipped / bad id).  For each expert: bcnt[e][b] = the block's count.
// The block is walked in sub-blocks of 512 entries, one per thread, so
// ranks keep flat order: earlier sub-blocks (carry), then earlier warps of
// this sub-block (per-warp counts), then lower lanes (match_any peers).
__global__ void __launch_bounds__(kHistThreads)
    k_hist(const int32_t *__restrict__ ids, int64_t n, int E, int64_t B, int stride,
           int32_t *__restrict__ bcnt, int32_t *__restrict__ pos)
{
    extern __shared__ __align__(16) uint8_t hist_smem[];
    uint8_t *cnt = hist_smem;                                  // [16 warps][E] counts
    int *carry = reinterpret_cast<int *>(hist_smem + kHistWarps * E);  // [E]
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t lane = tid & 31, lt = lanemask_lt();
    for (int e = tid; e < E; e += kHistThreads)
        carry[e] = 0;
    pdl_wait();

    const int64_t start = int64_t(blockIdx.x) * B;
    const int64_t end = min(n, start + B);
    for (int64_t s0 = start; s0 < end; s0 += kHistThreads) {
        for (int v = tid; v < E; v += kHistThreads)  // 16*E bytes = E vectors of 16
            reinterpret_cast<uint4 *>(cnt)[v] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        const int64_t i = s0 + tid;
        const int id = i < end ? ids[i] : -1;
        const bool ok = id >= 0 && id < E;
        const uint32_t key = ok ? uint32_t(id) : (0x80000000u | lane);
        const uint32_t peers = __match_any_sync(kFull, key);
        if (ok && lane == uint32_t(__ffs(peers) - 1))
            cnt[warp * E + id] = uint8_t(__popc(peers));
        __syncthreads();
        if (i < end) {
            int r = id == -1 ? kRankSkipped : kRankBadId;
            if (ok) {
                r = carry[id] + __popc(peers & lt);
                for (int w2 = 0; w2 < warp; ++w2)
                    r += cnt[w2 * E + id];
            }
            pos[i] = r;
        }
        __syncthreads();
        for (int e = tid; e < E; e += kHistThreads) {
            int c = 0;
#pragma unroll
            for (int w2 = 0; w2 < kHistWarps; ++w2)
                c += cnt[w2 * E + e];
            carry[e] += c;
        }
        __syncthreads();
    }
    for (int e = tid; e < E; e += kHistThreads)
        bcnt[int64_t(e) * stride + blockIdx.x] = carry[e];
}

__device__ __forceinline__ int take(int b, int nblk, int v)
{
    return b < nblk ? v : 0;
}

// One CTA.  For each expert (ascending id): c_e = sum of its block counts,
// padded size P_e = ceil(c_e / tm) * tm, offsets[e] = exclusive scan of P_e.
// Each expert's row of block counts (int4 loads) is replaced in place by
// block bases (first row of the expert's entries of that block); the tail
// rows [offsets[e] + c_e, offsets[e] + P_e) get srt_tok = -1, srt_w = +0,
// and the tile table gets the expert's tiles.  Resets the status word.
__global__ void __launch_bounds__(kScanThreads)
    k_scan_pad(int32_t *__restrict__ bcnt, int nblk, int stride, int E, int tm, int64_t cap,
               int32_t *__restrict__ offsets, int32_t *__restrict__ counts,
               int32_t *__restrict__ srt_tok, float *__restrict__ srt_w,
               int32_t *__restrict__ tile_expert, uint32_t *__restrict__ status)
{
    __shared__ int warp_incl[kScanThreads / 32];
    pdl_launch_dependents();
    pdl_wait();

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t n_tiles_cap = cap / tm;
    const int nq = stride / 4;
    int64_t carry = 0;  // padded rows of the experts before this slice

    for (int base = 0; base < E; base += kScanThreads) {
        const int e = base + tid;
        int4 *row = reinterpret_cast<int4 *>(bcnt + int64_t(min(e, E - 1)) * stride);
        int c = 0;
        if (e < E) {
#pragma unroll 8
            for (int q = 0; q < nq; ++q) {
                const int4 v = row[q];
                const int b = 4 * q;
                c += take(b, nblk, v.x) + take(b + 1, nblk, v.y) + take(b + 2, nblk, v.z) +
                     take(b + 3, nblk, v.w);
            }
        }
        const int P = e < E ? (c + tm - 1) / tm * tm : 0;

        // block-wide exclusive scan of P (warp shuffles, then warp totals)
        int v = P;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, v, o);
            if (lane >= o)
                v += t;
        }
        if (lane == 31)
            warp_incl[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int wv = warp_incl[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(kFull, wv, o);
                if (lane >= o)
                    wv += t;
            }
            warp_incl[lane] = wv;
        }
        __syncthreads();
        const int64_t off = carry + (v - P) + (warp > 0 ? warp_incl[warp - 1] : 0);
        const int slice_total = warp_incl[kScanThreads / 32 - 1];
        __syncthreads();  // warp_incl is reused by the next slice

        if (e < E) {
            offsets[e] = int32_t(off);
            counts[e] = c;
            int run = int(off);
#pragma unroll 8
            for (int q = 0; q < nq; ++q) {
                const int4 cv = row[q];
                const int b = 4 * q;
                int4 o;
                o.x = run;
                run += take(b, nblk, cv.x);
                o.y = run;
                run += take(b + 1, nblk, cv.y);
                o.z = run;
                run += take(b + 2, nblk, cv.z);
                o.w = run;
                run += take(b + 3, nblk, cv.w);
                row[q] = o;
            }
            for (int64_t r = off + c; r < off + P && r < cap; ++r) {
                srt_tok[r] = -1;
                srt_w[r] = 0.0f;
            }
            for (int64_t t = off / tm; t < (off + P) / tm && t < n_tiles_cap; ++t)
                tile_expert[t] = e;
        }
        carry += slice_total;
    }
    if (tid == 0) {
        offsets[E] = int32_t(carry);
        *status = carry > cap ? MOE_STATUS_OVERFLOW : 0u;
    }
}

// One thread per flat entry: row = base[e][block] + rank (left in pos by
// k_hist); pos[i] = row, srt_tok[row] = token, srt_w[row] = weight (bit copy).
__global__ void __launch_bounds__(kPlaceThreads)
    k_place(const int32_t *__restrict__ ids, const float *__restrict__ w, int64_t n, int k,
            int64_t B, int stride, int64_t cap, const int32_t *__restrict__ bbase,
            int32_t *__restrict__ pos, int32_t *__restrict__ srt_tok, float *__restrict__ srt_w,
            uint32_t *__restrict__ status)
{
    pdl_launch_dependents();
    pdl_wait();
    bool bad = false;
    const int64_t nthreads = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += nthreads) {
        const int r = pos[i];
        if (r >= 0) {
            const int e = ids[i];
            const int row = bbase[int64_t(e) * stride + i / B] + r;
            pos[i] = row;
            if (row < cap) {
                srt_tok[row] = int32_t(i / k);
                srt_w[row] = w[i];
            }
        } else if (r == kRankBadId) {
            bad = true;
            pos[i] = -1;
        }
    }
    if (__any_sync(kFull, bad) && (threadIdx.x & 31) == 0)
        atomicOr(status, MOE_STATUS_BAD_ID);
}

}  // namespace

cudaError_t launch_plan(const int32_t *ids, const float *w, int T, int k, int E, int tm,
                        int32_t *offsets, int32_t *counts, int32_t *srt_tok, float *srt_w,
                        int32_t *pos, int32_t *tile_expert, int64_t cap, uint32_t *status,
                        int32_t *bcnt, cudaStream_t stream)
{
    const int64_t n = int64_t(T) * k;
    const int64_t B = plan_block_entries(n);
    const int nblk = plan_num_blocks(n);
    const int stride = plan_count_stride(n);
    cudaError_t err;
    if (nblk > 0) {
        const size_t hist_smem = size_t(E) * (kHistWarps + sizeof(int));
        err = ensure_smem_limit(reinterpret_cast<const void *>(k_hist), kSlotHist,
                                size_t(MOE_MAX_EXPERTS) * (kHistWarps + sizeof(int)));
        if (err != cudaSuccess)
            return err;
        err = launch_pdl(k_hist, dim3(nblk), dim3(kHistThreads), hist_smem, stream, ids, n, E, B,
                         stride, bcnt, pos);
        if (err != cudaSuccess)
            return err;
    }
    err = launch_pdl(k_scan_pad, dim3(1), dim3(kScanThreads), 0, stream, bcnt, nblk, stride, E,
                     tm, cap, offsets, counts, srt_tok, srt_w, tile_expert, status);
    if (err != cudaSuccess || nblk == 0)
        return err;
    const int64_t want = (n + kPlaceThreads - 1) / kPlaceThreads;
    const int64_t most = int64_t(device_sm_count()) * 8;
    return launch_pdl(k_place, dim3(unsigned(want < most ? want : most)), dim3(kPlaceThreads), 0,
                      stream, ids, w, n, k, B, stride, cap, (const int32_t *)bcnt, pos, srt_tok,
                      srt_w, status);
}

}  // namespace moe
