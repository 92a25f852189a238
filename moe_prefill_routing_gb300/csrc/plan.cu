// Routing plan: per-block expert histogram -> single-CTA padded scan with the
// tail-row fill -> stable place by warp match/ballot rank.
//
// "Round 4 Track C: Prefill MoE Plan (mm_clear + mm_hist + mm_scan + mm_place)
// & Epilogue / Gather Audit", section 1:
//  - item 1: the histogram writes every (block, expert) count, so nothing has
//    to be cleared; the scan, which already knows each expert's first row,
//    count and padded size, writes the -1 tail rows itself;
//  - item 2: the rank of an entry among the earlier entries of its block
//    with the same expert is found without a serial per-thread loop.  Here a
//    warp takes 32 entries at a time: __match_any_sync groups the lanes with
//    the same expert, popc of the lower peers is the rank inside the warp,
//    and one running count per expert (shared memory) carries the rank
//    across the warp's steps.  This does not depend on top-k and has no
//    counter that can overflow.
//  - item 3: one CTA for the whole histogram+scan was slower than a multi-CTA
//    histogram plus a one-CTA scan; the same split is kept.
#include "../../include/moe_prefill.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kHistThreads = 512;
constexpr int kScanThreads = 1024;
constexpr int kPlaceWarps = 4;
constexpr uint32_t kFull = 0xffffffffu;

// bcnt[b][e] = number of entries of block b routed to expert e, for every e.
__global__ void __launch_bounds__(kHistThreads)
    k_hist(const int32_t *__restrict__ ids, int64_t n, int E, int64_t B,
           int32_t *__restrict__ bcnt)
{
    extern __shared__ int hist[];
    pdl_launch_dependents();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        hist[e] = 0;
    __syncthreads();
    pdl_wait();

    const uint32_t lane = threadIdx.x & 31;
    const int64_t start = int64_t(blockIdx.x) * B;
    const int64_t end = min(n, start + B);
    for (int64_t i0 = start; i0 < end; i0 += blockDim.x) {
        const int64_t i = i0 + threadIdx.x;
        const int id = i < end ? ids[i] : -1;
        const bool ok = id >= 0 && id < E;
        // lanes holding the same expert add once, with their number
        const uint32_t key = ok ? uint32_t(id) : (0x80000000u | lane);
        const uint32_t peers = __match_any_sync(kFull, key);
        if (ok && lane == uint32_t(__ffs(peers) - 1))
            atomicAdd(&hist[id], __popc(peers));
    }
    __syncthreads();
    int32_t *row = bcnt + int64_t(blockIdx.x) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        row[e] = hist[e];
}

// One CTA.  For each expert (ascending id): c_e = sum of its block counts,
// padded size P_e = ceil(c_e / tm) * tm, offsets[e] = exclusive scan of P_e.
// The block counts are replaced in place by block bases (first row of the
// expert's entries of that block), the tail rows [offsets[e] + c_e,
// offsets[e] + P_e) get srt_tok = -1 and srt_w = +0, and the tile table gets
// the expert's tiles.  Resets the status word.
__global__ void __launch_bounds__(kScanThreads)
    k_scan_pad(int32_t *__restrict__ bcnt, int nblk, int E, int tm, int64_t cap,
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
    int64_t carry = 0;  // padded rows of the experts before this slice

    for (int base = 0; base < E; base += kScanThreads) {
        const int e = base + tid;
        int c = 0;
        if (e < E)
            for (int b = 0; b < nblk; ++b)
                c += bcnt[int64_t(b) * E + e];
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
            int64_t run = off;
            for (int b = 0; b < nblk; ++b) {
                const int64_t idx = int64_t(b) * E + e;
                const int cnt = bcnt[idx];
                bcnt[idx] = int32_t(run);
                run += cnt;
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

// One warp per block of B entries, 32 entries per step in flat order.
// row(i) = base[b][e] + (entries of block b before i with expert e).
__global__ void __launch_bounds__(kPlaceWarps * 32)
    k_place(const int32_t *__restrict__ ids, const float *__restrict__ w, int64_t n, int k,
            int E, int64_t B, int nblk, int64_t cap, const int32_t *__restrict__ bbase,
            int32_t *__restrict__ pos, int32_t *__restrict__ srt_tok,
            float *__restrict__ srt_w, uint32_t *__restrict__ status)
{
    extern __shared__ int run_all[];  // kPlaceWarps x E running rows
    pdl_launch_dependents();
    pdl_wait();

    const uint32_t lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int b = blockIdx.x * kPlaceWarps + warp;
    if (b >= nblk)
        return;
    int *run = run_all + warp * E;
    for (int e = lane; e < E; e += 32)
        run[e] = bbase[int64_t(b) * E + e];
    __syncwarp();

    const uint32_t lt = lanemask_lt();
    const int64_t start = int64_t(b) * B;
    const int64_t end = min(n, start + B);
    bool bad = false;

    int64_t i = start + lane;
    int id_next = i < end ? ids[i] : -1;
    float w_next = i < end ? w[i] : 0.0f;
    for (int64_t i0 = start; i0 < end; i0 += 32, i += 32) {
        const bool valid = i < end;
        const int id = id_next;
        const float wi = w_next;
        // fetch the next step's entry before working on this one
        const int64_t in = i + 32;
        id_next = in < end ? ids[in] : -1;
        w_next = in < end ? w[in] : 0.0f;

        const bool ok = valid && id >= 0 && id < E;
        bad |= valid && (id < -1 || id >= E);
        const uint32_t key = ok ? uint32_t(id) : (0x80000000u | lane);
        const uint32_t peers = __match_any_sync(kFull, key);
        const int leader = __ffs(peers) - 1;
        int first = 0;
        if (ok && lane == uint32_t(leader)) {
            first = run[id];
            run[id] = first + __popc(peers);
        }
        first = __shfl_sync(kFull, first, leader);
        if (ok) {
            const int row = first + __popc(peers & lt);
            pos[i] = row;
            if (row < cap) {
                srt_tok[row] = int32_t(i / k);
                srt_w[row] = wi;
            }
        } else if (valid) {
            pos[i] = -1;
        }
        __syncwarp();
    }
    if (__any_sync(kFull, bad) && lane == 0)
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
    cudaError_t err;
    if (nblk > 0) {
        const size_t hist_smem = size_t(E) * sizeof(int);
        err = launch_pdl(k_hist, dim3(nblk), dim3(kHistThreads), hist_smem, stream, ids, n, E,
                         B, bcnt);
        if (err != cudaSuccess)
            return err;
    }
    err = launch_pdl(k_scan_pad, dim3(1), dim3(kScanThreads), 0, stream, bcnt, nblk, E, tm,
                     cap, offsets, counts, srt_tok, srt_w, tile_expert, status);
    if (err != cudaSuccess || nblk == 0)
        return err;
    const size_t place_smem = size_t(kPlaceWarps) * E * sizeof(int);
    err = ensure_smem_limit(reinterpret_cast<const void *>(k_place), kSlotPlace,
                            size_t(kPlaceWarps) * MOE_MAX_EXPERTS * sizeof(int));
    if (err != cudaSuccess)
        return err;
    return launch_pdl(k_place, dim3((nblk + kPlaceWarps - 1) / kPlaceWarps),
                      dim3(kPlaceWarps * 32), place_smem, stream, ids, w, n, k, E, B, nblk,
                      cap, (const int32_t *)bcnt, pos, srt_tok, srt_w, status);
}

}  // namespace moe
