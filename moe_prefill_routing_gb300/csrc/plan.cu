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
//    histogram plus a one-CTA scan, because one CTA cannot use the whole GPU.
//    On GB300 the launch and completion gaps between three small kernels
//    cost more than the work, so chunks of up to 64K entries run the whole
//    plan in ONE launch of a thread-block cluster (16 CTAs
//    where the GPU can place them, else 8; 256 threads each): each CTA counts
//    and ranks its share of the entries, then, through distributed shared
//    memory and hardware cluster barriers, each CTA scans a share of the
//    experts and hands every CTA the first row of each expert for its share
//    of entries.  Larger inputs use the three kernels below.
#include "../../include/moe_prefill.h"
#include "internal.h"
#include "ptx.cuh"

#include <atomic>

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

// ---- one-launch plan for a thread-block cluster --------------------------------

constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;
constexpr int kCSteps = 16;  // 32-entry steps per warp, held in registers
constexpr int kClusterMax = 16;
constexpr int kCEntriesPerCta = kCWarps * kCSteps * 32;  // 4096

constexpr size_t cluster_smem_bytes(int E)
{
    return size_t(kCWarps) * E * sizeof(uint16_t) + 2 * sizeof(int) * size_t(E) +
           (kClusterMax + kCWarps) * sizeof(int);
}

// CTA c of the cluster owns flat entries [c*chunk, (c+1)*chunk), split into
// eight contiguous warp ranges, and experts [c*epc, (c+1)*epc).
// Phase 1: each warp walks its range 32 entries at a time with a running
// count per expert (match_any peers share one update), which gives each
// entry its rank in the warp range; an in-place prefix of the eight warp
// counts per expert turns that into the rank in the CTA range and leaves the
// CTA's count per expert.  Phase 2 (owners, over distributed shared memory):
// the expert's count over all CTAs, its padded size, its first row by a scan
// over the owned experts plus the totals of the CTAs before, the tail fill,
// the tile table, and for every CTA the first row of the expert's entries in
// that CTA.  Phase 3: row = that first row + rank.
__global__ void __launch_bounds__(kCThreads, 1)
    k_plan_cluster(const int32_t *__restrict__ ids, const float *__restrict__ w, int64_t n, int k,
                   int E, int tm, int64_t cap, int64_t chunk, int32_t *__restrict__ offsets,
                   int32_t *__restrict__ counts, int32_t *__restrict__ srt_tok,
                   float *__restrict__ srt_w, int32_t *__restrict__ pos,
                   int32_t *__restrict__ tile_expert, uint32_t *__restrict__ status)
{
    extern __shared__ __align__(16) uint8_t csm[];
    uint16_t *cntw = reinterpret_cast<uint16_t *>(csm);                   // [8 warps][E]
    int *carry = reinterpret_cast<int *>(csm + kCWarps * E * sizeof(uint16_t));  // [E]
    int *rowbase = carry + E;                                             // [E]
    int *tot = rowbase + E;                                               // [16]
    int *warp_tot = tot + kClusterMax;                                    // [8]
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t lane = tid & 31, lt = lanemask_lt();
    const int C = int(cluster_nctarank()), c = int(cluster_ctarank());

    pdl_launch_dependents();
    for (int v = tid; v < E; v += kCThreads)  // 16*E bytes = E vectors of 16
        reinterpret_cast<uint4 *>(cntw)[v] = make_uint4(0u, 0u, 0u, 0u);
    pdl_wait();
    if (c == 0 && tid == 0)
        *status = 0u;

    // ---- phase 1: ranks inside the warp range, then inside the CTA range -------
    const int64_t cta_lo = int64_t(c) * chunk;
    const int64_t cta_hi = min(n, cta_lo + chunk);
    const int64_t wchunk = (chunk + kCWarps - 1) / kCWarps;
    const int64_t w_lo = min(cta_hi, cta_lo + warp * wchunk);
    const int64_t w_hi = min(cta_hi, w_lo + wchunk);
    int my_id[kCSteps], my_rank[kCSteps];
#pragma unroll
    for (int s = 0; s < kCSteps; ++s) {
        const int64_t i = w_lo + s * 32 + lane;
        my_id[s] = i < w_hi ? ids[i] : -1;
        my_rank[s] = -1;
    }
    __syncthreads();  // counters zeroed
    uint16_t *mycnt = cntw + warp * E;
#pragma unroll
    for (int s = 0; s < kCSteps; ++s) {
        if (w_lo + s * 32 < w_hi) {  // the same for the whole warp
            const int id = my_id[s];
            const bool ok = w_lo + s * 32 + lane < w_hi && id >= 0 && id < E;
            const uint32_t key = ok ? uint32_t(id) : (0x80000000u | lane);
            const uint32_t peers = __match_any_sync(kFull, key);
            const int leader = __ffs(peers) - 1;
            int first = 0;
            if (ok && lane == uint32_t(leader)) {
                first = mycnt[id];
                mycnt[id] = uint16_t(first + __popc(peers));
            }
            first = __shfl_sync(kFull, first, leader);
            if (ok)
                my_rank[s] = first + __popc(peers & lt);
            __syncwarp();
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kCThreads) {  // warp counts -> prefix over warps
        int run = 0;
#pragma unroll
        for (int w2 = 0; w2 < kCWarps; ++w2) {
            const int t = cntw[w2 * E + e];
            cntw[w2 * E + e] = uint16_t(run);
            run += t;
        }
        carry[e] = run;
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kCSteps; ++s)
        if (my_rank[s] >= 0)
            my_rank[s] += mycnt[my_id[s]];
    cluster_sync();  // every CTA's counts are final

    // ---- phase 2: owners scan their experts ------------------------------------
    const int epc = (E + C - 1) / C;
    const int J = (epc + kCThreads - 1) / kCThreads;  // experts per thread (1 or 2)
    int cc[2][kClusterMax], ce[2] = {0, 0}, P[2] = {0, 0};
    int tsum = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int li = tid * J + j;
        const int e = c * epc + li;
        const bool own = j < J && li < epc && e < E;
#pragma unroll
        for (int c2 = 0; c2 < kClusterMax; ++c2) {
            cc[j][c2] = 0;
            if (own && c2 < C) {
                cc[j][c2] = dsmem_ld(dsmem_addr(&carry[e], uint32_t(c2)));
                ce[j] += cc[j][c2];
            }
        }
        P[j] = own ? (ce[j] + tm - 1) / tm * tm : 0;
        tsum += P[j];
    }
    int v = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (int(lane) >= o)
            v += t;
    }
    if (lane == 31)
        warp_tot[warp] = v;
    __syncthreads();
    int before = 0, S = 0;
#pragma unroll
    for (int w2 = 0; w2 < kCWarps; ++w2) {
        before += w2 < warp ? warp_tot[w2] : 0;
        S += warp_tot[w2];
    }
    const int t_excl = before + v - tsum;
    if (tid == 0)
        for (int c2 = 0; c2 < C; ++c2)
            dsmem_st(dsmem_addr(&tot[c], uint32_t(c2)), S);
    cluster_sync();  // every CTA knows every CTA's padded total

    int64_t base = 0, total = 0;
    for (int c2 = 0; c2 < C; ++c2) {
        base += c2 < c ? tot[c2] : 0;
        total += tot[c2];
    }
    int64_t off = base + t_excl;
    const int64_t n_tiles_cap = cap / tm;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int li = tid * J + j;
        const int e = c * epc + li;
        if (j < J && li < epc && e < E) {
            offsets[e] = int32_t(off);
            counts[e] = ce[j];
            int64_t run = off;
#pragma unroll
            for (int c2 = 0; c2 < kClusterMax; ++c2) {
                if (c2 < C) {
                    dsmem_st(dsmem_addr(&rowbase[e], uint32_t(c2)), int(run));
                    run += cc[j][c2];
                }
            }
            for (int64_t r = off + ce[j]; r < off + P[j] && r < cap; ++r) {
                srt_tok[r] = -1;
                srt_w[r] = 0.0f;
            }
            for (int64_t t = off / tm; t < (off + P[j]) / tm && t < n_tiles_cap; ++t)
                tile_expert[t] = e;
        }
        off += P[j];
    }
    if (c == C - 1 && tid == 0) {
        offsets[E] = int32_t(total);
        if (total > cap)
            atomicOr(status, MOE_STATUS_OVERFLOW);
    }
    cluster_sync();  // every CTA holds the first row of each expert's entries

    // ---- phase 3: place ----------------------------------------------------------
    bool bad = false;
#pragma unroll
    for (int s = 0; s < kCSteps; ++s) {
        const int64_t i = w_lo + s * 32 + lane;
        if (i < w_hi) {
            const int id = my_id[s];
            if (my_rank[s] >= 0) {
                const int row = rowbase[id] + my_rank[s];
                pos[i] = row;
                if (row < cap) {
                    srt_tok[row] = int32_t(i / k);
                    srt_w[row] = w[i];
                }
            } else {
                pos[i] = -1;
                bad |= id != -1;
            }
        }
    }
    if (__any_sync(kFull, bad) && lane == 0)
        atomicOr(status, MOE_STATUS_BAD_ID);
}

// Cluster size that fits this device (16, else 8, else 0 = none); once per device.
int plan_cluster_size()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    const int v = cached[dev].load(std::memory_order_acquire);
    if (v != 0)
        return v > 0 ? v : 0;
    int chosen = -1;
    bool refused = false;
    const void *fn = reinterpret_cast<const void *>(k_plan_cluster);
    const size_t smem = cluster_smem_bytes(MOE_MAX_EXPERTS);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
        refused = true;
    } else {
        for (int C : {16, 8}) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(C);
            cfg.blockDim = dim3(kCThreads);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = C;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int nclusters = 0;
            if (cudaOccupancyMaxActiveClusters(&nclusters, fn, &cfg) != cudaSuccess) {
                refused = true;
            } else if (nclusters >= 1) {
                chosen = C;
                break;
            }
        }
    }
    if (refused)
        cudaGetLastError();  // a refused cluster size is not the caller's error
    cached[dev].store(chosen, std::memory_order_release);
    return chosen > 0 ? chosen : 0;
}

}  // namespace

cudaError_t launch_plan(const int32_t *ids, const float *w, int T, int k, int E, int tm,
                        int32_t *offsets, int32_t *counts, int32_t *srt_tok, float *srt_w,
                        int32_t *pos, int32_t *tile_expert, int64_t cap, uint32_t *status,
                        int32_t *bcnt, cudaStream_t stream)
{
    const int64_t n = int64_t(T) * k;
    const int C = n > 0 ? plan_cluster_size() : 0;
    if (C > 0 && n <= int64_t(C) * kCEntriesPerCta && E <= C * 2 * kCThreads) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C);
        cfg.blockDim = dim3(kCThreads);
        cfg.dynamicSmemBytes = cluster_smem_bytes(E);
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        const int64_t chunk = (n + C - 1) / C;
        return cudaLaunchKernelEx(&cfg, k_plan_cluster, ids, w, n, k, E, tm, cap, chunk, offsets,
                                  counts, srt_tok, srt_w, pos, tile_expert, status);
    }
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
