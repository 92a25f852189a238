// Routing plan: per-expert counts, an exclusive scan padded to tm with the
// tail rows filled, and a stable place.
//
// "Round 4 Track C: Prefill MoE Plan (mm_clear + mm_hist + mm_scan + mm_place)
// & Epilogue / Gather Audit", section 1:
//  - item 1: every (block, expert) count is written, so nothing has to be
//    cleared; the scan, which knows each expert's first row, count and
//    padded size, writes the -1 tail rows itself;
//  - item 2: the rank of an entry among the earlier entries of its block
//    with the same expert is found without a serial per-thread loop: each
//    warp walks a contiguous range 32 entries at a time with a running count
//    per expert in shared memory; the lanes that hold the same expert are
//    grouped (through per-warp lane words in shared memory, ballots or
//    __match_any_sync, see warp_walk) and popc of the lower peers gives the
//    rank inside a step; the warps' counts, prefixed over the warps, place
//    each warp's range after the earlier ones.  No counter can overflow and
//    nothing depends on top-k;
//  - item 3: one CTA for the whole histogram+scan was slower than a
//    multi-CTA histogram plus a one-CTA scan, because one CTA cannot use the
//    whole GPU.  On GB300 the launch and completion gaps between small
//    kernels cost more than the work, so chunks of up to 64K entries run the
//    whole plan in ONE launch of a thread-block cluster (16 CTAs where the
//    GPU can place them, else 8; 256 threads each): each CTA counts and
//    ranks its share, then, through distributed shared memory and hardware
//    cluster barriers, each CTA scans a share of the experts and hands every
//    CTA the first row of each expert for its share of entries.
// Larger inputs, where the plan is bound by its HBM traffic, run four
// kernels over blocks of 4096 entries, chained with programmatic dependent
// launch: count (each block's count per expert), column scan (per expert,
// the rows of the earlier blocks of the same group of 256 blocks, and each
// group's total), expert scan (the groups' totals prefixed, offsets, tail
// rows), place (the ranks walked again, in registers, the scatter and the
// tile table).
// The ranks are recomputed rather than stored between the passes, so the
// entries are read twice and pos, srt_tok and srt_w written once.
#include "../../include/moe_prefill.h"
#include "internal.h"
#include "ptx.cuh"

#include <atomic>

namespace moe {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

// ---- multi-kernel plan for large inputs ------------------------------------------

constexpr int kPThreads = 256;  // 8 warps, each walking 16 steps of 32 entries
constexpr int kPWarps = kPThreads / 32;
constexpr int kPSteps = 16;
static_assert(kPWarps * kPSteps * 32 == kPlanBlockEntries, "entries per block");
constexpr int kColThreads = 1024;  // column scan: 32 warps x 32 experts
constexpr int kScanThreads = 1024;

// 16 * E bytes of per-warp 16-bit counters: E vectors of 16 bytes.
__device__ __forceinline__ void zero_warp_counts(uint16_t *cntw, int E)
{
    for (int v = threadIdx.x; v < E; v += kPThreads)
        reinterpret_cast<uint4 *>(cntw)[v] = make_uint4(0u, 0u, 0u, 0u);
}

// Count: bcnt[b][e] = entries of block b (kPlanBlockEntries flat entries)
// routed to expert e.  Only the totals matter here, so shared-memory atomics
// count (the order of the adds does not change a sum of ones).  A CTA counts
// blocks blockIdx.x, + gridDim.x, ...; the next block's ids are loaded while
// the current block's counts are written out.
constexpr int kCountCtasPerSm = 8;

__global__ void __launch_bounds__(kPThreads)
    k_count(const int32_t *__restrict__ ids, int64_t n, int nblk, int E,
            int32_t *__restrict__ bcnt)
{
    extern __shared__ __align__(16) uint8_t psm[];
    int *cnt = reinterpret_cast<int *>(psm);  // [E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    for (int e = threadIdx.x; e < E; e += kPThreads)
        cnt[e] = 0;
    pdl_wait();
    int id[kPSteps];
    auto load = [&](int b) {
        const int64_t lo = int64_t(b) * kPlanBlockEntries + warp * kPSteps * 32;
        const int64_t hi = min(n, lo + kPSteps * 32);
#pragma unroll
        for (int s = 0; s < kPSteps; ++s) {
            const int64_t i = lo + s * 32 + lane;
            id[s] = i < hi ? ids[i] : -1;
        }
    };
    load(blockIdx.x);
    for (int b = blockIdx.x; b < nblk; b += gridDim.x) {
        __syncthreads();  // counters zero
#pragma unroll
        for (int s = 0; s < kPSteps; ++s)  // out-of-range entries were loaded as -1
            if (id[s] >= 0 && id[s] < E)
                atomicAdd(&cnt[id[s]], 1);
        if (b + int(gridDim.x) < nblk)
            load(b + gridDim.x);
        __syncthreads();
        int32_t *row = bcnt + int64_t(b) * E;
        for (int e = threadIdx.x; e < E; e += kPThreads) {
            row[e] = cnt[e];
            cnt[e] = 0;
        }
    }
}

// Column scan, per group of kPlanGroupBlocks blocks and 32 experts per CTA
// (grid: expert slices x groups): bcnt[b][e] <- entries of expert e in the
// group's blocks before b, and gsum[g][e] = the group's total.  Warp w sums
// a contiguous segment of the group's blocks, the segment sums are prefixed
// in shared memory, and each warp rewrites its segment.  Rows are read 32
// experts (128 bytes) at a time.
__global__ void __launch_bounds__(kColThreads)
    k_colscan(int32_t *__restrict__ bcnt, int nblk, int E, int32_t *__restrict__ gsum)
{
    __shared__ int seg_sum[kColThreads / 32][32];
    pdl_launch_dependents();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 32 + lane;
    const bool valid = e < E;
    const int g0 = blockIdx.y * kPlanGroupBlocks;
    const int gn = min(nblk - g0, kPlanGroupBlocks);
    const int seg = (gn + kColThreads / 32 - 1) / (kColThreads / 32);
    const int b0 = g0 + min(gn, warp * seg), b1 = g0 + min(gn, (warp + 1) * seg);
    int sum = 0;
    if (valid) {
#pragma unroll 8
        for (int b = b0; b < b1; ++b)
            sum += bcnt[int64_t(b) * E + e];
    }
    seg_sum[warp][lane] = sum;
    __syncthreads();
    int run = 0, total = 0;
    for (int w2 = 0; w2 < kColThreads / 32; ++w2) {
        run += w2 < warp ? seg_sum[w2][lane] : 0;
        total += seg_sum[w2][lane];
    }
    if (valid) {
#pragma unroll 8
        for (int b = b0; b < b1; ++b) {
            const int64_t i = int64_t(b) * E + e;
            const int v = bcnt[i];
            bcnt[i] = run;
            run += v;
        }
        if (warp == 0)
            gsum[int64_t(blockIdx.y) * E + e] = total;
    }
}

// Expert scan (one CTA): counts[e] = the sum of the groups' totals, each
// total replaced by the rows of e in the earlier groups; offsets[e] = sum
// over e' < e of counts[e'] rounded up to tm, offsets[E] = R_pad; the tail
// rows [offsets[e] + counts[e], offsets[e + 1]) get srt_tok = -1 and srt_w =
// +0; with fill_tiles (no place kernel follows, i.e. no entries)
// tile_expert[t] = e for the tiles of e.  Resets the status word (the place
// adds bad-id bits after).
__global__ void __launch_bounds__(kScanThreads)
    k_scan_experts(int32_t *__restrict__ gsum, int ngroups, int32_t *__restrict__ counts, int E,
                   int tm, int64_t cap, int32_t *__restrict__ offsets,
                   int32_t *__restrict__ srt_tok, float *__restrict__ srt_w,
                   int32_t *__restrict__ tile_expert, uint32_t *__restrict__ status,
                   bool fill_tiles)
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
        if (e < E) {
            for (int g0 = 0; g0 < ngroups; g0 += 16) {  // 16 loads in flight, then the stores
                int t[16];
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    t[u] = g0 + u < ngroups ? gsum[int64_t(g0 + u) * E + e] : 0;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    if (g0 + u < ngroups)
                        gsum[int64_t(g0 + u) * E + e] = c;
                    c += t[u];
                }
            }
            counts[e] = c;
        }
        const int P = (c + tm - 1) / tm * tm;
        int v = P;  // block-wide exclusive scan: warp shuffles, then warp totals
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
            for (int64_t r = off + c; r < off + P && r < cap; ++r) {
                srt_tok[r] = -1;
                srt_w[r] = 0.0f;
            }
            if (fill_tiles)
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

// Division of a flat index (< 2^31) by k through one multiply-high, the
// method of Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication" (PLDI 1994), section 4: with l = ceil(log2 k) and
// m = floor(2^32 (2^l - k) / k) + 1, n / k = (t + ((n - t) >> min(l, 1)))
// >> max(l - 1, 0) for t = mulhi(m, n), exact for every 32-bit n.
struct DivK {
    uint32_t m;
    int s1, s2;
};

DivK make_divk(uint32_t k)
{
    int l = 0;
    while ((uint64_t(1) << l) < k)
        ++l;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - k)) / k + 1;
    return DivK{uint32_t(m), l < 1 ? l : 1, l > 1 ? l - 1 : 0};
}

__device__ __forceinline__ uint32_t div_k(uint32_t n, DivK d)
{
    const uint32_t t = __umulhi(d.m, n);
    return (t + ((n - t) >> d.s1)) >> d.s2;
}

// A warp walks its range 32 entries (one step) at a time; the lanes of a
// step that hold the same expert are found in one of three ways.  kWalkOr
// (E <= kOrWalkMaxE): each warp keeps a 32-bit word per expert in shared
// memory, every lane ORs its bit into its expert's word and reads back the
// whole set (one shared atomic and one load per step).  Above that the
// per-warp words would not fit: kWalkBallot intersects one ballot per bit of
// the id (plus one for validity), kWalkMatch uses __match_any_sync; measured,
// the first is faster in the place kernel of large inputs, the second in the
// one-launch cluster plan.
constexpr int kWalkOr = 0, kWalkBallot = 1, kWalkMatch = 2;
constexpr int kOrWalkMaxE = 1024;
constexpr int kMaxIdBits = 12;  // ids < MOE_MAX_EXPERTS = 4096
static_assert(MOE_MAX_EXPERTS <= (1 << kMaxIdBits), "id bits");

// Place (each CTA loops over blocks, the grid being the CTAs the GPU holds
// at once): block b walks its entries again (same ranges, same ranks),
// prefixes the warps' counts per expert, and gives each entry row = offsets[e] +
// (rows of e in earlier blocks) + (its rank among the block's entries of e).
// A block's entries of one expert fill consecutive rows, so their rows,
// weights and block-local indices are first put in shared memory in expert
// order and then written out run after run: neighbouring lanes write
// neighbouring rows of srt_tok and srt_w (pos keeps flat order).  The kernel
// also fills the tile table: tile t belongs to the expert whose rows hold
// row t * tm.
constexpr size_t place_smem_bytes(int E, bool or_walk)
{
    return size_t(kPWarps) * E * (sizeof(uint16_t) + (or_walk ? sizeof(uint32_t) : 0)) +
           size_t(3 * E + 2) * sizeof(int) +
           size_t(kPlanBlockEntries) * (sizeof(int) + sizeof(float) + sizeof(uint16_t));
}

// Rank of each entry of this warp's range [lo, hi) (at most kPSteps * 32
// entries) among the earlier entries of the range with the same expert, with
// running counts per expert in mycnt (and, for kWalkOr, the per-expert lane
// words in mypm, zero between steps).  v holds the ids on entry and, on
// exit, (rank << 16 | id) for a valid id, -1 otherwise; bad is set for an id
// outside [0, E) other than -1.
template <int WALK>
__device__ __forceinline__ void warp_walk(int (&v)[kPSteps], int64_t lo, int64_t hi, int E,
                                          uint16_t *mycnt, uint32_t *mypm, bool &bad)
{
    const uint32_t lane = threadIdx.x & 31, lt = lanemask_lt();
    const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;
#pragma unroll
    for (int s = 0; s < kPSteps; ++s) {
        if (lo + s * 32 < hi) {  // the same for the whole warp
            const bool in = lo + s * 32 + lane < hi;
            const int e = v[s];
            const bool ok = in && e >= 0 && e < E;
            bad |= in && !ok && e != -1;
            uint32_t peers;
            if (WALK == kWalkOr) {
                if (ok)
                    atomicOr(&mypm[e], 1u << lane);
                __syncwarp();
                peers = ok ? mypm[e] : (1u << lane);
            } else if (WALK == kWalkMatch) {
                peers = __match_any_sync(kFull, ok ? uint32_t(e) : (0x80000000u | lane));
            } else {
                const uint32_t vb = __ballot_sync(kFull, ok);
                peers = ok ? vb : (1u << lane);
#pragma unroll
                for (int bit = 0; bit < kMaxIdBits; ++bit) {
                    if (bit < nbits) {  // the same for the whole warp
                        const bool set = (uint32_t(e) >> bit) & 1u;
                        const uint32_t bb = __ballot_sync(kFull, set);
                        peers &= set ? bb : ~bb;
                    }
                }
            }
            // every lane reads its expert's running count (lanes of one
            // expert read the same word), then the lowest of them moves it on
            const int first = ok ? int(mycnt[e]) : 0;
            __syncwarp();
            if (ok && lane == uint32_t(__ffs(peers) - 1)) {
                mycnt[e] = uint16_t(first + __popc(peers));
                if (WALK == kWalkOr)
                    mypm[e] = 0u;
            }
            v[s] = ok ? ((first + __popc(peers & lt)) << 16) | e : -1;
            __syncwarp();
        } else {
            v[s] = -1;
        }
    }
}

// 80 registers a thread: three CTAs of 256 threads per SM.
template <bool OR_WALK>
__global__ void __launch_bounds__(kPThreads, 3)
    k_place_blocks(const int32_t *__restrict__ ids, const float *__restrict__ w, int64_t n,
                   DivK kd, int E, int tm, int64_t cap, const int32_t *__restrict__ offsets,
                   const int32_t *__restrict__ bcnt, int nblk, int32_t *__restrict__ pos,
                   int32_t *__restrict__ srt_tok, float *__restrict__ srt_w,
                   int32_t *__restrict__ tile_expert, uint32_t *__restrict__ status)
{
    extern __shared__ __align__(16) uint8_t psm[];
    uint16_t *cntw = reinterpret_cast<uint16_t *>(psm);  // [8][E]
    uint32_t *pm = reinterpret_cast<uint32_t *>(psm + kPWarps * E * sizeof(uint16_t));  // [8][E]
    int *rowbase = reinterpret_cast<int *>(
        psm + kPWarps * E * (sizeof(uint16_t) + (OR_WALK ? sizeof(uint32_t) : 0)));  // [E]
    int *loc = rowbase + E;      // [E + 1] block-local first slot of each expert
    int *s_off = loc + E + 1;    // [E + 1] offsets
    int *s_row = s_off + E + 1;  // [4096] the block's entries in expert order: row,
    float *s_w = reinterpret_cast<float *>(s_row + kPlanBlockEntries);       // weight,
    uint16_t *s_li = reinterpret_cast<uint16_t *>(s_w + kPlanBlockEntries);  // local index
    __shared__ int warp_tot[kPWarps];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();
    zero_warp_counts(cntw, E);
    if (OR_WALK)
        for (int v = tid; v < 2 * E; v += kPThreads)
            reinterpret_cast<uint4 *>(pm)[v] = make_uint4(0u, 0u, 0u, 0u);
    // everything is read after the wait: this launch may begin before the
    // count kernel's own wait for whatever wrote the ids has ended
    pdl_wait();
    int v[kPSteps];
    float wv[kPSteps];
    auto load_ids = [&](int bb) {
        const int64_t blo = int64_t(bb) * kPlanBlockEntries + warp * kPSteps * 32;
        const int64_t bhi = min(n, blo + kPSteps * 32);
#pragma unroll
        for (int s = 0; s < kPSteps; ++s) {
            const int64_t i = blo + s * 32 + lane;
            v[s] = i < bhi ? ids[i] : -1;
        }
    };
    // CTA c places blocks c, c + gridDim.x, ... (grid: the CTAs the GPU holds
    // at once); the next block's ids are loaded while this block's runs are
    // written out
    load_ids(blockIdx.x);
    for (int b = blockIdx.x; b < nblk; b += gridDim.x) {
        const int64_t blk_lo = int64_t(b) * kPlanBlockEntries;
        const int64_t lo = blk_lo + warp * kPSteps * 32;
        const int64_t hi = min(n, lo + kPSteps * 32);
#pragma unroll
        for (int s = 0; s < kPSteps; ++s) {
            const int64_t i = lo + s * 32 + lane;
            wv[s] = i < hi ? w[i] : 0.0f;
        }
        __syncthreads();
        bool bad = false;
        warp_walk<OR_WALK ? kWalkOr : kWalkBallot>(v, lo, hi, E, cntw + warp * E, pm + warp * E,
                                                   bad);
        if (__any_sync(kFull, bad) && lane == 0)
            atomicOr(status, MOE_STATUS_BAD_ID);
        __syncthreads();
        // per expert: warp counts -> prefix over warps, the block's total, and
        // an exclusive scan of the totals over the experts (contiguous runs of J
        // experts per thread, then warp shuffles and warp totals)
        const int32_t *brow = bcnt + int64_t(b) * E;
        const int32_t *grow = bcnt + (int64_t(nblk) + b / kPlanGroupBlocks) * E;
        const int J = (E + kPThreads - 1) / kPThreads;
        const int e0 = min(E, tid * J), e1 = min(E, e0 + J);
        int tsum = 0;
        for (int e = e0; e < e1; ++e) {
            int run = 0;
#pragma unroll
            for (int w2 = 0; w2 < kPWarps; ++w2) {
                const int t = cntw[w2 * E + e];
                cntw[w2 * E + e] = uint16_t(run);
                run += t;
            }
            loc[e] = run;  // the block's count for now
            tsum += run;
            s_off[e] = offsets[e];
            rowbase[e] = s_off[e] + grow[e] + brow[e];
        }
        if (tid == 0)
            s_off[E] = offsets[E];
        int sc = tsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, sc, o);
            if (lane >= o)
                sc += t;
        }
        if (lane == 31)
            warp_tot[warp] = sc;
        __syncthreads();
        int slot0 = sc - tsum, total = 0;
#pragma unroll
        for (int w2 = 0; w2 < kPWarps; ++w2) {
            slot0 += w2 < warp ? warp_tot[w2] : 0;
            total += warp_tot[w2];
        }
        for (int e = e0; e < e1; ++e) {
            const int c = loc[e];
            loc[e] = slot0;
            slot0 += c;
        }
        __syncthreads();
        // each entry: its rank in the block, pos in flat order, its sorted slot
        const uint16_t *mycnt = cntw + warp * E;
#pragma unroll
        for (int s = 0; s < kPSteps; ++s) {
            const int64_t i = lo + s * 32 + lane;
            if (i < hi) {
                const int p = v[s];
                if (p >= 0) {
                    const int e = p & 0xffff, r = mycnt[e] + (p >> 16);
                    const int row = rowbase[e] + r;
                    pos[i] = row;
                    const int slot = loc[e] + r;
                    s_row[slot] = row;
                    s_w[slot] = wv[s];
                    s_li[slot] = uint16_t(i - blk_lo);
                } else {
                    pos[i] = -1;
                }
            }
        }
        __syncthreads();
        zero_warp_counts(cntw, E);  // the lane words are left zero by every step
        if (b + int(gridDim.x) < nblk)
            load_ids(b + gridDim.x);
        for (int j = tid; j < total; j += kPThreads) {
            const int row = s_row[j];
            if (row < cap) {
                srt_tok[row] = int32_t(div_k(uint32_t(blk_lo + s_li[j]), kd));
                srt_w[row] = s_w[j];
            }
        }
    }
    // tile table, spread over the grid
    const int64_t R = min(int64_t(s_off[E]), cap);
    const int64_t ntiles = R / tm;
    for (int64_t t = int64_t(blockIdx.x) * kPThreads + tid; t < ntiles;
         t += int64_t(gridDim.x) * kPThreads) {
        const int64_t r = t * tm;
        int l = 0, h = E - 1;  // the last e with offsets[e] <= r
        while (l < h) {
            const int mid = (l + h + 1) >> 1;
            if (s_off[mid] <= r)
                l = mid;
            else
                h = mid - 1;
        }
        tile_expert[t] = l;
    }
}

// ---- one-launch plan for a thread-block cluster --------------------------------

constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;
constexpr int kCSteps = 16;  // 32-entry steps per warp, held in registers
constexpr int kClusterMax = 16;
constexpr int kCEntriesPerCta = kCWarps * kCSteps * 32;  // 4096
static_assert(kCSteps == kPSteps, "the cluster plan walks with warp_walk");

constexpr size_t cluster_smem_bytes(int E, bool or_walk)
{
    return size_t(kCWarps) * E * (sizeof(uint16_t) + (or_walk ? sizeof(uint32_t) : 0)) +
           2 * sizeof(int) * size_t(E) + (kClusterMax + kCWarps) * sizeof(int);
}

// CTA c of the cluster owns flat entries [c*chunk, (c+1)*chunk), split into
// eight contiguous warp ranges, and experts [c*epc, (c+1)*epc).
// Phase 1: each warp walks its range 32 entries at a time with a running
// count per expert (the lanes of one expert share one update), which gives
// each entry its rank in the warp range; an in-place prefix of the eight
// warp counts per expert turns that into the rank in the CTA range and
// leaves the CTA's count per expert.  Phase 2 (owners, over distributed shared memory):
// the expert's count over all CTAs, its padded size, its first row by a scan
// over the owned experts plus the totals of the CTAs before, the tail fill,
// the tile table, and for every CTA the first row of the expert's entries in
// that CTA.  Phase 3: row = that first row + rank.
template <bool OR_WALK>
__global__ void __launch_bounds__(kCThreads, 1)
    k_plan_cluster(const int32_t *__restrict__ ids, const float *__restrict__ w, int64_t n,
                   DivK kd, int E, int tm, int64_t cap, int64_t chunk, int32_t *__restrict__ offsets,
                   int32_t *__restrict__ counts, int32_t *__restrict__ srt_tok,
                   float *__restrict__ srt_w, int32_t *__restrict__ pos,
                   int32_t *__restrict__ tile_expert, uint32_t *__restrict__ status)
{
    extern __shared__ __align__(16) uint8_t csm[];
    uint16_t *cntw = reinterpret_cast<uint16_t *>(csm);                   // [8 warps][E]
    uint32_t *pm = reinterpret_cast<uint32_t *>(csm + kCWarps * E * sizeof(uint16_t));  // [8][E]
    int *carry = reinterpret_cast<int *>(
        csm + kCWarps * E * (sizeof(uint16_t) + (OR_WALK ? sizeof(uint32_t) : 0)));  // [E]
    int *rowbase = carry + E;                                             // [E]
    int *tot = rowbase + E;                                               // [16]
    int *warp_tot = tot + kClusterMax;                                    // [8]
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t lane = tid & 31, lt = lanemask_lt();
    const int C = int(cluster_nctarank()), c = int(cluster_ctarank());

    pdl_launch_dependents();
    for (int v = tid; v < (OR_WALK ? 3 : 1) * E; v += kCThreads)  // 16 (48) * E bytes
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
    int ent[kCSteps];  // ids, then (rank << 16 | id) or -1
    float wv[kCSteps];
#pragma unroll
    for (int s = 0; s < kCSteps; ++s) {
        const int64_t i = w_lo + s * 32 + lane;
        ent[s] = i < w_hi ? ids[i] : -1;
        wv[s] = i < w_hi ? w[i] : 0.0f;
    }
    __syncthreads();  // counters zeroed
    uint16_t *mycnt = cntw + warp * E;
    bool bad = false;  // reported after the cluster barriers (CTA 0 resets the status)
    warp_walk<OR_WALK ? kWalkOr : kWalkMatch>(ent, w_lo, w_hi, E, mycnt, pm + warp * E, bad);
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
        if (ent[s] >= 0)
            ent[s] += int(mycnt[ent[s] & 0xffff]) << 16;
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
#pragma unroll
    for (int s = 0; s < kCSteps; ++s) {
        const int64_t i = w_lo + s * 32 + lane;
        if (i < w_hi) {
            const int p = ent[s];
            if (p >= 0) {
                const int row = rowbase[p & 0xffff] + (p >> 16);
                pos[i] = row;
                if (row < cap) {
                    srt_tok[row] = int32_t(div_k(uint32_t(i), kd));
                    srt_w[row] = wv[s];
                }
            } else {
                pos[i] = -1;
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
    // both instantiations get their opt-in sizes; the larger one decides
    const void *fn_or = reinterpret_cast<const void *>(k_plan_cluster<true>);
    const void *fn = reinterpret_cast<const void *>(k_plan_cluster<false>);
    const size_t smem_or = cluster_smem_bytes(kOrWalkMaxE, true);
    const size_t smem = cluster_smem_bytes(MOE_MAX_EXPERTS, false);
    static_assert(cluster_smem_bytes(kOrWalkMaxE, true) <= cluster_smem_bytes(MOE_MAX_EXPERTS, false),
                  "the occupancy check below covers both instantiations");
    if (cudaFuncSetAttribute(fn_or, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_or)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fn_or, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
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
        const bool or_walk = E <= kOrWalkMaxE;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C);
        cfg.blockDim = dim3(kCThreads);
        cfg.dynamicSmemBytes = cluster_smem_bytes(E, or_walk);
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
        return cudaLaunchKernelEx(&cfg, or_walk ? k_plan_cluster<true> : k_plan_cluster<false>,
                                  ids, w, n, make_divk(uint32_t(k)), E, tm, cap, chunk, offsets,
                                  counts, srt_tok, srt_w, pos, tile_expert, status);
    }
    const int nblk = plan_num_blocks(n);
    const int ngroups = plan_num_groups(nblk);
    int32_t *gsum = bcnt + int64_t(nblk) * E;  // [ngroups][E] after the blocks' rows
    const size_t cnt_smem = size_t(E) * sizeof(int);
    const bool or_walk = E <= kOrWalkMaxE;
    const void *place_fn = or_walk ? reinterpret_cast<const void *>(k_place_blocks<true>)
                                   : reinterpret_cast<const void *>(k_place_blocks<false>);
    // the opt-in size covers every E this instantiation takes
    const size_t max_place_smem = or_walk ? place_smem_bytes(kOrWalkMaxE, true)
                                          : place_smem_bytes(MOE_MAX_EXPERTS, false);
    cudaError_t err;
    if (nblk > 0) {
        err = ensure_smem_limit(place_fn, or_walk ? kSlotPlaceOr : kSlotPlace, max_place_smem);
        if (err == cudaSuccess)
            err = launch_pdl(k_count, dim3(std::min(nblk, device_sm_count() * kCountCtasPerSm)),
                             dim3(kPThreads), cnt_smem, stream, ids, n, nblk, E, bcnt);
        if (err == cudaSuccess)
            err = launch_pdl(k_colscan, dim3((E + 31) / 32, ngroups), dim3(kColThreads), 0, stream,
                             bcnt, nblk, E, gsum);
        if (err != cudaSuccess)
            return err;
    }
    err = launch_pdl(k_scan_experts, dim3(1), dim3(kScanThreads), 0, stream, gsum, ngroups,
                     counts, E, tm, cap, offsets, srt_tok, srt_w, tile_expert, status, nblk == 0);
    if (err != cudaSuccess || nblk == 0)
        return err;
    int per_sm = 0;  // resident place CTAs per SM for this E (shared memory and registers)
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, or_walk ? k_place_blocks<true> : k_place_blocks<false>, kPThreads,
            place_smem_bytes(E, or_walk)) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();  // a failed query is not the caller's error
        per_sm = 1;
    }
    const int pgrid = std::min(nblk, device_sm_count() * per_sm);
    return launch_pdl(or_walk ? k_place_blocks<true> : k_place_blocks<false>, dim3(pgrid),
                      dim3(kPThreads), place_smem_bytes(E, or_walk), stream, ids, w, n,
                      make_divk(uint32_t(k)), E, tm, cap, static_cast<const int32_t *>(offsets),
                      static_cast<const int32_t *>(bcnt), nblk, pos, srt_tok, srt_w,
                      tile_expert, status);
}

}  // namespace moe
