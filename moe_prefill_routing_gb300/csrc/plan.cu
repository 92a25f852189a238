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
// Larger inputs run four kernels over blocks of 4096 entries, chained with
// programmatic dependent launch: count (each block's count per expert),
// column scan (per expert, the rows of the earlier blocks of the same group
// of 256 blocks, and each group's total), expert scan (the groups' totals
// prefixed, counts, offsets), place (the ranks walked again, the block's
// entries put in expert order in shared memory and written out run after
// run, pos, the tail rows and the tile table).
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
// over e' < e of counts[e'] rounded up to tm, offsets[E] = R_pad.  Resets the
// status word (the place kernel adds bad-id bits after).  The tail rows and
// the tile table are the place kernel's, which runs over the whole GPU.
__global__ void __launch_bounds__(kScanThreads)
    k_scan_experts(int32_t *__restrict__ gsum, int ngroups, int32_t *__restrict__ counts, int E,
                   int tm, int64_t cap, int32_t *__restrict__ offsets,
                   uint32_t *__restrict__ status)
{
    __shared__ int warp_incl[kScanThreads / 32];
    pdl_launch_dependents();
    pdl_wait();
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
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
        if (e < E)
            offsets[e] = int32_t(off);
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
// step that hold the same expert are found in one of two ways.  kWalkOr
// (E <= kOrWalkMaxE): each warp keeps a 32-bit word per expert in shared
// memory, every lane ORs its bit into its expert's word and reads back the
// whole set (one shared atomic and one load per step).  Above that the
// per-warp words would not fit and kWalkMatch uses __match_any_sync.
constexpr int kWalkOr = 0, kWalkMatch = 2;
constexpr int kOrWalkMaxE = 1024;

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
            } else {
                peers = __match_any_sync(kFull, ok ? uint32_t(e) : (0x80000000u | lane));
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

// ---- place for large inputs -------------------------------------------------------
//
// Each CTA loops over blocks of kPlanBlockEntries flat entries (the grid being
// the CTAs the GPU holds at once).  A block is placed in four phases:
//  - walk: each warp walks its 512 entries 32 at a time; the lanes of a step
//    holding the same expert are found either through per-warp lane words in
//    shared memory (each lane ORs its bit into its expert's word) or from
//    ballots: one per bit of the id, combined per group of 5 bits into, for
//    lane b, the lanes whose digit is b, and read back with one shuffle per
//    group.  Each lane reads its expert's running count in this warp (shared
//    memory), the lowest lane of the set moves it on, and popc of the lower
//    lanes of the set gives the entry's rank in the warp's range;
//  - per expert (a thread per contiguous slice of experts): the warps'
//    counts prefixed over the warps, the block's count, its exclusive scan
//    over the experts (the start of the expert's run in the block's
//    expert-sorted order), and the row of the run's first slot, so that
//    row = slot + delta[e];
//  - each entry: slot = its warp's first slot for the expert + its rank;
//    pos (flat order, coalesced) = slot + delta[e]; the entry's key goes to
//    slot in shared memory;
//  - write-out: slot j of the sorted block to row j + delta[e], so that
//    neighbouring lanes write neighbouring rows of srt_tok and srt_w.
// The next block's ids, weights and count rows are copied into shared memory
// (cp.async) while the current one is placed.
constexpr int kQThreads = 256;
constexpr int kQWarps = kQThreads / 32;
constexpr int kQSteps = kPlanBlockEntries / kQThreads;  // 16 entries a lane
constexpr int kLiBits = 12;                              // local index in a block
static_assert(kPlanBlockEntries == (1 << kLiBits), "keys are (expert << 12) | local index");
static_assert(kQWarps == 8, "counter vectors: E (counts) and 2 * E (lane words) of 16 bytes");
static_assert(MOE_MAX_EXPERTS <= (1 << (32 - kLiBits)), "expert ids fit in a key");
constexpr int kMaxIdBits = 12;  // ids < MOE_MAX_EXPERTS = 4096
static_assert(MOE_MAX_EXPERTS <= (1 << kMaxIdBits), "id bits");
// The OR walk's lane words share the sorted keys' buffer (the walk ends
// before the first key is placed): 8 warps x E words fit in it for E <= 512.
constexpr int kPlaceOrWalkMaxE = 512;

// ids, weights and sorted keys (a word per entry; the OR walk's per-warp
// lane words share the keys' buffer), the per-warp running counts (16 bits),
// then the block's count row (then the runs' deltas), its group's row and the
// offsets.
constexpr size_t place_smem_bytes(int E)
{
    return size_t(3) * kPlanBlockEntries * sizeof(uint32_t) + size_t(kQWarps) * E * sizeof(uint16_t) +
           size_t(3 * E + 1) * sizeof(int);
}
static_assert(kQWarps * 512 <= kPlanBlockEntries, "lane words of the OR walk fit in the keys' buffer");

__device__ __forceinline__ void cp_async4(void *sdst, const void *gsrc)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(sdst)), "l"(gsrc)
                 : "memory");
}

// 16 bytes, of which the first src_bytes are read (the rest are zero-filled).
__device__ __forceinline__ void cp_async16(void *sdst, const void *gsrc, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(sdst)),
                 "l"(gsrc), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Waits until at most one committed group of this thread is still in flight.
__device__ __forceinline__ void cp_async_wait_all_but_one()
{
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// The nb (<= kPlanBlockEntries) words src[0, nb) into dst; vec: src is
// 16-byte aligned, so 16-byte copies (the last one partial).
__device__ __forceinline__ void copy_block_words(uint32_t *dst, const void *src, int nb, bool vec)
{
    const uint32_t *s = static_cast<const uint32_t *>(src);
    if (vec) {
        for (int c = threadIdx.x; c * 4 < nb; c += kQThreads)
            cp_async16(dst + 4 * c, s + 4 * c, uint32_t(min(4, nb - 4 * c)) * 4u);
    } else {
        for (int i = threadIdx.x; i < nb; i += kQThreads)
            cp_async4(dst + i, s + i);
    }
}

// The lanes of this step holding a valid id equal to this lane's (for a valid
// lane), from ballots: for each group of up to 5 id bits, lane b forms the set
// of valid lanes whose digit in that group is b (lsel[i] is all ones where bit
// i of the lane index is 0), and every lane reads the set of its own digit
// from that lane.  NBITS: bits of an id (ids < 2^NBITS).
template <int NBITS>
__device__ __forceinline__ uint32_t ballot_peers(uint32_t e, bool ok,
                                                 const uint32_t (&lsel)[5])
{
    const uint32_t vb = __ballot_sync(kFull, ok);
    uint32_t peers = vb;
#pragma unroll
    for (int g = 0; g * 5 < NBITS; ++g) {
        constexpr int kMaxW = 5;
        const int wg = NBITS - 5 * g < kMaxW ? NBITS - 5 * g : kMaxW;
        uint32_t m = vb;
#pragma unroll
        for (int bit = 0; bit < kMaxW; ++bit)
            if (bit < wg)
                m &= __ballot_sync(kFull, (e >> (5 * g + bit)) & 1u) ^ lsel[bit];
        peers &= __shfl_sync(kFull, m, int((e >> (5 * g)) & ((1u << wg) - 1u)));
    }
    return peers;
}

template <int NBITS, bool OR_WALK>
__global__ void __launch_bounds__(kQThreads, 3)
    k_place_blocks(const int32_t *__restrict__ ids, const float *__restrict__ w, int64_t n,
                   DivK kd, int E, int tm, int64_t cap, const int32_t *__restrict__ offsets,
                   const int32_t *__restrict__ counts, const int32_t *__restrict__ bcnt, int nblk,
                   int32_t *__restrict__ pos, int32_t *__restrict__ srt_tok,
                   float *__restrict__ srt_w, int32_t *__restrict__ tile_expert,
                   uint32_t *__restrict__ status, bool vec_in)
{
    extern __shared__ __align__(16) uint8_t psm[];
    uint32_t *s_ids = reinterpret_cast<uint32_t *>(psm);  // [4096] the block's ids
    float *s_w = reinterpret_cast<float *>(s_ids + kPlanBlockEntries);             // weights
    uint32_t *sorted = reinterpret_cast<uint32_t *>(s_w + kPlanBlockEntries);      // keys
    uint32_t *pm = sorted;  // [8][E] lane words of the OR walk, during the walk only
    uint16_t *cntw = reinterpret_cast<uint16_t *>(sorted + kPlanBlockEntries);     // [8][E]
    int *s_brow = reinterpret_cast<int *>(cntw + kQWarps * E);
    int *s_grow = s_brow + E;  // [E] block's count row, then delta; group's row
    int *s_off = s_grow + E;   // [E + 1]
    __shared__ int warp_tot[kQWarps];

    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t lane = tid & 31, lt = lanemask_lt();
    uint32_t lsel[5];
#pragma unroll
    for (int bit = 0; bit < 5; ++bit)
        lsel[bit] = (lane >> bit) & 1u ? 0u : kFull;
    pdl_launch_dependents();
    for (int v = tid; v < E; v += kQThreads)  // counts: E vectors of 16 bytes
        reinterpret_cast<uint4 *>(cntw)[v] = make_uint4(0u, 0u, 0u, 0u);
    if (OR_WALK)  // lane words: 2 * E vectors
        for (int v = tid; v < 2 * E; v += kQThreads)
            reinterpret_cast<uint4 *>(pm)[v] = make_uint4(0u, 0u, 0u, 0u);
    // everything is read after the wait: this launch may begin before the
    // count kernel's own wait for whatever wrote the ids has ended
    pdl_wait();
    for (int e = tid; e <= E; e += kQThreads)
        s_off[e] = offsets[e];
    auto block_len = [&](int bb) {
        return int(min(int64_t(kPlanBlockEntries), n - int64_t(bb) * kPlanBlockEntries));
    };
    if (int(blockIdx.x) < nblk) {
        const int64_t lo = int64_t(blockIdx.x) * kPlanBlockEntries;
        copy_block_words(s_ids, ids + lo, block_len(blockIdx.x), vec_in);
        cp_async_commit();
        copy_block_words(reinterpret_cast<uint32_t *>(s_w), w + lo, block_len(blockIdx.x), vec_in);
        cp_async_commit();
    }
    uint16_t *mycnt = cntw + warp * E;
    uint32_t *mypm = pm + warp * E;
    const int J = (E + kQThreads - 1) / kQThreads;  // experts per thread in the scans
    const int e0 = min(E, tid * J), e1 = min(E, e0 + J);
    bool bad = false;
    for (int b = blockIdx.x; b < nblk; b += gridDim.x) {
        const int64_t blk_lo = int64_t(b) * kPlanBlockEntries;
        const int nb = block_len(b);
        const int next = b + int(gridDim.x);
        cp_async_wait_all_but_one();  // this block's ids (its weights may be in flight)
        __syncthreads();              // ... every thread's; the counters are zero
        {
            const int32_t *brow = bcnt + int64_t(b) * E;
            const int32_t *grow = bcnt + (int64_t(nblk) + b / kPlanGroupBlocks) * E;
            for (int e = tid; e < E; e += kQThreads) {
                cp_async4(&s_brow[e], brow + e);
                cp_async4(&s_grow[e], grow + e);
            }
            cp_async_commit();
        }
        // ---- walk: each entry's rank in its warp's range ----------------------
        const int lo = warp * (kQSteps * 32);  // the warp's range in the block
        int v[kQSteps];  // (rank << 16) | expert, or -1
#pragma unroll
        for (int s = 0; s < kQSteps; ++s) {
            const int li = lo + s * 32 + int(lane);
            const bool in = li < nb;
            const int e = in ? int(s_ids[li]) : -1;
            const bool ok = e >= 0 && e < E;
            bad |= in && !ok && e != -1;
            if (lo + s * 32 < nb) {  // the same for the whole warp
                uint32_t peers;
                if (OR_WALK) {
                    if (ok)
                        atomicOr(&mypm[e], 1u << lane);
                    __syncwarp();
                    peers = ok ? mypm[e] : 0u;
                } else {
                    peers = ballot_peers<NBITS>(uint32_t(e), ok, lsel);
                }
                // every lane reads its expert's running count (lanes of one
                // expert read the same word), then the lowest of them moves it on
                const int first = ok ? int(mycnt[e]) : 0;
                __syncwarp();
                if (ok && (peers & lt) == 0u) {
                    mycnt[e] = uint16_t(first + __popc(peers));
                    if (OR_WALK)
                        mypm[e] = 0u;
                }
                v[s] = ok ? ((first + __popc(peers & lt)) << 16) | e : -1;
                __syncwarp();
            } else {
                v[s] = -1;
            }
        }
        __syncthreads();  // every warp's counts; every id read
        if (next < nblk)  // the next block's ids may come in
            copy_block_words(s_ids, ids + int64_t(next) * kPlanBlockEntries, block_len(next),
                             vec_in);
        cp_async_commit();
        // ---- per expert: warps prefixed, the run's start and its row delta -----
        // (warp 0's first slot for an expert is the run's start: until the
        // scan over the experts is known, its word holds the block's count)
        int tsum = 0;
        for (int e = e0; e < e1; ++e) {
            int run = 0;
#pragma unroll
            for (int w2 = 0; w2 < kQWarps; ++w2) {
                const int t = cntw[w2 * E + e];
                cntw[w2 * E + e] = uint16_t(run);
                run += t;
            }
            cntw[e] = uint16_t(run);
            tsum += run;
        }
        int sc = tsum;  // scan of the block's counts over the experts
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, sc, o);
            if (int(lane) >= o)
                sc += t;
        }
        if (lane == 31)
            warp_tot[warp] = sc;
        cp_async_wait_all_but_one();  // this block's weights and count rows
        __syncthreads();
        int start = sc - tsum, nv = 0;
#pragma unroll
        for (int w2 = 0; w2 < kQWarps; ++w2) {
            start += w2 < warp ? warp_tot[w2] : 0;
            nv += warp_tot[w2];
        }
        for (int e = e0; e < e1; ++e) {
            const int c = cntw[e];
            cntw[e] = uint16_t(start);
#pragma unroll
            for (int w2 = 1; w2 < kQWarps; ++w2)
                cntw[w2 * E + e] += uint16_t(start);
            // the run's first row less its first slot: offsets + rows of the
            // earlier groups + rows of the group's earlier blocks - start
            s_brow[e] += s_off[e] + s_grow[e] - start;
            start += c;
        }
        __syncthreads();
        // ---- each entry: its slot, pos, and its key in expert order -------------
#pragma unroll
        for (int s = 0; s < kQSteps; ++s) {
            const int li = lo + s * 32 + int(lane);
            if (li < nb) {
                const int p = v[s];
                int row = -1;
                if (p >= 0) {
                    const int e = p & 0xffff;
                    const int slot = int(mycnt[e]) + (p >> 16);
                    row = slot + s_brow[e];
                    sorted[slot] = (uint32_t(e) << kLiBits) | uint32_t(li);
                }
                pos[blk_lo + li] = row;
            }
        }
        __syncthreads();
        for (int q = tid; q < E; q += kQThreads)  // counters for the next block
            reinterpret_cast<uint4 *>(cntw)[q] = make_uint4(0u, 0u, 0u, 0u);
        // ---- write-out: slot j to row j + delta, neighbouring lanes neighbouring rows
        uint32_t key[kQSteps];
#pragma unroll
        for (int u = 0; u < kQSteps; ++u) {
            const int j = u * kQThreads + tid;
            key[u] = j < nv ? sorted[j] : 0u;
        }
#pragma unroll
        for (int u = 0; u < kQSteps; ++u) {
            const int j = u * kQThreads + tid;
            const uint32_t li = key[u] & ((1u << kLiBits) - 1u);
            const int row = j + s_brow[key[u] >> kLiBits];
            const float wt = s_w[li];
            if (j < nv && row < cap) {
                srt_tok[row] = int32_t(div_k(uint32_t(blk_lo) + li, kd));
                srt_w[row] = wt;
            }
        }
        __syncthreads();
        if (OR_WALK)  // the keys' buffer holds the next walk's lane words: zero
            for (int q = tid; q < 2 * E; q += kQThreads)
                reinterpret_cast<uint4 *>(pm)[q] = make_uint4(0u, 0u, 0u, 0u);
        if (next < nblk)  // every weight of this block has been read
            copy_block_words(reinterpret_cast<uint32_t *>(s_w),
                             w + int64_t(next) * kPlanBlockEntries, block_len(next), vec_in);
        cp_async_commit();
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy outlives the CTA
    if (__any_sync(kFull, bad) && lane == 0)
        atomicOr(status, MOE_STATUS_BAD_ID);
    // tail rows of each expert (srt_tok = -1, srt_w = +0) and the tile table,
    // spread over the grid
    for (int e = int(blockIdx.x) * kQThreads + tid; e < E; e += int(gridDim.x) * kQThreads)
        for (int64_t r = int64_t(s_off[e]) + counts[e]; r < s_off[e + 1] && r < cap; ++r) {
            srt_tok[r] = -1;
            srt_w[r] = 0.0f;
        }
    const int64_t R = min(int64_t(s_off[E]), cap);
    const int64_t ntiles = R / tm;
    for (int64_t t = int64_t(blockIdx.x) * kQThreads + tid; t < ntiles;
         t += int64_t(gridDim.x) * kQThreads) {
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
    // the place kernel: lanes of one expert from shared-memory lane words
    // (E <= kPlaceOrWalkMaxE) or from ballots on the id's bits
    const bool or_walk = E <= kPlaceOrWalkMaxE;
    const int nbits = E > 1 ? 32 - __builtin_clz(unsigned(E - 1)) : 0;
    using PlaceFn = void (*)(const int32_t *, const float *, int64_t, DivK, int, int, int64_t,
                             const int32_t *, const int32_t *, const int32_t *, int, int32_t *,
                             int32_t *, float *, int32_t *, uint32_t *, bool);
    static constexpr PlaceFn kBallot[kMaxIdBits + 1] = {
        k_place_blocks<0, false>,  k_place_blocks<1, false>,  k_place_blocks<2, false>,
        k_place_blocks<3, false>,  k_place_blocks<4, false>,  k_place_blocks<5, false>,
        k_place_blocks<6, false>,  k_place_blocks<7, false>,  k_place_blocks<8, false>,
        k_place_blocks<9, false>,  k_place_blocks<10, false>, k_place_blocks<11, false>,
        k_place_blocks<12, false>};
    const PlaceFn place_fn = or_walk ? k_place_blocks<0, true> : kBallot[nbits];
    const size_t place_smem = place_smem_bytes(E);
    cudaError_t err;
    if (nblk > 0) {
        // the opt-in size covers every E of this kernel's instantiation
        err = or_walk ? ensure_smem_limit(reinterpret_cast<const void *>(place_fn), kSlotPlaceOr,
                                          place_smem_bytes(kPlaceOrWalkMaxE))
                      : ensure_smem_limit(reinterpret_cast<const void *>(place_fn),
                                          kSlotPlaceBallot0 + nbits, place_smem_bytes(1 << nbits));
        if (err == cudaSuccess)
            err = launch_pdl(k_count, dim3(std::min(nblk, device_sm_count() * kCountCtasPerSm)),
                             dim3(kPThreads), cnt_smem, stream, ids, n, nblk, E, bcnt);
        if (err == cudaSuccess)
            err = launch_pdl(k_colscan, dim3((E + 31) / 32, ngroups), dim3(kColThreads), 0, stream,
                             bcnt, nblk, E, gsum);
        if (err != cudaSuccess)
            return err;
    }
    // with no entries every expert is empty: no tail rows, no tiles
    err = launch_pdl(k_scan_experts, dim3(1), dim3(kScanThreads), 0, stream, gsum, ngroups,
                     counts, E, tm, cap, offsets, status);
    if (err != cudaSuccess || nblk == 0)
        return err;
    int per_sm = 0;  // resident place CTAs per SM for this E (shared memory and registers)
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, place_fn, kQThreads, place_smem) !=
            cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();  // a failed query is not the caller's error
        per_sm = 1;
    }
    const int pgrid = std::min(nblk, device_sm_count() * per_sm);
    const bool vec_in =
        ((reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(w)) & 15) == 0;
    return launch_pdl(place_fn, dim3(pgrid), dim3(kQThreads), place_smem, stream, ids, w, n,
                      make_divk(uint32_t(k)), E, tm, cap, static_cast<const int32_t *>(offsets),
                      static_cast<const int32_t *>(counts), static_cast<const int32_t *>(bcnt),
                      nblk, pos, srt_tok, srt_w, tile_expert, status, vec_in);
}

}  // namespace moe
