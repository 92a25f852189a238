// Grouped expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged by TMA.
//
// "Batched resident MoE experts on Apple Silicon: a flat parallel expert
// pass", section 1: every routed row goes through its expert's gate/up
// projection, the gated activation and the weighted down projection.  Here
// the rows arrive grouped by expert (the plan's offsets), so each expert is
// one GEMM over its rows, and all experts run in one persistent launch per
// projection:
//
//   gate/up: H[r]  = bf16(silu(xs[r] Wg[e]) * (xs[r] Wu[e]))
//   down:    Ys[r] = bf16(srt_w[r] * (H[r] Wd[e]))
//
// Swap-AB: the weight is the MMA's A operand (M = 128 output features) and
// the expert's rows are its B operand (N = the unit's rows, a multiple of 16,
// at most 128), so an expert with few rows still fills the M = 128 tile.
// Each stage holds two A tiles and one B tile and feeds two accumulators:
// gate/up uses (Wg, Wu) over the same 128 features; down uses two adjacent
// 128-feature tiles of Wd, so one H tile serves 256 output features.
// Weights are [E, K, M] with M contiguous, i.e. MN-major A tiles read by one
// 3-D tensor map per weight (the expert is the outer coordinate); activation
// rows are K-major B tiles.  Both use 128-byte swizzled shared memory.
//
// Work unit = (expert chunk of <= 128 rows, 128 (gate/up) or 256 (down)
// output features), numbered chunk-major so that the tiles of one chunk
// (same activation rows) and the chunks of one big expert (same weight
// tile) run close together in time and share L2.  Each CTA (one per SM)
// walks units u = blockIdx.x + i*grid.
//
// Warp roles: warp 0 issues TMA copies into a ring of shared-memory stages,
// warp 1 issues tcgen05.mma into one of two TMEM accumulators, warps 2-5
// read the accumulator with tcgen05.ld, apply the epilogue, stage 16 rows of
// bf16 in shared memory, and one thread writes them out with a TMA store.
//
// Weight modes (WM): kBf16: bf16 weights and rows; kWiden: E4M3 weights,
// bf16 rows; kNative: E4M3 weights and E4M3 rows.
// kWiden: the weights are E4M3 codes with a per-(expert, output feature) scale
// (see quant.cu).  TMA brings the 8-bit tiles into the stage ring (half the
// bytes of bf16), eight more warps (6-13) widen them to bf16 -- exactly: every
// E4M3 value is a bf16 value -- into a second ring laid out as the bf16
// tiles would be (MN-major, 128-byte swizzle), and the epilogue multiplies
// each accumulator row (one output feature) by its scale.  The MMAs are the
// same bf16 MMAs.
// kNative: the weight codes are stored K-major ([E, f, d] for gate/up,
// [E, d, f] for down) and the rows (routed x rows, or H rows for down) are
// E4M3 codes with a power-of-two scale per row (rows.cu); both go straight
// to tcgen05.mma.kind::f8f6f4, K = 128 per stage in the same 128-byte rows
// (a K that is not a multiple of 128 ends in a stage whose upper half the
// TMA fills with zeros), and the epilogue multiplies by feature scale times
// row scale.
// Every output element is written by one CTA with a fixed K order: results
// are deterministic.  Every wait is bounded (2 s); on a timeout the CTA
// stops, lets its copies and MMAs land, frees TMEM and sets
// MOE_STATUS_TIMEOUT.
#include "../../include/moe_prefill.h"
#include "internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace moe {
namespace {

constexpr int BM = 128;                           // MMA M: output features per tile
constexpr int BK = 64;                            // K per stage: 64 bf16 = one 128-byte row
constexpr int BN = 128;                           // max rows per unit (MMA N)
constexpr int UMMA_K = 16;                        // K of one kind::f16 MMA
constexpr uint32_t kABoxBytes = 64 * BK * 2;      // 64 features x 64 K rows
constexpr uint32_t kATileBytes = 2 * kABoxBytes;  // 128 features
constexpr uint32_t kBTileBytes = BN * BK * 2;     // 128 rows x 64 K
constexpr int kThreads = 192;      // producer, MMA (A tile 0), four epilogue warps
constexpr int kConvThreads = 256;     // eight warps widening E4M3 tiles (W8)
constexpr int kConvThreadsMx4 = 256;  // warps decoding MXFP4 tiles
// One more warp, the last of the CTA, issues the MMAs of A tile 1.  Measured
// on GB300, a thread that waits on a stage's mbarrier and then issues that
// stage's MMAs cannot keep the tensor pipe busy once the MMAs are short (a
// unit of <= 128 rows): eight MMAs of 128 x 64 x 16 with the wait and the
// commit took 720 cycles a stage from one thread, 512 when two threads each
// waited and issued the MMAs of one accumulator.
constexpr int kIssuers = 2;
constexpr int kMaxWarps =
    (kThreads + (kConvThreads > kConvThreadsMx4 ? kConvThreads : kConvThreadsMx4)) / 32 + 1;
constexpr int kEpiThreads = 128;
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s for the stop path

constexpr int kStages = 4;
constexpr int kStagesMx4 = 7;  // no widened tiles in shared memory: room for more stages
constexpr uint32_t kStageBytes = 2 * kATileBytes + kBTileBytes;  // two A tiles + one B tile
constexpr uint32_t kAccCols = 2 * BN;                            // two accumulators per buffer
constexpr uint32_t kTmemCols = 2 * kAccCols;                     // double-buffered
constexpr int kStageRows = 16;                                   // rows per epilogue chunk
constexpr uint32_t kStgBytes = 2 * kStageRows * 256 * 2;         // two chunks of <= 256 features
// kWiden: a stage holds two E4M3 tiles (128 features x 64 K, 1 byte each,
// rows of 128 bytes unswizzled) and the B tile; two more slots hold the
// widened bf16 A tiles.  Shared memory in stages is the same 192 KB either
// way.  (kNative stages have the bf16 layout's sizes: two 128 x 128-byte A
// tiles and one B tile.)
constexpr uint32_t kA8TileBytes = BM * BK;                       // 8 KB
constexpr uint32_t kStageBytesW8 = 2 * kA8TileBytes + kBTileBytes;
constexpr int kConvSlots = 2;
constexpr uint32_t kConvSlotBytes = 2 * kATileBytes;
constexpr int kMx4Slots = 4;      // kMx4: decoded A tiles in tensor memory, four slots
constexpr uint32_t kMx4SlotCol = kAccCols;       // first TMEM column of the slots (256)
constexpr uint32_t kMx4SlotCols = 2 * (BK / 2);  // a slot: two tiles of 32 columns (64 K each)
constexpr int kMaxSlots = kConvSlots > kMx4Slots ? kConvSlots : kMx4Slots;

enum WeightMode : int { kBf16 = 0, kWiden = 1, kNative = 2, kMx4 = 3 };

// kMx4: MXFP4 weights -- 4-bit E2M1 codes, two per byte along K (the
// reduction axis; [E, M, K/2], eight codes to a 32-bit word: k = 8i + 2j at
// bits 4j .. 4j + 3, k = 8i + 2j + 1 at bits 16 + 4j .. 19 + 4j), and one
// power-of-two scale 2^(S-127) per (expert, block of 32 along K, output
// feature) ([E, K/32, M] exponent bytes).  A stage holds the B rows first
// (16 KB, 1024-byte aligned), then per A tile the codes (128 features x 32
// bytes) and the scales (2 blocks x 128 bytes).  The decoding warps turn
// code x 2^(S-127) into bf16 (exact: every such value is a bf16 value) and
// write each A tile straight into tensor memory (tcgen05.st: lane = output
// feature, one 32-bit column per two K), where the MMAs read it as their A
// operand ([a_tmem] form); B stays in shared memory.  The decoded tiles
// never pass through shared memory (staging them there, swizzled for the
// MMAs, measured 398-404 us against 316 us for the full layer's gate/up,
// with either decode).  Tensor memory then holds one accumulator buffer (columns 0 ..
// 255) and four decoded-A slots (256 .. 511); the epilogue of a unit and the
// next unit's MMAs do not overlap.  The epilogue applies no scale.
constexpr uint32_t kMx4CodeBytes = BM * BK / 2;   // 4 KB: 128 features x 64 K, 4 bits each
constexpr uint32_t kMx4ScaleBytes = BM * (BK / 32);  // 256 B: 128 features x 2 blocks
constexpr uint32_t kMx4TileBytes = kMx4CodeBytes + kMx4ScaleBytes;
constexpr uint32_t kStageBytesMx4 = (kBTileBytes + 2 * kMx4TileBytes + 1023) / 1024 * 1024;

// Tensor maps of the B rows: boxes of 128, 64, 32 and 16 rows (h[i] holds
// 128 >> i rows).  A unit's rows arrive in ONE copy per stage, of the
// smallest box that holds them (at most twice the rows): measured, the
// number of TMA copies per stage, not their bytes, bounded the ring's intake
// (eight 16-row boxes per stage: long-prompt gate/up 390 us; one 128-row
// box: 289 us; exact boxes of 128/64/32/16 rows, up to four: 304 us).
// With gathered rows (tma_gather4) h[0] is the token-row map.
constexpr int kRowMaps = 4;
struct RowMaps {
    CUtensorMap h[kRowMaps];
};

template <int WM>
struct Cfg {
    static constexpr bool kW8 = WM == kWiden || WM == kMx4;  // widening warps
    static constexpr int kConvT = WM == kMx4 ? kConvThreadsMx4 : kConvThreads;
    static constexpr int kThreadsK = (kW8 ? kThreads + kConvT : kThreads) + 32;
    static constexpr int kMmaWarp1 = kThreadsK / 32 - 1;  // issues the MMAs of A tile 1
    static constexpr int kS = WM == kMx4 ? kStagesMx4 : kStages;  // stages in the ring
    static constexpr uint32_t kStageB =
        WM == kMx4 ? kStageBytesMx4 : kW8 ? kStageBytesW8 : kStageBytes;
    // where the A tiles and the B rows sit in a stage
    static constexpr uint32_t kAOff = WM == kMx4 ? kBTileBytes : 0u;
    static constexpr uint32_t kBOff =
        WM == kMx4 ? 0u : WM == kWiden ? 2 * kA8TileBytes : 2 * kATileBytes;
    static constexpr uint32_t kRingBytes =
        kS * kStageB + (WM == kWiden ? kConvSlots * kConvSlotBytes : 0u);
    static constexpr int kSlots = WM == kMx4 ? kMx4Slots : kConvSlots;  // widened-tile slots
    static constexpr int kAccBufs = WM == kMx4 ? 1 : 2;  // accumulator buffers in TMEM
    static constexpr int kKStep = WM == kNative ? 128 : BK;  // K elements per stage
};

// GATED: gate/up (A tiles = Wg and Wu over the same 128 features, output H).
// !GATED: down (A tiles = Wd over features m0 and m0 + 128, output Ys).
template <bool GATED>
struct Kind {
    static constexpr int kUnitM = GATED ? BM : 2 * BM;  // output features per unit
};

template <int S>
struct Ctrl {
    uint64_t full[S];
    uint64_t empty[S];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t conv_full[kMaxSlots];   // W8: widened A tiles ready (one arrival per warp)
    uint64_t conv_empty[kMaxSlots];  // W8: the MMAs are done with a slot
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int epi_stop;  // set only by epilogue threads; read by all four warps after a barrier
    int warp_sum[kMaxWarps];
};

struct FfnArgs {
    const int32_t *offsets;
    const int32_t *srt_tok;  // gate/up with gathered rows: token of each row, -1 for pad rows
    const float *srt_w;  // down only
    uint16_t *out;       // H (gate/up) or Ys (down), bf16 bits, [cap, M]
    uint32_t *status;    // may be null
    int64_t cap;
    int E;
    int K;  // reduction extent: d (gate/up) or f (down)
    int M;  // output features: f (gate/up) or d (down)
    int stall_cta;  // self-test only: this CTA's first stage waits for 16 bytes
                    // that never come; -1 in every normal launch
    const float *scale0;  // E4M3: scales [E, M] of A tile 0's weight (Wg or Wd)
    const float *scale1;  // E4M3: scales [E, M] of A tile 1's weight (Wu or Wd)
    const int32_t *row_exp;  // kNative: each row's scale exponent (row scale 2^e)
};

template <int WM>
constexpr size_t ffn_smem_bytes(int E)
{
    return 1024 + size_t(Cfg<WM>::kRingBytes) + kStgBytes + sizeof(Ctrl<Cfg<WM>::kS>) +
           2 * BN * sizeof(int) + size_t(E + 1) * sizeof(int);
}
static_assert(ffn_smem_bytes<kBf16>(MOE_MAX_EXPERTS) <= 227 * 1024, "shared memory per CTA");
static_assert(ffn_smem_bytes<kWiden>(MOE_MAX_EXPERTS) <= 227 * 1024, "shared memory per CTA");
static_assert(ffn_smem_bytes<kNative>(MOE_MAX_EXPERTS) <= 227 * 1024, "shared memory per CTA");
static_assert(ffn_smem_bytes<kMx4>(MOE_MAX_EXPERTS) <= 227 * 1024, "shared memory per CTA");

// Bounded wait that ignores the abort flag (used while stopping).
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kDrainLimitNs)
            return;
}

__device__ __forceinline__ int expert_chunks(const int32_t *off, int e, int64_t cap, bool &bad)
{
    const int lo = off[e], hi = off[e + 1];
    if (lo < 0 || hi < lo || int64_t(hi) > cap || (lo & 15) || (hi & 15)) {
        bad = true;
        return 0;
    }
    return (hi - lo + BN - 1) / BN;
}

// chunk_start[e] = chunks of experts < e (chunks of <= BN rows); returns the
// total.  Experts whose offsets are not ascending multiples of 16 inside cap
// get no chunks and raise MOE_STATUS_BAD_OFFSETS.  All threads take part.
__device__ int build_chunk_table(const int32_t *off, int E, int64_t cap, int *cs, int *warp_sum,
                                 uint32_t *status)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthr = blockDim.x, nwarps = nthr >> 5;
    const int per = (E + nthr - 1) / nthr;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    bool bad = false;
    int local = 0;
    for (int e = e0; e < e1; ++e)
        local += expert_chunks(off, e, cap, bad);
    int v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o)
            v += t;
    }
    if (lane == 31)
        warp_sum[warp] = v;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < nwarps; ++w) {
        before += w < warp ? warp_sum[w] : 0;
        total += warp_sum[w];
    }
    int run = before + v - local;
    for (int e = e0; e < e1; ++e) {
        cs[e] = run;
        run += expert_chunks(off, e, cap, bad);
    }
    if (tid == 0)
        cs[E] = total;
    if (bad && status)
        atomicOr(status, MOE_STATUS_BAD_OFFSETS);
    __syncthreads();
    return total;
}

struct Unit {
    int e, row0, nrows, mt;
};

__device__ __forceinline__ Unit map_unit(int64_t u, int n_mt, const int *cs, int E,
                                         const int32_t *off)
{
    const int c = int(u / n_mt);
    Unit r;
    r.mt = int(u - int64_t(c) * n_mt);
    int lo = 0, hi = E - 1;  // the expert e with cs[e] <= c < cs[e+1]
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cs[mid] <= c)
            lo = mid;
        else
            hi = mid - 1;
    }
    r.e = lo;
    r.row0 = off[lo] + (c - cs[lo]) * BN;
    r.nrows = min(BN, off[lo + 1] - r.row0);
    return r;
}

__device__ __forceinline__ uint16_t bf16_bits(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ void epi_bar()
{
    asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
}

// 16 E4M3 codes (one 16-byte chunk) -> 16 bf16 values (two 16-byte
// chunks), exactly: E4M3 -> f16 is exact, and so is f16 -> f32 -> bf16 for
// values that came from E4M3 (at most 4 significant bits, exponents inside
// bf16's range).
__device__ __forceinline__ void widen_e4m3x16(const uint4 v, uint4 &lo, uint4 &hi)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __nv_fp8x2_storage_t pair =
            static_cast<__nv_fp8x2_storage_t>((w[i >> 1] >> (16 * (i & 1))) & 0xffffu);
        const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3));
        const __nv_bfloat162 b = __float22bfloat162_rn(__half22float2(h));
        o[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// 2^(S-127) as an fp32 value, exactly (S = 0: the subnormal 2^-127).
__device__ __forceinline__ float mx_scale(uint32_t S)
{
    return __uint_as_float(S ? S << 23 : 0x00400000u);
}

// Two E2M1 codes (pair j of a code word: k even and odd) -> the bf16 pair
// value(code) x 2^-126 (low half: the even k), exactly: the three magnitude
// bits (e1 e0 m) placed at bf16 bits 8..6 are the exponent field e1 e0 and
// the mantissa's top bit, which reads value(code) x 2^-126 for every code
// (e = 0 lands on the subnormal 2^-127 = 0.5 x 2^-126), and the sign at bit
// 15.  A code word holds pair j's even code at bits 4j..4j+3 and its odd
// code 16 bits higher; masked out (w & 0x000F000F << 4j) and multiplied by
// 2^(6-4j) + 2^(12-4j) (j = 0, 1; the word shifted right by 8 first for
// j = 2, 3), each code lands at bits 6..9 and, again, 12..15 of its half
// without carries; the final mask keeps the magnitude from the first copy
// and the sign from the second.
__device__ __forceinline__ uint32_t e2m1_pair_bits(uint32_t w, int j)
{
    const uint32_t x = (j & 2) ? w >> 8 : w;
    return (j & 1) ? ((x & 0x00F000F0u) * 0x104u) & 0x81C081C0u
                   : ((x & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
}

// Pair j of a code word as the two-code byte (the even k in the low four
// bits) the f16 conversion takes.
__device__ __forceinline__ uint32_t e2m1_pair_byte(uint32_t w, int j)
{
    return ((w >> (4 * j)) & 0xFu) | (((w >> (16 + 4 * j)) & 0xFu) << 4);
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One stage of an MXFP4 A tile -> bf16 in tensor memory.  Decoding thread
// ct (eight warps) takes tile ct >> 7 and output feature m = 32 (warp mod 4)
// + lane, the TMEM lane its warp may write: the feature's 64 codes of the
// stage (32 bytes) and its two block scales, 64 bf16 values = 32 columns at
// slot + 32 t (column j: k = 2j low, 2j + 1 high), one tcgen05.st.  The
// value is code x 2^(S-127): from the bit placement above times the bf16
// 2^(S-1) (one bf16x2 multiply, exact while S <= 128: weights below 8 in
// magnitude); a block with a larger S takes the f16 conversion and an fp32
// multiply, exact as well.
__device__ __forceinline__ void decode_mx4_tile(const uint8_t *src, int ct, int nt,
                                                uint32_t slot_taddr)
{
    // a warp may write only its own quadrant of TMEM lanes: warp index mod 4
    const int t = ct >> 7, lane = ct & 31, q = int(threadIdx.x >> 5) & 3;
    if (t >= nt)
        return;
    const int m = 32 * q + lane;
    const uint8_t *tile = src + t * kMx4TileBytes;
    // the feature's 32 bytes in two 16-byte loads, the halves in a lane-dependent
    // order so that each quarter-warp covers all 32 banks
    const int h0 = (lane >> 2) & 1;
    const uint4 c0 = *reinterpret_cast<const uint4 *>(tile + m * 32 + 16 * h0);
    const uint4 c1 = *reinterpret_cast<const uint4 *>(tile + m * 32 + 16 * (h0 ^ 1));
    const uint4 lo = h0 ? c1 : c0, hi = h0 ? c0 : c1;  // k 0..31 (block 0), 32..63 (block 1)
    const uint32_t s0 = tile[kMx4CodeBytes + m], s1 = tile[kMx4CodeBytes + BM + m];
    const uint32_t cw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t v[32];
    if (s0 <= 128u && s1 <= 128u) {
        const uint32_t sc0 = ((s0 + 126u) << 7) * 0x10001u, sc1 = ((s1 + 126u) << 7) * 0x10001u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t sc = i < 4 ? sc0 : sc1;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const uint32_t u = e2m1_pair_bits(cw[i], b);
                const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&u),
                                                 *reinterpret_cast<const __nv_bfloat162 *>(&sc));
                v[4 * i + b] = *reinterpret_cast<const uint32_t *>(&r);
            }
        }
    } else {
        const float x0 = mx_scale(s0), x1 = mx_scale(s1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float x = i < 4 ? x0 : x1;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float2 f = __half22float2(__half2(__nv_cvt_fp4x2_to_halfraw2(
                    static_cast<__nv_fp4x2_storage_t>(e2m1_pair_byte(cw[i], b)), __NV_E2M1)));
                const __nv_bfloat162 r = __floats2bfloat162_rn(f.x * x, f.y * x);
                v[4 * i + b] = *reinterpret_cast<const uint32_t *>(&r);
            }
        }
    }
    tmem_st_32x32b_x32(slot_taddr + (uint32_t(32 * q) << 16) + uint32_t(t) * (BK / 2), v);
    tmem_st_wait();
}

// GATHER: the B rows of a unit are token rows of x fetched by index
// (srt_tok, four rows per TMA gather4) instead of consecutive rows of xs.
// WM: weight mode (kBf16, kWiden, kNative), see the top of this file.
// map_s0, map_s1: kMx4 only, the scale exponents of A tiles 0 and 1.
template <bool GATED, bool GATHER, int WM>
__global__ void __launch_bounds__(Cfg<WM>::kThreadsK, 1)
    k_ffn(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
          const __grid_constant__ RowMaps map_b, const __grid_constant__ CUtensorMap map_out,
          const __grid_constant__ CUtensorMap map_s0, const __grid_constant__ CUtensorMap map_s1,
          const FfnArgs p)
{
    constexpr bool W8 = Cfg<WM>::kW8, A8 = WM == kNative, MX4 = WM == kMx4;
    constexpr bool SCALED = WM == kWiden || WM == kNative;  // scales in the epilogue
    static_assert(!(GATHER && SCALED), "gathered rows come with bf16 weights only");
    constexpr int S = Cfg<WM>::kS;
    constexpr int UM = Kind<GATED>::kUnitM;
    constexpr uint32_t SB = Cfg<WM>::kStageB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *conv = smem + S * SB;  // kWiden: widened A tiles, kConvSlots slots
    uint16_t *stg = reinterpret_cast<uint16_t *>(smem + Cfg<WM>::kRingBytes);
    Ctrl<S> *ctl = reinterpret_cast<Ctrl<S> *>(smem + Cfg<WM>::kRingBytes + kStgBytes);
    int *row_tok = reinterpret_cast<int *>(ctl + 1);  // [BN] tokens of the unit's rows
    float *row_w = reinterpret_cast<float *>(row_tok + BN);  // [BN] routing weights (down)
    // kNative: the unit's row scales (gate/up has no routing weights to stage)
    float *row_s = GATED ? row_w : reinterpret_cast<float *>(row_tok);
    int *chunk_start = row_tok + 2 * BN;
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], kIssuers);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tmem_full[b], kIssuers);
            mbar_init(&ctl->tmem_empty[b], kEpiThreads);
        }
        for (int c = 0; c < Cfg<WM>::kSlots; ++c) {
            mbar_init(&ctl->conv_full[c], Cfg<WM>::kConvT / 32);
            mbar_init(&ctl->conv_empty[c], kIssuers);
        }
        mbar_init(&ctl->mma_done, kIssuers);
        ctl->abort_flag = 0;
        ctl->epi_stop = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&map_a0);
        if (GATED)
            prefetch_tmap(&map_a1);
        for (int i = 0; i < (GATHER ? 1 : kRowMaps); ++i)
            prefetch_tmap(&map_b.h[i]);
        prefetch_tmap(&map_out);
        if (MX4) {
            prefetch_tmap(&map_s0);
            if (GATED)
                prefetch_tmap(&map_s1);
        }
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;

    pdl_wait();
    pdl_launch_dependents();

    const int total_chunks =
        build_chunk_table(p.offsets, p.E, p.cap, chunk_start, ctl->warp_sum, p.status);
    const int n_mt = (p.M + UM - 1) / UM;
    const int nk = (p.K + Cfg<WM>::kKStep - 1) / Cfg<WM>::kKStep;
    const int64_t total_units = int64_t(total_chunks) * n_mt;

    // first feature of A tile t of a unit starting at feature m0
    auto tile_base = [](int m0, int t) { return GATED ? m0 : m0 + t * BM; };

    if (warp == 0) {
        // ---- TMA producer (lane 0 issues; with GATHER the warp loads row indices) ----
        int stage = 0;
        uint32_t phase = 0, issued = 0, issued_par = 0;
        bool ok = true;
        uint32_t stall_bytes = int(blockIdx.x) == p.stall_cta ? 16u : 0u;
        for (int64_t u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
            const Unit w = map_unit(u, n_mt, chunk_start, p.E, p.offsets);
            if (GATHER) {
                // the previous unit's gather4s took their rows as operands at issue
                for (int r = int(lane); r < w.nrows; r += 32)
                    row_tok[r] = p.srt_tok[w.row0 + r];
                __syncwarp();
            }
            if (lane == 0) {
                const int m0 = w.mt * UM;
                uint32_t boxes = 0;  // 64-feature boxes per stage that hold real features
                for (int t = 0; t < 2; ++t)
                    for (int h = 0; h < 2; ++h)
                        boxes += tile_base(m0, t) + 64 * h < p.M;
                // kWiden: one E4M3 box of 128 features per A tile that starts
                // inside M (features past M are zero-filled and still counted)
                const uint32_t a_bytes =
                    MX4  ? (1u + uint32_t(tile_base(m0, 1) < p.M)) * kMx4TileBytes
                    : W8 ? (1u + uint32_t(tile_base(m0, 1) < p.M)) * kA8TileBytes
                    : A8 ? (1u + uint32_t(tile_base(m0, 1) < p.M)) * kATileBytes  // 128 x 128 codes
                         : boxes * kABoxBytes;
                // B: one copy of the smallest 16/32/64/128-row box holding the
                // unit's rows (128-byte rows in every mode)
                const int box_i = w.nrows > BN / 2 ? 0 : w.nrows > BN / 4 ? 1 : w.nrows > BN / 8 ? 2 : 3;
                const uint32_t b_rows = GATHER ? uint32_t(w.nrows) : uint32_t(BN >> box_i);
                const uint32_t bytes = a_bytes + b_rows * uint32_t(BK * 2);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint64_t *fb = &ctl->full[stage];
                    mbar_arrive_expect_tx(fb, bytes + stall_bytes);
                    stall_bytes = 0;
                    uint8_t *sa = smem + stage * SB + Cfg<WM>::kAOff;
                    const int k0 = kb * Cfg<WM>::kKStep;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const CUtensorMap *m = (GATED && t == 1) ? &map_a1 : &map_a0;
                        if (MX4) {
                            // codes [E, M, K/2]: (byte column along K, feature,
                            // expert); scales [E, K/32, M]: (feature, block, expert)
                            if (tile_base(m0, t) < p.M) {
                                uint8_t *st = sa + t * kMx4TileBytes;
                                tma_load_3d(st, m, fb, k0 / 2, tile_base(m0, t), w.e);
                                tma_load_3d(st + kMx4CodeBytes, (GATED && t == 1) ? &map_s1 : &map_s0,
                                            fb, tile_base(m0, t), k0 / 32, w.e);
                            }
                        } else if (W8) {
                            if (tile_base(m0, t) < p.M)
                                tma_load_3d(sa + t * kA8TileBytes, m, fb, tile_base(m0, t), k0,
                                            w.e);
                        } else if (A8) {
                            // K-major codes [E, M, K]: coordinates (k, feature, expert)
                            if (tile_base(m0, t) < p.M)
                                tma_load_3d(sa + t * kATileBytes, m, fb, k0, tile_base(m0, t),
                                            w.e);
                        } else {
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int f0 = tile_base(m0, t) + 64 * h;
                                if (f0 < p.M)
                                    tma_load_3d(sa + t * kATileBytes + h * kABoxBytes, m, fb, f0,
                                                k0, w.e);
                            }
                        }
                    }
                    uint8_t *sb = smem + stage * SB + Cfg<WM>::kBOff;
                    if (GATHER) {
                        for (int j = 0; j < w.nrows; j += 4)
                            tma_gather4(sb + j * (BK * 2), &map_b.h[0], fb, k0, row_tok[j],
                                        row_tok[j + 1], row_tok[j + 2], row_tok[j + 3]);
                    } else {
                        // the unit's rows in one box of 16, 32, 64 or 128 rows, the
                        // smallest that holds them; rows past the unit (the next
                        // expert's, or zero past cap) are loaded and not used
                        tma_load_2d(sb, &map_b.h[box_i], fb, k0, w.row0);
                    }
                    issued |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            ok = __shfl_sync(kFull, ok, 0);
            __syncwarp();
        }
        if (lane == 0) {
            // every stage must be released by the MMA side before the CTA exits
            for (int i = 0; ok && i < S; ++i) {
                ok = mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)  // stopped: let the copies already issued land
                for (int s = 0; s < S; ++s)
                    if ((issued >> s) & 1u)
                        mbar_drain(&ctl->full[s], (issued_par >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == 1 || warp == Cfg<WM>::kMmaWarp1) {
        // ---- MMA issuers: warp 1 for A tile 0, the last warp for A tile 1 ----
        const int tsel = warp == 1 ? 0 : 1;
        if (lane == 0) {
            int stage = 0, abuf = 0, cslot = 0;
            uint32_t phase = 0, aphase = 0, cphase = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
                const Unit w = map_unit(u, n_mt, chunk_start, p.E, p.offsets);
                const int m0 = w.mt * UM;
                // this issuer's A tile holds real features (tile 0 always does)
                const bool mine = tsel == 0 || tile_base(m0, 1) < p.M;
                if (!mbar_wait(&ctl->tmem_empty[abuf], aphase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d0 = tmem_base + uint32_t(abuf) * kAccCols + uint32_t(tsel) * BN;
                // kMx4: this issuer's decoded A tile in the slot's TMEM columns
                const uint32_t a_tm = tmem_base + kMx4SlotCol + uint32_t(tsel) * (BK / 2);
                const uint32_t idesc = A8 ? idesc_e4m3_f32(BM, uint32_t(w.nrows))
                                          : idesc_bf16_f32(BM, uint32_t(w.nrows), MX4 ? 0u : 1u, 0u);
                for (int kb = 0; kb < nk; ++kb) {
                    // kMx4: the decoding warps arrive on conv_full only after they
                    // saw the stage full (its B rows with its codes), so the
                    // issuers wait on conv_full alone
                    if ((!MX4 && !mbar_wait(&ctl->full[stage], phase, abort_flag)) ||
                        (W8 && !mbar_wait(&ctl->conv_full[cslot], cphase, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sst = smem_u32(smem + stage * SB);
                    const uint32_t sa = (W8 ? smem_u32(conv + cslot * kConvSlotBytes) : sst) +
                                        uint32_t(tsel) * kATileBytes;  // this issuer's A tile
                    const uint32_t sb = sst + Cfg<WM>::kBOff;
                    if (!mine) {
                        // no MMAs; the commits below still count this issuer's arrival
                    } else if (MX4) {
                        // A from tensor memory: K = 16 (8 columns) per instruction
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk)
                            tc_mma_f16_tmem_a(d0, a_tm + uint32_t(cslot) * kMx4SlotCols + kk * 8,
                                              smem_desc_sw128(sb + kk * UMMA_K * 2, 16, 1024),
                                              idesc, (kb | kk) != 0);
                    } else if (A8) {
                        // both operands K-major 128-byte rows; K = 32 codes (32 bytes)
                        // per instruction, four per stage
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_f8(d0, smem_desc_sw128(sa + kk * 32, 16, 1024),
                                      smem_desc_sw128(sb + kk * 32, 16, 1024), idesc,
                                      (kb | kk) != 0);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk)
                            // A: MN-major, one 128-byte row per K index, the K step moves
                            // 16 rows; B: K-major rows of 128 B, the K step moves 32 B
                            // inside the row.
                            tc_mma_f16(d0, smem_desc_sw128(sa + kk * UMMA_K * 128, kABoxBytes, 1024),
                                       smem_desc_sw128(sb + kk * UMMA_K * 2, 16, 1024), idesc,
                                       (kb | kk) != 0);
                    }
                    tc_commit(&ctl->empty[stage]);  // frees the stage once these MMAs finish
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (W8) {
                        tc_commit(&ctl->conv_empty[cslot]);
                        if (++cslot == Cfg<WM>::kSlots) {
                            cslot = 0;
                            cphase ^= 1u;
                        }
                    }
                }
                if (!ok)
                    break;
                tc_commit(&ctl->tmem_full[abuf]);
                if (++abuf == Cfg<WM>::kAccBufs) {
                    abuf = 0;
                    aphase ^= 1u;
                }
            }
            // all MMAs issued here have completed once this arrives
            tc_commit(&ctl->mma_done);
            mbar_drain(&ctl->mma_done, 0);
        }
        __syncwarp();
    } else if (W8 && warp >= kThreads / 32) {
        // ---- widening (W8): E4M3 A tiles of a stage -> bf16 tiles of a slot ----
        const int ct = int(threadIdx.x) - kThreads;  // 0 .. Cfg<WM>::kConvT - 1
        int stage = 0, cslot = 0;
        uint32_t phase = 0, cphase = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
            const Unit w = map_unit(u, n_mt, chunk_start, p.E, p.offsets);
            const int nt = 1 + int(tile_base(w.mt * UM, 1) < p.M);  // A tiles loaded
            for (int kb = 0; kb < nk; ++kb) {
                if (!mbar_wait(&ctl->full[stage], phase, abort_flag) ||
                    !mbar_wait(&ctl->conv_empty[cslot], cphase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = smem + stage * SB + Cfg<WM>::kAOff;
                uint8_t *dst = conv + cslot * kConvSlotBytes;
                if (MX4) {
                    // the MMAs that last read this slot's columns are done
                    tc_fence_after_sync();
                    decode_mx4_tile(src, ct, nt,
                                    tmem_base + kMx4SlotCol + uint32_t(cslot) * kMx4SlotCols);
                } else {
                // a tile is 64 K rows x 8 chunks of 16 codes.  Chunk c of row
                // r (features 16c..16c+15)
                // becomes the 16-byte chunks 2(c&3) and 2(c&3)+1 of row r of
                // 64-feature box c>>2, each placed at its index XOR (r mod 8),
                // the 128-byte swizzle a TMA load of the bf16 box would apply.
                // all of a thread's loads first, then the widening and stores:
                // kPer independent chains instead of one after another
                constexpr int kPer = 2 * 512 / kConvThreads;
                uint4 v[kPer];
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int g = ct + i * kConvThreads;
                    if (g < 512 * nt)
                        v[i] = *reinterpret_cast<const uint4 *>(src + (g >> 9) * kA8TileBytes +
                                                                ((g >> 3) & 63) * 128 + (g & 7) * 16);
                }
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int g = ct + i * kConvThreads;
                    if (g < 512 * nt) {
                        const int t = g >> 9, r = (g >> 3) & 63, c = g & 7;
                        uint4 lo, hi;
                        widen_e4m3x16(v[i], lo, hi);
                        uint8_t *row = dst + t * kATileBytes + (c >> 2) * kABoxBytes + r * 128;
                        const int j0 = 2 * (c & 3);
                        *reinterpret_cast<uint4 *>(row + ((j0 ^ (r & 7)) << 4)) = lo;
                        *reinterpret_cast<uint4 *>(row + (((j0 + 1) ^ (r & 7)) << 4)) = hi;
                    }
                }
                }
                if (MX4)
                    tc_fence_before_sync();  // this thread's tensor-memory stores, done
                else
                    fence_proxy_async_smem();  // the widened tiles -> visible to the MMAs
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ctl->conv_full[cslot]);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++cslot == Cfg<WM>::kSlots) {
                    cslot = 0;
                    cphase ^= 1u;
                }
            }
        }
    } else {
        // ---- epilogue: TMEM -> registers -> shared (16 rows) -> TMA store ----
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const int fq = q * 32 + int(lane);
        const int et = int(threadIdx.x) - 64;  // 0..127; thread 0 issues the stores
        int abuf = 0;
        uint32_t aphase = 0, chunk = 0;
        // What a unit's epilogue reads from global memory is loaded ahead in
        // registers: the offsets bounding its expert two units ahead, then
        // (from those) its rows' routing weights and exponents and its
        // features' scales one unit ahead, so no load's latency falls
        // between one unit's stores and the next unit's TMEM reads.
        struct Ahead {  // unit index split and the expert's offsets (in flight)
            int c, mt, e, oa, ob;
        };
        struct Vals {  // per-thread values of a unit (in flight)
            float rw, s0, s1;
            int rx;
        };
        auto ahead_of = [&](int64_t uu) {
            Ahead a;
            a.c = int(uu / n_mt);
            a.mt = int(uu - int64_t(a.c) * n_mt);
            int lo = 0, hi = p.E - 1;  // the expert e with chunk_start[e] <= c < chunk_start[e+1]
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (chunk_start[mid] <= a.c)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            a.e = lo;
            a.oa = p.offsets[lo];
            a.ob = p.offsets[lo + 1];
            return a;
        };
        auto unit_of = [&](const Ahead &a) {
            Unit r;
            r.mt = a.mt;
            r.e = a.e;
            r.row0 = a.oa + (a.c - chunk_start[a.e]) * BN;
            r.nrows = min(BN, a.ob - r.row0);
            return r;
        };
        auto vals_of = [&](const Unit &uw) {
            Vals v{1.0f, 1.0f, 1.0f, 0};
            if (!GATED && et < uw.nrows)  // the rows' routing weights
                v.rw = p.srt_w[uw.row0 + et];
            if (A8 && et < uw.nrows)  // the rows' scale exponents
                v.rx = p.row_exp[uw.row0 + et];
            if (SCALED) {  // E4M3 weights: this thread's output feature in both A tiles
                const int64_t eb = int64_t(uw.e) * p.M;
                const int um0 = uw.mt * UM;
                const int fa = tile_base(um0, 0) + fq, fb = tile_base(um0, 1) + fq;
                v.s0 = fa < p.M ? p.scale0[eb + fa] : 0.0f;
                v.s1 = fb < p.M ? p.scale1[eb + fb] : 0.0f;
            }
            return v;
        };
        const int64_t ustep = gridDim.x;
        Unit wnext{};
        Vals vnext{1.0f, 1.0f, 1.0f, 0};
        Ahead anext{};
        if (int64_t(blockIdx.x) < total_units) {
            wnext = unit_of(ahead_of(blockIdx.x));
            vnext = vals_of(wnext);
        }
        if (int64_t(blockIdx.x) + ustep < total_units)
            anext = ahead_of(int64_t(blockIdx.x) + ustep);
        for (int64_t u = blockIdx.x; u < total_units; u += ustep) {
            const Unit w = wnext;
            const Vals vals = vnext;
            if (u + ustep < total_units) {  // its offsets were loaded one unit ago
                wnext = unit_of(anext);
                vnext = vals_of(wnext);
            }
            if (u + 2 * ustep < total_units)
                anext = ahead_of(u + 2 * ustep);
            const int m0 = w.mt * UM;
            const bool use1 = tile_base(m0, 1) < p.M;
            const float sc0 = vals.s0, sc1 = vals.s1;
            // The four warps stop together or not at all: they meet at named
            // barriers below.  epi_stop is written before this barrier and read
            // after it; the next write can only come after the unit's chunk
            // barriers, which every thread reaches after its read.
            if (!GATED && et < w.nrows)  // read by every thread of the unit's chunks
                row_w[et] = vals.rw;
            if (A8 && et < w.nrows)  // the rows' scales 2^e
                row_s[et] = ldexpf(1.0f, vals.rx);
            if (!mbar_wait(&ctl->tmem_full[abuf], aphase, abort_flag))
                *reinterpret_cast<volatile int *>(&ctl->epi_stop) = 1;
            epi_bar();
            if (*reinterpret_cast<volatile int *>(&ctl->epi_stop))
                break;
            tc_fence_after_sync();
            const uint32_t t0 =
                tmem_base + (uint32_t(q * 32) << 16) + uint32_t(abuf) * kAccCols;
            for (int c0 = 0; c0 < w.nrows; c0 += kStageRows, ++chunk) {
                uint16_t *sg = stg + (chunk & 1u) * (kStageRows * 256);
                uint32_t a[16], b[16];
                tmem_ld_32x32b_x16(t0 + uint32_t(c0), a);
                if (GATED || use1)
                    tmem_ld_32x32b_x16(t0 + BN + uint32_t(c0), b);
                tmem_ld_wait();
                float v0[16], v1[16];
                const float *rs = row_s + c0;
                if (GATED) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float s0 = A8 ? sc0 * rs[j] : sc0, s1 = A8 ? sc1 * rs[j] : sc1;
                        const float g = SCALED ? __uint_as_float(a[j]) * s0 : __uint_as_float(a[j]);
                        const float up =
                            SCALED ? __uint_as_float(b[j]) * s1 : __uint_as_float(b[j]);
                        v0[j] = __fdividef(g, 1.0f + __expf(-g)) * up;
                    }
                } else {
                    const float *wr = row_w + c0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float s0 = A8 ? sc0 * rs[j] : sc0, s1 = A8 ? sc1 * rs[j] : sc1;
                        const float o0 = SCALED ? __uint_as_float(a[j]) * s0 : __uint_as_float(a[j]);
                        const float o1 = SCALED ? __uint_as_float(b[j]) * s1 : __uint_as_float(b[j]);
                        v0[j] = wr[j] * o0;
                        v1[j] = use1 ? wr[j] * o1 : 0.0f;
                    }
                }
                // the bulk store that last read this staging buffer (two chunks
                // back) must be done with it before it is overwritten
                if (et == 0)
                    bulk_wait_read<1>();
                epi_bar();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    sg[j * UM + fq] = bf16_bits(v0[j]);
                    if (!GATED)
                        sg[j * UM + BM + fq] = bf16_bits(v1[j]);
                }
                fence_proxy_async_smem();  // staged rows -> visible to the bulk copy
                epi_bar();
                // 16 rows x UM features leave as one TMA store; features past M
                // fall outside the tensor and are not written
                if (et == 0) {
                    tma_store_2d(&map_out, sg, m0, w.row0 + c0);
                    bulk_commit();
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&ctl->tmem_empty[abuf]);
            if (++abuf == Cfg<WM>::kAccBufs) {
                abuf = 0;
                aphase ^= 1u;
            }
        }
        if (et == 0)
            bulk_wait<0>();  // every store written before the CTA (and its smem) goes
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
    if (threadIdx.x == 0 && ctl->abort_flag && p.status)
        atomicOr(p.status, MOE_STATUS_TIMEOUT);
}

// ---- host: tensor maps ------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// bf16 (or, with `u8`, byte) tensor map, 128-byte swizzle unless `plain`;
// dims innermost first.
cudaError_t encode_bf16(CUtensorMap *m, const void *base, uint32_t rank, const cuuint64_t *dims,
                        const cuuint64_t *strides_bytes, const cuuint32_t *box, bool plain = false,
                        bool u8 = false)
{
    cudaError_t err = get_encoder();
    if (err != cudaSuccess)
        return err;
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                rank, const_cast<void *>(base),
                                dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                plain ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Weight [E, K, M] (M contiguous): boxes of 64 features x 64 K rows of one expert.
cudaError_t weight_map(CUtensorMap *m, const void *W, int E, int K, int M)
{
    const cuuint64_t dims[3] = {cuuint64_t(M), cuuint64_t(K), cuuint64_t(E)};
    const cuuint64_t strides[2] = {cuuint64_t(M) * 2, cuuint64_t(M) * K * 2};
    const cuuint32_t box[3] = {64, BK, 1};
    return encode_bf16(m, W, 3, dims, strides, box);
}

// E4M3 weight codes [E, K, M] (M contiguous): unswizzled boxes of 128
// features x 64 K rows of one expert (rows of 128 bytes).
cudaError_t weight_map_e4m3(CUtensorMap *m, const void *Wq, int E, int K, int M)
{
    const cuuint64_t dims[3] = {cuuint64_t(M), cuuint64_t(K), cuuint64_t(E)};
    const cuuint64_t strides[2] = {cuuint64_t(M), cuuint64_t(M) * K};
    const cuuint32_t box[3] = {BM, BK, 1};
    return encode_bf16(m, Wq, 3, dims, strides, box, true, true);
}

// K-major E4M3 weight codes [E, M, K] (K contiguous): 128-byte-swizzled
// boxes of 128 K x 128 features of one expert.
cudaError_t weight_map_e4m3_kmajor(CUtensorMap *m, const void *Wq, int E, int K, int M)
{
    const cuuint64_t dims[3] = {cuuint64_t(K), cuuint64_t(M), cuuint64_t(E)};
    const cuuint64_t strides[2] = {cuuint64_t(K), cuuint64_t(K) * M};
    const cuuint32_t box[3] = {128, BM, 1};
    return encode_bf16(m, Wq, 3, dims, strides, box, false, true);
}

// E4M3 rows [cap, K] (K contiguous): boxes of 128, 64, 32, 16 rows x 128 K codes.
cudaError_t rows_map_e4m3(RowMaps *m, const void *X, int64_t cap, int K)
{
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(cap)};
    const cuuint64_t strides[1] = {cuuint64_t(K)};
    for (int i = 0; i < kRowMaps; ++i) {
        const cuuint32_t box[2] = {128, cuuint32_t(BN >> i)};
        const cudaError_t e = encode_bf16(&m->h[i], X, 2, dims, strides, box, false, true);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// MXFP4 codes [E, M, K/2] (two K a byte): unswizzled boxes of 32 bytes (64
// K) x 128 features of one expert.
cudaError_t mx4_code_map(CUtensorMap *m, const void *Wq, int E, int K, int M)
{
    const cuuint64_t dims[3] = {cuuint64_t(K / 2), cuuint64_t(M), cuuint64_t(E)};
    const cuuint64_t strides[2] = {cuuint64_t(K / 2), cuuint64_t(K / 2) * M};
    const cuuint32_t box[3] = {BK / 2, BM, 1};
    return encode_bf16(m, Wq, 3, dims, strides, box, true, true);
}

// MXFP4 scale exponents [E, K/32, M]: unswizzled boxes of 128 features x 2
// blocks (64 K) of one expert.
cudaError_t mx4_scale_map(CUtensorMap *m, const void *S, int E, int K, int M)
{
    const cuuint64_t dims[3] = {cuuint64_t(M), cuuint64_t(K / 32), cuuint64_t(E)};
    const cuuint64_t strides[2] = {cuuint64_t(M), cuuint64_t(M) * (K / 32)};
    const cuuint32_t box[3] = {BM, BK / 32, 1};
    return encode_bf16(m, S, 3, dims, strides, box, true, true);
}

// Rows [cap, K] (K contiguous): boxes of 128, 64, 32, 16 rows x 64 K.
cudaError_t rows_map(RowMaps *m, const void *X, int64_t cap, int K)
{
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(cap)};
    const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
    for (int i = 0; i < kRowMaps; ++i) {
        const cuuint32_t box[2] = {BK, cuuint32_t(BN >> i)};
        const cudaError_t e = encode_bf16(&m->h[i], X, 2, dims, strides, box);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// Token rows [T, K] read four at a time by index: one-row boxes of 64 K
// (in h[0]; the other maps are unused).
cudaError_t token_rows_map(RowMaps *rm, const void *X, int T, int K)
{
    CUtensorMap *m = &rm->h[0];
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(T)};
    const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
    const cuuint32_t box[2] = {BK, 1};
    return encode_bf16(m, X, 2, dims, strides, box);
}

// Output rows [cap, M] written 16 rows x `width` features at a time from a
// dense (unswizzled) staging tile.
cudaError_t out_map(CUtensorMap *m, void *Y, int64_t cap, int M, int width)
{
    const cuuint64_t dims[2] = {cuuint64_t(M), cuuint64_t(cap)};
    const cuuint64_t strides[1] = {cuuint64_t(M) * 2};
    const cuuint32_t box[2] = {cuuint32_t(width), cuuint32_t(kStageRows)};
    return encode_bf16(m, Y, 2, dims, strides, box, true);
}

}  // namespace

cudaError_t launch_ffn_gate_up(const void *xs, const void *Wg, const void *Wu,
                               const int32_t *offsets, int E, int d, int f, int64_t cap,
                               void *H, uint32_t *status, cudaStream_t stream, int stall_cta)
{
    CUtensorMap mg, mu, mo;
    RowMaps mx;
    cudaError_t err;
    if ((err = weight_map(&mg, Wg, E, d, f)) != cudaSuccess ||
        (err = weight_map(&mu, Wu, E, d, f)) != cudaSuccess ||
        (err = rows_map(&mx, xs, cap, d)) != cudaSuccess ||
        (err = out_map(&mo, H, cap, f, Kind<true>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<true, false, kBf16>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotGateUp,
                            ffn_smem_bytes<kBf16>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, nullptr, nullptr, static_cast<uint16_t *>(H), status, cap, E, d, f,
                    stall_cta, nullptr, nullptr, nullptr};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kBf16>::kThreadsK), ffn_smem_bytes<kBf16>(E),
                      stream, mg, mu, mx, mo, mo, mo, a);
}

cudaError_t launch_ffn_gate_up_rows(const void *x, int T, const int32_t *srt_tok, const void *Wg,
                                    const void *Wu, const int32_t *offsets, int E, int d, int f,
                                    int64_t cap, void *H, uint32_t *status, cudaStream_t stream)
{
    CUtensorMap mg, mu, mo;
    RowMaps mx;
    cudaError_t err;
    if ((err = weight_map(&mg, Wg, E, d, f)) != cudaSuccess ||
        (err = weight_map(&mu, Wu, E, d, f)) != cudaSuccess ||
        (err = token_rows_map(&mx, x, T, d)) != cudaSuccess ||
        (err = out_map(&mo, H, cap, f, Kind<true>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<true, true, kBf16>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotGateUpRows,
                            ffn_smem_bytes<kBf16>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, srt_tok, nullptr, static_cast<uint16_t *>(H), status, cap, E, d, f,
                    -1, nullptr, nullptr, nullptr};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kBf16>::kThreadsK), ffn_smem_bytes<kBf16>(E),
                      stream, mg, mu, mx, mo, mo, mo, a);
}

cudaError_t launch_ffn_down(const void *H, const void *Wd, const int32_t *offsets,
                            const float *srt_w, int E, int d, int f, int64_t cap, void *Ys,
                            uint32_t *status, cudaStream_t stream)
{
    CUtensorMap mw, mo;
    RowMaps mh;
    cudaError_t err;
    if ((err = weight_map(&mw, Wd, E, f, d)) != cudaSuccess ||
        (err = rows_map(&mh, H, cap, f)) != cudaSuccess ||
        (err = out_map(&mo, Ys, cap, d, Kind<false>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<false, false, kBf16>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotDown,
                            ffn_smem_bytes<kBf16>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, nullptr, srt_w, static_cast<uint16_t *>(Ys), status, cap, E, f, d,
                    -1, nullptr, nullptr, nullptr};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kBf16>::kThreadsK), ffn_smem_bytes<kBf16>(E),
                      stream, mw, mw, mh, mo, mo, mo, a);
}

cudaError_t launch_ffn_gate_up_e4m3(const void *xs, const uint8_t *Wg, const float *sg,
                                    const uint8_t *Wu, const float *su, const int32_t *offsets,
                                    int E, int d, int f, int64_t cap, void *H, uint32_t *status,
                                    cudaStream_t stream)
{
    CUtensorMap mg, mu, mo;
    RowMaps mx;
    cudaError_t err;
    if ((err = weight_map_e4m3(&mg, Wg, E, d, f)) != cudaSuccess ||
        (err = weight_map_e4m3(&mu, Wu, E, d, f)) != cudaSuccess ||
        (err = rows_map(&mx, xs, cap, d)) != cudaSuccess ||
        (err = out_map(&mo, H, cap, f, Kind<true>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<true, false, kWiden>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotGateUpE4m3,
                            ffn_smem_bytes<kWiden>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, nullptr, nullptr, static_cast<uint16_t *>(H), status, cap, E, d, f,
                    -1, sg, su, nullptr};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kWiden>::kThreadsK), ffn_smem_bytes<kWiden>(E),
                      stream, mg, mu, mx, mo, mo, mo, a);
}

cudaError_t launch_ffn_gate_up_native(const uint8_t *xs8, const int32_t *xexp, const uint8_t *Wg,
                                      const float *sg, const uint8_t *Wu, const float *su,
                                      const int32_t *offsets, int E, int d, int f, int64_t cap,
                                      void *H, uint32_t *status, cudaStream_t stream)
{
    CUtensorMap mg, mu, mo;
    RowMaps mx;
    cudaError_t err;
    if ((err = weight_map_e4m3_kmajor(&mg, Wg, E, d, f)) != cudaSuccess ||
        (err = weight_map_e4m3_kmajor(&mu, Wu, E, d, f)) != cudaSuccess ||
        (err = rows_map_e4m3(&mx, xs8, cap, d)) != cudaSuccess ||
        (err = out_map(&mo, H, cap, f, Kind<true>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<true, false, kNative>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotGateUpNative,
                            ffn_smem_bytes<kNative>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, nullptr, nullptr, static_cast<uint16_t *>(H), status, cap, E, d, f,
                    -1, sg, su, xexp};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kNative>::kThreadsK), ffn_smem_bytes<kNative>(E),
                      stream, mg, mu, mx, mo, mo, mo, a);
}

cudaError_t launch_ffn_down_native(const uint8_t *H8, const int32_t *hexp, const uint8_t *Wd,
                                   const float *sd, const int32_t *offsets, const float *srt_w,
                                   int E, int d, int f, int64_t cap, void *Ys, uint32_t *status,
                                   cudaStream_t stream)
{
    CUtensorMap mw, mo;
    RowMaps mh;
    cudaError_t err;
    if ((err = weight_map_e4m3_kmajor(&mw, Wd, E, f, d)) != cudaSuccess ||
        (err = rows_map_e4m3(&mh, H8, cap, f)) != cudaSuccess ||
        (err = out_map(&mo, Ys, cap, d, Kind<false>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<false, false, kNative>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotDownNative,
                            ffn_smem_bytes<kNative>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, nullptr, srt_w, static_cast<uint16_t *>(Ys), status, cap, E, f, d,
                    -1, sd, sd, hexp};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kNative>::kThreadsK), ffn_smem_bytes<kNative>(E),
                      stream, mw, mw, mh, mo, mo, mo, a);
}

cudaError_t launch_ffn_down_e4m3(const void *H, const uint8_t *Wd, const float *sd,
                                 const int32_t *offsets, const float *srt_w, int E, int d, int f,
                                 int64_t cap, void *Ys, uint32_t *status, cudaStream_t stream)
{
    CUtensorMap mw, mo;
    RowMaps mh;
    cudaError_t err;
    if ((err = weight_map_e4m3(&mw, Wd, E, f, d)) != cudaSuccess ||
        (err = rows_map(&mh, H, cap, f)) != cudaSuccess ||
        (err = out_map(&mo, Ys, cap, d, Kind<false>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<false, false, kWiden>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotDownE4m3,
                            ffn_smem_bytes<kWiden>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, nullptr, srt_w, static_cast<uint16_t *>(Ys), status, cap, E, f, d,
                    -1, sd, sd, nullptr};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kWiden>::kThreadsK), ffn_smem_bytes<kWiden>(E),
                      stream, mw, mw, mh, mo, mo, mo, a);
}

cudaError_t launch_ffn_gate_up_mxfp4(const void *xs, const uint8_t *Wg, const uint8_t *sg,
                                     const uint8_t *Wu, const uint8_t *su, const int32_t *offsets,
                                     int E, int d, int f, int64_t cap, void *H, uint32_t *status,
                                     cudaStream_t stream)
{
    CUtensorMap mg, mu, msg, msu, mo;
    RowMaps mx;
    cudaError_t err;
    if ((err = mx4_code_map(&mg, Wg, E, d, f)) != cudaSuccess ||
        (err = mx4_code_map(&mu, Wu, E, d, f)) != cudaSuccess ||
        (err = mx4_scale_map(&msg, sg, E, d, f)) != cudaSuccess ||
        (err = mx4_scale_map(&msu, su, E, d, f)) != cudaSuccess ||
        (err = rows_map(&mx, xs, cap, d)) != cudaSuccess ||
        (err = out_map(&mo, H, cap, f, Kind<true>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<true, false, kMx4>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotGateUpMx4,
                            ffn_smem_bytes<kMx4>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, nullptr, nullptr, static_cast<uint16_t *>(H), status, cap, E, d, f,
                    -1, nullptr, nullptr, nullptr};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kMx4>::kThreadsK), ffn_smem_bytes<kMx4>(E),
                      stream, mg, mu, mx, mo, msg, msu, a);
}

cudaError_t launch_ffn_down_mxfp4(const void *H, const uint8_t *Wd, const uint8_t *sd,
                                  const int32_t *offsets, const float *srt_w, int E, int d, int f,
                                  int64_t cap, void *Ys, uint32_t *status, cudaStream_t stream)
{
    CUtensorMap mw, msd, mo;
    RowMaps mh;
    cudaError_t err;
    if ((err = mx4_code_map(&mw, Wd, E, f, d)) != cudaSuccess ||
        (err = mx4_scale_map(&msd, sd, E, f, d)) != cudaSuccess ||
        (err = rows_map(&mh, H, cap, f)) != cudaSuccess ||
        (err = out_map(&mo, Ys, cap, d, Kind<false>::kUnitM)) != cudaSuccess)
        return err;
    auto kern = k_ffn<false, false, kMx4>;
    err = ensure_smem_limit(reinterpret_cast<const void *>(kern), kSlotDownMx4,
                            ffn_smem_bytes<kMx4>(MOE_MAX_EXPERTS));
    if (err != cudaSuccess)
        return err;
    const FfnArgs a{offsets, nullptr, srt_w, static_cast<uint16_t *>(Ys), status, cap, E, f, d,
                    -1, nullptr, nullptr, nullptr};
    return launch_pdl(kern, dim3(device_sm_count()), dim3(Cfg<kMx4>::kThreadsK), ffn_smem_bytes<kMx4>(E),
                      stream, mw, mw, mh, mo, msd, msd, a);
}

}  // namespace moe
