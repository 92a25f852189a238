/*
 * moe_prefill.h -- C ABI of the GB300 (sm_103a) routed MoE prefill layer.
 *
 * The layer of one prefill chunk runs in four stages, each one call below:
 *
 *   moe_plan        routing plan: per-block expert histogram, exclusive scan
 *                   with each expert padded to a multiple of tm (tail rows
 *                   set to -1), stable place -> srt_tok / srt_w / pos
 *                   ("Round 4 Track C: Prefill MoE Plan (mm_clear + mm_hist +
 *                   mm_scan + mm_place) & Epilogue / Gather Audit", section 1
 *                   items 1-2, section 3)
 *   moe_gather      token rows copied into expert-sorted order (same page,
 *                   section 1 item 4)
 *   moe_expert_ffn  grouped expert FFN: gate/up projection, SwiGLU, down
 *                   projection scaled by the routing weight ("Batched resident
 *                   MoE experts on Apple Silicon: a flat parallel expert
 *                   pass", section 1); split into moe_ffn_gate_up and
 *                   moe_ffn_down for callers that time or check them apart
 *   moe_combine     per-token sum of its k weighted rows in slot order
 *                   (same page, section 3)
 *
 * moe_layer_forward runs all four on one stream; moe_prefill_forward_host
 * runs it over a sequence of chunks held in host memory.
 *
 * Conventions shared by every call
 *  - Tensors are caller-owned DEVICE pointers, row-major and contiguous
 *    (moe_prefill_forward_host alone takes host buffers for x, ids, w, y).
 *    16-bit tensors are passed as void* and hold bf16 (or fp16 where a
 *    dtype argument allows it).  16-bit row tensors (x, xs, H, Ys, y and
 *    the weights) must be 16-byte aligned, int32/fp32 arrays 4-byte aligned
 *    and workspaces 256-byte aligned (MOE_ERR_ALIGN otherwise).
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and returns once its kernels are enqueued.  The library never
 *    allocates device memory, never synchronises the host (except
 *    moe_read_status, on request) and keeps no per-call state (the one
 *    exception: moe_prefill_forward_host creates two copy streams per device
 *    on first use and a few events per call).  Kernels are chained with
 *    programmatic dependent launch.
 *  - Flat entry i = t*k + j is token t's slot j.  An expert id of -1 marks a
 *    skipped slot: it gets no row, pos = -1 and adds nothing to y.
 *  - Sizes that depend on the routing (R_pad = offsets[E], the padded row
 *    count) stay on the device; kernels size their grids for the capacity
 *    `cap` and read R_pad on the device.
 *  - A return value < 0 is an argument error found on the host before
 *    anything is enqueued (or MOE_ERR_CUDA if a launch failed).  Errors in
 *    the data (an id outside [-1, E), bad offsets, a wait that ran out its
 *    time limit) are recorded as bits of a device status word.
 *
 * The device must be sm_103 (GB300); the kernels are built for sm_103a only.
 */
#ifndef MOE_PREFILL_H
#define MOE_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points are exported from the shared library (built with hidden
 * default visibility). */
#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Same type as cudaStream_t; declared here so that this header needs no
 * CUDA header. */
struct CUstream_st;
typedef struct CUstream_st *moe_stream_t;

/* dtype of 16-bit activation rows */
#define MOE_DT_BF16 0
#define MOE_DT_F16 1

/* return codes */
#define MOE_OK 0
#define MOE_ERR_NULL (-1)      /* a required pointer is NULL */
#define MOE_ERR_SHAPE (-2)     /* a size is outside its documented range */
#define MOE_ERR_CAPACITY (-3)  /* cap < moe_capacity(T, k, E, tm) */
#define MOE_ERR_WORKSPACE (-4) /* ws_bytes smaller than required */
#define MOE_ERR_ALIGN (-5)     /* a pointer is not aligned as required */
#define MOE_ERR_CUDA (-6)      /* a CUDA call or a kernel launch failed */
#define MOE_ERR_DTYPE (-7)     /* unsupported dtype */

/* bits of the device status word */
#define MOE_STATUS_BAD_ID 1u      /* an id outside [-1, E): that slot was skipped */
#define MOE_STATUS_OVERFLOW 2u    /* padded rows exceeded cap: rows >= cap dropped */
#define MOE_STATUS_BAD_OFFSETS 4u /* offsets not ascending multiples of 16 within cap:
                                     that expert was skipped by the FFN */
#define MOE_STATUS_TIMEOUT 8u     /* a pipeline wait inside a GEMM ran out its
                                     time limit (about 2 s); the kernel stopped */

/* limits */
#define MOE_MAX_EXPERTS 4096
#define MOE_MAX_TOPK 256
#define MOE_MAX_TM 1024

/*
 * Rows that always hold the padded plan: T*k + min(E, T*k)*(tm-1).
 * Every expert pads at most tm-1 rows and at most min(E, T*k) experts are
 * routed to.  srt_tok, srt_w, xs, H and Ys need this many rows.
 * Returns -1 for negative or out-of-range sizes.
 */
MOE_API int64_t moe_capacity(int T, int k, int E, int tm);

/*
 * Device workspace of moe_plan, in bytes: a 256-byte header holding the
 * status word (uint32 at offset 0) followed by the per-block and per-group
 * expert counts of the multi-kernel plan.
 */
MOE_API size_t moe_plan_workspace_bytes(int T, int k, int E);

/*
 * moe_plan -- the routing plan ("Round 4 Track C: Prefill MoE Plan ...",
 * section 1 items 1-2; buffers as listed in section 3).
 *
 * in   ids      int32 [T, k]  expert of each (token, slot); -1 = skipped
 * in   w        fp32  [T, k]  routing weight of each (token, slot)
 * out  offsets  int32 [E+1]   offsets[e] = first row of expert e; offsets[E] = R_pad.
 *                             Each expert owns ceil(counts[e]/tm)*tm rows, in
 *                             ascending expert id.
 * out  counts   int32 [E]     routed rows of each expert
 * out  srt_tok  int32 [cap]   token of each row; -1 in pad rows
 * out  srt_w    fp32  [cap]   routing weight of each row (bit copy); +0 in pad rows
 * out  pos      int32 [T, k]  row of each (token, slot); -1 for a skipped slot
 * out  tile_expert int32 [cap/tm]  expert owning rows [n*tm, (n+1)*tm)
 * ws                          moe_plan_workspace_bytes(T, k, E) bytes
 *
 * Inside an expert, rows keep increasing flat index (token order, then
 * slot): the plan is a stable counting sort and is unique, so it is
 * bit-exact.  Only rows < R_pad and tiles < R_pad/tm are written.
 * Sizes: 0 <= T, 1 <= k <= MOE_MAX_TOPK, 1 <= E <= MOE_MAX_EXPERTS,
 * 1 <= tm <= MOE_MAX_TM, T*k < 2^31, cap >= moe_capacity(T, k, E, tm).
 * The status word is reset by every call; ids outside [-1, E) set
 * MOE_STATUS_BAD_ID and are treated as skipped.
 */
MOE_API int moe_plan(const int32_t *ids, const float *w, int T, int k, int E, int tm,
             int32_t *offsets, int32_t *counts, int32_t *srt_tok, float *srt_w,
             int32_t *pos, int32_t *tile_expert, int64_t cap, void *ws,
             size_t ws_bytes, moe_stream_t stream);

/*
 * moe_plan_noalloc -- moe_plan for callers that cannot allocate device memory.
 *
 * The paper has no counterpart: this is an interface addition.  moe_plan
 * needs a caller-provided workspace for its per-block expert counts.  Some
 * callers cannot obtain one: a serving process whose memory manager has
 * already reserved all of the GPU's memory for its own pool, or a plug-in
 * that is handed buffers by a host application and has no allocator of its
 * own.  This entry point computes exactly what moe_plan computes (same
 * kernels, same outputs, bit for bit) but keeps that scratch in a fixed
 * array inside the library, MOE_PLAN_NOALLOC_SCRATCH_BYTES of device memory
 * that every GPU which loads the library holds until the process exits.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments are those of moe_plan, without ws / ws_bytes and with
 *   status   uint32* device word that receives the MOE_STATUS_* bits of this
 *            call (reset by the call), or NULL to leave them in a word inside
 *            the library's array, which the caller cannot read: pass a word
 *            whenever a bad id or an overflow must be detected.
 * Limit: (B + ceil(B / 256)) x E <= MOE_PLAN_NOALLOC_MAX_COUNTS with
 * B = ceil(T*k / 4096) (one row of E counts per block of 4096 entries and
 * one per group of 256 blocks): T*k up to 2M entries with E = 512, up to
 * 262144 with E = 4096.  Larger sizes return MOE_ERR_WORKSPACE.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and keeps it for the life of the
 * process; make that first call before any stream capture, and do not use
 * this entry point after a cudaDeviceReset of that device (the array may
 * then sit at another address).  Every call on a device shares the same array and leaves
 * its contents behind; nothing in it has to start at zero (every count the
 * kernels read is written first by the same call), but calls that overlap on
 * the GPU (on different streams without ordering) race on it and must not
 * be issued.
 */
#define MOE_PLAN_NOALLOC_MAX_COUNTS 266240
#define MOE_PLAN_NOALLOC_SCRATCH_BYTES (256 + 4 * MOE_PLAN_NOALLOC_MAX_COUNTS)
MOE_API int moe_plan_noalloc(const int32_t *ids, const float *w, int T, int k, int E, int tm,
                             int32_t *offsets, int32_t *counts, int32_t *srt_tok, float *srt_w,
                             int32_t *pos, int32_t *tile_expert, int64_t cap, uint32_t *status,
                             moe_stream_t stream);

/*
 * moe_gather -- rows into expert-sorted order (same page, section 1 item 4).
 *
 * in   x        16-bit [T, d]   token activations (dtype MOE_DT_BF16 or MOE_DT_F16)
 * in   srt_tok  int32 [cap]     from moe_plan
 * in   offsets  int32 [E+1]     from moe_plan (R_pad = offsets[E] read on the device)
 * out  xs       16-bit [cap, d] xs[r] = x[srt_tok[r]]; all-zero bits where srt_tok[r] = -1.
 *                               Rows >= R_pad are not written.
 * d must be a positive multiple of 8 (16-byte rows).  A bit copy.
 */
MOE_API int moe_gather(const void *x, int dtype, int T, int d, const int32_t *srt_tok,
               const int32_t *offsets, int E, int64_t cap, void *xs,
               moe_stream_t stream);

/*
 * moe_ffn_gate_up -- grouped gate/up projection with SwiGLU.
 *
 * For each expert e and each of its rows r in [offsets[e], offsets[e+1]):
 *   g = xs[r] . Wg[e],  u = xs[r] . Wu[e]   (bf16 operands, fp32 accumulation)
 *   H[r] = bf16(silu(g) * u),  silu(z) = z / (1 + e^-z)
 * in   xs       bf16 [cap, d]
 * in   Wg, Wu   bf16 [E, d, f]
 * in   offsets  int32 [E+1]   ascending multiples of 16, offsets[E] <= cap
 * out  H        bf16 [cap, f] rows < R_pad written
 * in   status   uint32* device word to OR error bits into, or NULL
 * d and f must be positive multiples of 64.
 */
MOE_API int moe_ffn_gate_up(const void *xs, const void *Wg, const void *Wu,
                    const int32_t *offsets, int E, int d, int f, int64_t cap,
                    void *H, uint32_t *status, moe_stream_t stream);

/*
 * moe_ffn_gate_up_rows -- moe_ffn_gate_up reading each routed row straight
 * from the token activations: row r of expert e is x[srt_tok[r]] (a zero
 * row where srt_tok[r] = -1), fetched four rows at a time by TMA gather4,
 * so the gathered copy xs is never written.  Same arithmetic and result as
 * moe_gather followed by moe_ffn_gate_up, bit for bit.  On GB300 the
 * gather4 loads make this slower than the separate 128-bit gather plus tiled
 * loads, so moe_layer_forward does not use it.
 * in   x        bf16 [T, d]
 * in   srt_tok  int32 [cap]   from moe_plan
 * other arguments as in moe_ffn_gate_up.
 */
MOE_API int moe_ffn_gate_up_rows(const void *x, int T, const int32_t *srt_tok, const void *Wg,
                                 const void *Wu, const int32_t *offsets, int E, int d, int f,
                                 int64_t cap, void *H, uint32_t *status, moe_stream_t stream);

/*
 * moe_ffn_down -- grouped down projection scaled by the routing weight.
 *
 *   Ys[r] = bf16(srt_w[r] * (H[r] . Wd[e]))   (fp32 accumulation)
 * in   H        bf16 [cap, f]
 * in   Wd       bf16 [E, f, d]
 * in   offsets  int32 [E+1]
 * in   srt_w    fp32 [cap]
 * out  Ys       bf16 [cap, d] rows < R_pad written
 */
MOE_API int moe_ffn_down(const void *H, const void *Wd, const int32_t *offsets,
                 const float *srt_w, int E, int d, int f, int64_t cap, void *Ys,
                 uint32_t *status, moe_stream_t stream);

/* moe_expert_ffn -- moe_ffn_gate_up then moe_ffn_down; H is caller scratch
 * of cap*f bf16. */
MOE_API int moe_expert_ffn(const void *xs, const void *Wg, const void *Wu, const void *Wd,
                   const int32_t *offsets, const float *srt_w, int E, int d, int f,
                   int64_t cap, void *H, void *Ys, uint32_t *status,
                   moe_stream_t stream);

/*
 * moe_combine -- y[t] = sum over j = 0..k-1, in that order, of Ys[pos[t*k+j]]
 * ("Batched resident MoE experts on Apple Silicon ...", section 3: the same
 * per-token top-k summation order).  fp32 accumulation from zero, one bf16
 * rounding at the end; slots with pos = -1 add nothing.
 * in   Ys   bf16 [*, d]   weighted expert rows (from moe_ffn_down)
 * in   pos  int32 [T, k]
 * out  y    bf16 [T, d]
 * d must be a positive multiple of 8.
 */
MOE_API int moe_combine(const void *Ys, const int32_t *pos, int T, int k, int d, void *y,
                moe_stream_t stream);

/* Fields of the moe_layer_forward workspace (byte offsets, see
 * moe_workspace_layout).  The plan's own workspace (status word + counts)
 * sits at offset 0, so moe_read_status works on either workspace. */
#define MOE_WS_STATUS 0
#define MOE_WS_BCNT 1
#define MOE_WS_OFFSETS 2
#define MOE_WS_COUNTS 3
#define MOE_WS_SRT_TOK 4
#define MOE_WS_SRT_W 5
#define MOE_WS_POS 6
#define MOE_WS_TILE_EXPERT 7
#define MOE_WS_XS 8
#define MOE_WS_H 9
#define MOE_WS_YS 10
#define MOE_WS_TOTAL 11
#define MOE_WS_FIELDS 12

/* Device workspace of moe_layer_forward, in bytes (0 on bad sizes). */
MOE_API size_t moe_workspace_bytes(int T, int d, int E, int k, int f, int tm);

/* Byte offset of every MOE_WS_* field inside that workspace (out has
 * MOE_WS_FIELDS entries; out[MOE_WS_TOTAL] = total bytes).  Host only. */
MOE_API int moe_workspace_layout(int T, int d, int E, int k, int f, int tm, size_t *out);

/*
 * moe_layer_forward -- the whole routed MoE layer of one prefill chunk:
 * moe_plan -> moe_gather -> moe_ffn_gate_up -> moe_ffn_down -> moe_combine.
 *
 * in   x        bf16 [T, d]
 * in   ids, w   [T, k] as in moe_plan
 * in   Wg, Wu   bf16 [E, d, f];  Wd bf16 [E, f, d]
 * out  y        bf16 [T, d]
 * ws            moe_workspace_bytes(T, d, E, k, f, tm) bytes, 256-byte aligned;
 *               it holds the plan, xs, H and Ys (see moe_workspace_layout)
 * tm must be a multiple of 16; d and f multiples of 64.
 */
MOE_API int moe_layer_forward(const void *x, const int32_t *ids, const float *w,
                      const void *Wg, const void *Wu, const void *Wd, int T, int d,
                      int E, int k, int f, int tm, void *y, void *ws, size_t ws_bytes,
                      moe_stream_t stream);

/*
 * E4M3 expert weights.  "Round 4 Track C: Prefill MoE Plan ...", section 2,
 * runs the experts from quantized weight packs (8-, 4- and 2-bit block
 * formats).  The GEMMs stream the expert weights from HBM, so holding them
 * in 8 bits halves the layer's dominant traffic.  The packed form is the
 * OCP E4M3 format (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * largest finite 448) with one fp32 scale per expert and output feature:
 *   scale[e][m] = max_k |W[e][k][m]| / 448   (1 when that is 0)
 *   q[e][k][m]  = E4M3 nearest to W[e][k][m] / scale[e][m] (ties to even,
 *                 saturated at +-448), both divisions IEEE fp32
 * and the weight the GEMMs use is value(q) * scale.  Activations, H, Ys and
 * y stay bf16; accumulation is fp32.  The GEMMs widen each 8-bit tile to
 * bf16 in shared memory (exact) and apply the scale in their epilogue.
 *
 * moe_quantize_e4m3 -- W bf16 [E, K, M] (M = output features, contiguous)
 * -> q uint8 [E, K, M] (kmajor = 0) or [E, M, K] (kmajor = 1, K and M
 * multiples of 64; the layout moe_ffn_gate_up_f8 reads), scale fp32
 * [E, M].  W must be finite.  A one-time preparation, not part of the layer.
 */
MOE_API int moe_quantize_e4m3(const void *W, int E, int K, int M, uint8_t *q, float *scale,
                              int kmajor, moe_stream_t stream);

/* moe_ffn_gate_up / moe_ffn_down with E4M3 weights: Wg, Wu uint8 [E, d, f]
 * with scales sg, su fp32 [E, f]; Wd uint8 [E, f, d] with scales sd fp32
 * [E, d] (16-byte aligned codes, 4-byte aligned scales).  Everything else
 * as in the bf16 calls. */
MOE_API int moe_ffn_gate_up_e4m3(const void *xs, const uint8_t *Wg, const float *sg,
                                 const uint8_t *Wu, const float *su, const int32_t *offsets,
                                 int E, int d, int f, int64_t cap, void *H, uint32_t *status,
                                 moe_stream_t stream);
MOE_API int moe_ffn_down_e4m3(const void *H, const uint8_t *Wd, const float *sd,
                              const int32_t *offsets, const float *srt_w, int E, int d, int f,
                              int64_t cap, void *Ys, uint32_t *status, moe_stream_t stream);

/*
 * E4M3 activations for the gate/up projection, so that it runs on 8-bit
 * operands (tcgen05.mma.kind::f8f6f4) with no widening.  Each routed row
 * gets a power-of-two scale 2^e, e the smallest integer with
 * max |row| <= 448 * 2^e (0 for a zero or pad row); its codes are the
 * nearest E4M3 values of row * 2^-e (exact scaling, ties to even).
 *
 * moe_gather_e4m3 -- moe_gather with E4M3 rows: xs8 uint8 [cap, d] and
 * xexp int32 [cap] (the e of each row) for rows < R_pad.  d a multiple of
 * 16; x, xs8 16-byte aligned.
 *
 * moe_ffn_gate_up_f8 -- H[r] = bf16(silu(g) * u) with g = 2^xexp[r] *
 * sg[e] * (codes of row r . Wg codes), fp32 accumulation, likewise u: Wg, Wu
 * K-major E4M3 codes [E, f, d] (moe_quantize_e4m3 with kmajor = 1), scales
 * [E, f].
 *
 * moe_rows_e4m3 -- the same per-row quantization of H [cap, f] bf16 itself
 * (rows < offsets[E]): H8 uint8 [cap, f], hexp int32 [cap].  f a multiple
 * of 16.
 *
 * moe_ffn_down_f8 -- Ys[r] = bf16(srt_w[r] * 2^hexp[r] * sd[e] * (codes of
 * H row r . Wd codes)), fp32 accumulation: Wd K-major E4M3 codes [E, d, f]
 * (moe_quantize_e4m3 of Wd [E, f, d] with kmajor = 1), scales sd [E, d].
 */
MOE_API int moe_gather_e4m3(const void *x, int T, int d, const int32_t *srt_tok,
                            const int32_t *offsets, int E, int64_t cap, uint8_t *xs8,
                            int32_t *xexp, moe_stream_t stream);
MOE_API int moe_ffn_gate_up_f8(const uint8_t *xs8, const int32_t *xexp, const uint8_t *Wg,
                               const float *sg, const uint8_t *Wu, const float *su,
                               const int32_t *offsets, int E, int d, int f, int64_t cap, void *H,
                               uint32_t *status, moe_stream_t stream);
MOE_API int moe_rows_e4m3(const void *H, int f, const int32_t *offsets, int E, int64_t cap,
                          uint8_t *H8, int32_t *hexp, moe_stream_t stream);
MOE_API int moe_ffn_down_f8(const uint8_t *H8, const int32_t *hexp, const uint8_t *Wd,
                            const float *sd, const int32_t *offsets, const float *srt_w, int E,
                            int d, int f, int64_t cap, void *Ys, uint32_t *status,
                            moe_stream_t stream);

/* moe_layer_forward with E4M3 weights (as above); same workspace
 * (moe_workspace_bytes) and outputs. */
MOE_API int moe_layer_forward_e4m3(const void *x, const int32_t *ids, const float *w,
                                   const uint8_t *Wg, const float *sg, const uint8_t *Wu,
                                   const float *su, const uint8_t *Wd, const float *sd, int T,
                                   int d, int E, int k, int f, int tm, void *y, void *ws,
                                   size_t ws_bytes, moe_stream_t stream);

/* moe_layer_forward_f8 -- the layer with both projections on 8-bit
 * operands: moe_gather_e4m3 -> moe_ffn_gate_up_f8 (Wg, Wu K-major codes
 * [E, f, d]) -> moe_rows_e4m3 -> moe_ffn_down_f8 (Wd K-major codes
 * [E, d, f]) -> moe_combine.  Same workspace (the E4M3 rows and their
 * exponents, first of x then of H, sit in its xs field). */
MOE_API int moe_layer_forward_f8(const void *x, const int32_t *ids, const float *w,
                                 const uint8_t *Wg, const float *sg, const uint8_t *Wu,
                                 const float *su, const uint8_t *Wd, const float *sd, int T,
                                 int d, int E, int k, int f, int tm, void *y, void *ws,
                                 size_t ws_bytes, moe_stream_t stream);

/*
 * MXFP4 expert weights (4 bits a weight).  The same page (section 2) runs
 * experts from 4-bit block formats; here the 4-bit form is MXFP4 of the OCP
 * Microscaling (MX) specification: E2M1 elements (1 sign, 2 exponent bits
 * with bias 1, 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) in
 * blocks of 32 along K (the reduction axis), each block of each expert and
 * output feature sharing a power-of-two scale 2^(S-127), S one byte:
 *   x = floor(log2(max |W| over the block)) - 2, clamped to [-127, 127]
 *       (-127 for a block of zeros); S = x + 127
 *   code = E2M1 nearest to W / 2^x (ties to the even code, past 6
 *          saturated, the sign kept)
 * and the weight the GEMMs use is value(code) * 2^x, which is exactly a bf16
 * value.  Activations, H, Ys and y stay bf16, accumulation fp32: the layer
 * on MXFP4 weights is the bf16 layer on the dequantized weights.  The GEMMs
 * load the 4-bit codes and the scales with TMA and decode them to bf16 into
 * tensor memory, where the tensor cores read them.
 *
 * moe_quantize_mxfp4 -- W bf16 [E, K, M] (M = output features, contiguous;
 * K a multiple of 32, M even; 4-byte aligned) -> codes uint8 [E, M, K/2]
 * (each output feature's codes contiguous along K, eight to a little-endian
 * 32-bit word: the word of k = 8i .. 8i + 7 holds k = 8i + 2j in bits
 * 4j .. 4j + 3 and k = 8i + 2j + 1 in bits 16 + 4j .. 19 + 4j; 16-byte
 * aligned) and scales uint8 [E, K/32, M] (S).  W must be finite.  A one-time preparation, not
 * part of the layer.
 *
 * moe_ffn_gate_up_mxfp4 / moe_ffn_down_mxfp4 -- moe_ffn_gate_up /
 * moe_ffn_down with MXFP4 weights: Wg, Wu codes [E, f, d/2] with scales
 * xg, xu [E, d/32, f]; Wd codes [E, d, f/2] with scales xd [E, f/32, d]
 * (codes and scales 16-byte aligned).  Everything else as in the bf16 calls.
 *
 * moe_layer_forward_mxfp4 -- moe_layer_forward with MXFP4 weights (as
 * above); same workspace (moe_workspace_bytes) and outputs.
 */
MOE_API int moe_quantize_mxfp4(const void *W, int E, int K, int M, uint8_t *codes,
                               uint8_t *scales, moe_stream_t stream);
MOE_API int moe_ffn_gate_up_mxfp4(const void *xs, const uint8_t *Wg, const uint8_t *xg,
                                  const uint8_t *Wu, const uint8_t *xu, const int32_t *offsets,
                                  int E, int d, int f, int64_t cap, void *H, uint32_t *status,
                                  moe_stream_t stream);
MOE_API int moe_ffn_down_mxfp4(const void *H, const uint8_t *Wd, const uint8_t *xd,
                               const int32_t *offsets, const float *srt_w, int E, int d, int f,
                               int64_t cap, void *Ys, uint32_t *status, moe_stream_t stream);
MOE_API int moe_layer_forward_mxfp4(const void *x, const int32_t *ids, const float *w,
                                    const uint8_t *Wg, const uint8_t *xg, const uint8_t *Wu,
                                    const uint8_t *xu, const uint8_t *Wd, const uint8_t *xd,
                                    int T, int d, int E, int k, int f, int tm, void *y, void *ws,
                                    size_t ws_bytes, moe_stream_t stream);

/*
 * moe_prefill_forward_host -- moe_layer_forward over n_chunks prefill
 * chunks of T tokens each, taken from and returned to HOST memory.  The
 * pages run the layer chunk by chunk over a prompt ("Round 4 Track C:
 * Prefill MoE Plan ...", Table 2.1; "#372 Prompt path ...", prompts of
 * 2K-32K tokens); the host transfers and their overlap have no counterpart
 * there.  For every chunk c: x_h[c], ids_h[c], w_h[c] are copied to the
 * device, the layer runs on `stream`, and y is copied to y_h[c].  Two copy
 * streams (created once per device, shared by every call) and two sets of
 * staging buffers in ws let chunk c+1's inputs come in and chunk c-1's y go
 * out while chunk c runs.
 * in   x_h[c]    bf16 [T, d]  host memory, page-locked for the copies to overlap
 * in   ids_h[c]  int32 [T, k], w_h[c] fp32 [T, k]  host memory, as in moe_plan
 * out  y_h[c]    bf16 [T, d]  host memory
 * in   Wg, Wu, Wd, T, d, E, k, f, tm  device weights and shapes as in
 *                moe_layer_forward (T is the size of every chunk)
 * in   sg, su, sd  NULL for bf16 weights; with E4M3 weights (codes in Wg,
 *                Wu, Wd) their scales, as in moe_layer_forward_e4m3
 * in   act_e4m3  0, or 1 to run each chunk as moe_layer_forward_f8
 * ws            moe_prefill_host_workspace_bytes(...) device bytes, 256-byte
 *               aligned: the layer's workspace (moe_workspace_bytes, at offset
 *               0, so moe_read_status works on it) then the staging buffers
 * The pointer arrays are read during the call only; the host buffers must
 * stay valid, and x/ids/w unchanged, until `stream` has completed, which is
 * also when every y_h[c] is written.  Chunks may share input pointers; if
 * several y_h[c] are the same buffer it ends holding the last of them.
 * Returns MOE_ERR_* from the argument checks before anything is enqueued;
 * MOE_ERR_CUDA if a CUDA call fails part-way (synchronize the device before
 * reusing ws or the host buffers).  Calls from several host threads on one
 * device share the copy streams and so serialize their copies.
 */
MOE_API size_t moe_prefill_host_workspace_bytes(int T, int d, int E, int k, int f, int tm);
MOE_API int moe_prefill_forward_host(int n_chunks, const void *const *x_h,
                                     const int32_t *const *ids_h, const float *const *w_h,
                                     void *const *y_h, const void *Wg, const void *Wu,
                                     const void *Wd, const float *sg, const float *su,
                                     const float *sd, int act_e4m3, int T, int d, int E, int k,
                                     int f, int tm, void *ws, size_t ws_bytes,
                                     moe_stream_t stream);

/*
 * moe_read_status -- copy the status word at ws (a plan or layer workspace)
 * to *status, synchronising `stream` only.
 */
MOE_API int moe_read_status(const void *ws, moe_stream_t stream, uint32_t *status);

/*
 * moe_selftest_wait_limit -- failure-detection self-test of the GEMMs'
 * bounded waits.  Runs moe_ffn_gate_up on the given arguments with one
 * change: CTA `cta`'s first pipeline stage expects 16 bytes that never
 * arrive, so that CTA's waits run out their time limit (about 2 s), it lets
 * its issued copies and MMAs land, frees its tensor memory and stops; the
 * other CTAs finish normally.  Afterwards *status has MOE_STATUS_TIMEOUT set
 * and the context stays usable.  status must not be NULL.  Rows of the
 * stopped CTA's work units are left unwritten in H.  For tests only.
 */
MOE_API int moe_selftest_wait_limit(const void *xs, const void *Wg, const void *Wu,
                                    const int32_t *offsets, int E, int d, int f, int64_t cap,
                                    void *H, uint32_t *status, int cta, moe_stream_t stream);

/* Human-readable text of a return code. */
MOE_API const char *moe_status_str(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PREFILL_H */
