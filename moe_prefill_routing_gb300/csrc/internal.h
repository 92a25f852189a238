// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

// ---- routing plan (plan.cu) ------------------------------------------------

// Flat entries per block of the multi-kernel plan (inputs above the
// one-launch cluster plan): 8 warps x 16 steps x 32 entries.
constexpr int kPlanBlockEntries = 4096;

inline int plan_num_blocks(int64_t n)
{
    return static_cast<int>((n + kPlanBlockEntries - 1) / kPlanBlockEntries);
}

// The column scan over blocks runs in groups of this many blocks; the
// expert scan then adds the groups' totals.
constexpr int kPlanGroupBlocks = 256;

inline int plan_num_groups(int nblk)
{
    return (nblk + kPlanGroupBlocks - 1) / kPlanGroupBlocks;
}

// The multi-kernel plan's scratch: one row of E int32 per block (its
// counts, then the rows of its group's earlier blocks), then one per group
// (the group's totals, then the rows of the earlier groups).
inline int64_t plan_count_rows(int64_t n)
{
    const int nblk = plan_num_blocks(n);
    return int64_t(nblk) + plan_num_groups(nblk);
}

cudaError_t launch_plan(const int32_t *ids, const float *w, int T, int k, int E, int tm,
                        int32_t *offsets, int32_t *counts, int32_t *srt_tok, float *srt_w,
                        int32_t *pos, int32_t *tile_expert, int64_t cap, uint32_t *status,
                        int32_t *bcnt, cudaStream_t stream);

// ---- row kernels (rows.cu) ---------------------------------------------------

cudaError_t launch_gather(const void *x, int T, int d, const int32_t *srt_tok,
                          const int32_t *offsets, int E, int64_t cap, void *xs,
                          cudaStream_t stream);

cudaError_t launch_combine(const void *Ys, const int32_t *pos, int T, int k, int d, void *y,
                           cudaStream_t stream);

// ---- grouped expert GEMMs (ffn.cu) -------------------------------------------

// stall_cta >= 0 only in the failure-detection self-test (moe_selftest_wait_limit).
cudaError_t launch_ffn_gate_up(const void *xs, const void *Wg, const void *Wu,
                               const int32_t *offsets, int E, int d, int f, int64_t cap,
                               void *H, uint32_t *status, cudaStream_t stream,
                               int stall_cta = -1);

// gate/up with the B rows gathered from x [T, d] by srt_tok (no xs).
cudaError_t launch_ffn_gate_up_rows(const void *x, int T, const int32_t *srt_tok, const void *Wg,
                                    const void *Wu, const int32_t *offsets, int E, int d, int f,
                                    int64_t cap, void *H, uint32_t *status, cudaStream_t stream);

cudaError_t launch_ffn_down(const void *H, const void *Wd, const int32_t *offsets,
                            const float *srt_w, int E, int d, int f, int64_t cap, void *Ys,
                            uint32_t *status, cudaStream_t stream);

// E4M3 rows for the gate/up GEMM on E4M3 operands (codes [cap, d], row
// exponents [cap]); see rows.cu.
cudaError_t launch_gather_e4m3(const void *x, int T, int d, const int32_t *srt_tok,
                               const int32_t *offsets, int E, int64_t cap, uint8_t *xs8,
                               int32_t *xexp, cudaStream_t stream);

// The same quantization of the T token rows of x once (x8 [T, d], texp [T]),
// then the routed rows gathered as bytes with their exponents: equal to
// launch_gather_e4m3, without quantizing a token once per slot.
cudaError_t launch_quant_tokens_e4m3(const void *x, int T, int d, uint8_t *x8, int32_t *texp,
                                     cudaStream_t stream);
cudaError_t launch_gather_codes(const uint8_t *x8, const int32_t *texp, int T, int d,
                                const int32_t *srt_tok, const int32_t *offsets, int E,
                                int64_t cap, uint8_t *xs8, int32_t *xexp, cudaStream_t stream);

// E4M3 rows of H [cap, f] itself (rows < offsets[E]).
cudaError_t launch_rows_e4m3(const void *H, int f, const int32_t *offsets, int E, int64_t cap,
                             uint8_t *H8, int32_t *hexp, cudaStream_t stream);

// E4M3 weights (codes [E, K, M]) with fp32 scales [E, M]; see quant.cu.
cudaError_t launch_quantize_e4m3(const void *W, int E, int K, int M, uint8_t *q, float *scale,
                                 bool kmajor, cudaStream_t stream);
cudaError_t launch_ffn_gate_up_e4m3(const void *xs, const uint8_t *Wg, const float *sg,
                                    const uint8_t *Wu, const float *su, const int32_t *offsets,
                                    int E, int d, int f, int64_t cap, void *H, uint32_t *status,
                                    cudaStream_t stream);
// gate/up on E4M3 rows (xs8 [cap, d], row exponents xexp) and K-major E4M3
// weight codes Wg, Wu [E, f, d] with scales [E, f].
cudaError_t launch_ffn_gate_up_native(const uint8_t *xs8, const int32_t *xexp, const uint8_t *Wg,
                                      const float *sg, const uint8_t *Wu, const float *su,
                                      const int32_t *offsets, int E, int d, int f, int64_t cap,
                                      void *H, uint32_t *status, cudaStream_t stream);
// down on E4M3 rows of H (H8 [cap, f], exponents hexp) and K-major E4M3
// codes Wd [E, d, f] with scales [E, d].
cudaError_t launch_ffn_down_native(const uint8_t *H8, const int32_t *hexp, const uint8_t *Wd,
                                   const float *sd, const int32_t *offsets, const float *srt_w,
                                   int E, int d, int f, int64_t cap, void *Ys, uint32_t *status,
                                   cudaStream_t stream);
cudaError_t launch_ffn_down_e4m3(const void *H, const uint8_t *Wd, const float *sd,
                                 const int32_t *offsets, const float *srt_w, int E, int d, int f,
                                 int64_t cap, void *Ys, uint32_t *status, cudaStream_t stream);

// MXFP4 weights: codes [E, M, K/2] (4-bit E2M1 codes along K, eight to a
// 32-bit word in the order quant.cu gives) and scale exponents [E, K/32, M]
// (2^(S-127)); see quant.cu.  The GEMMs decode them to bf16 into tensor memory.
cudaError_t launch_quantize_mxfp4(const void *W, int E, int K, int M, uint8_t *codes,
                                  uint8_t *scales, cudaStream_t stream);
cudaError_t launch_ffn_gate_up_mxfp4(const void *xs, const uint8_t *Wg, const uint8_t *sg,
                                     const uint8_t *Wu, const uint8_t *su, const int32_t *offsets,
                                     int E, int d, int f, int64_t cap, void *H, uint32_t *status,
                                     cudaStream_t stream);
cudaError_t launch_ffn_down_mxfp4(const void *H, const uint8_t *Wd, const uint8_t *sd,
                                  const int32_t *offsets, const float *srt_w, int E, int d, int f,
                                  int64_t cap, void *Ys, uint32_t *status, cudaStream_t stream);

// ---- launch helpers (api.cu) -------------------------------------------------

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Raise a kernel's dynamic shared-memory limit once per device.
cudaError_t ensure_smem_limit(const void *kernel, int slot, size_t bytes);

// Launch with programmatic dependent launch allowed: the kernel may begin
// while its predecessor in the stream finishes; every kernel here calls
// griddepcontrol.wait before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Slots of ensure_smem_limit's per-device cache.
enum SmemSlot {
    kSlotPlaceOr = 0,      // the large-input place kernel with shared-memory lane words
    kSlotPlaceBallot0,     // ... with ballots, for ids of 0 .. 12 bits
    kSlotPlaceBallot12 = kSlotPlaceBallot0 + 12,
    kSlotHist,
    kSlotGateUp,
    kSlotGateUpRows,
    kSlotDown,
    kSlotGateUpE4m3,
    kSlotDownE4m3,
    kSlotGateUpNative,
    kSlotDownNative,
    kSlotGateUpMx4,
    kSlotDownMx4,
    kSlotCount
};

}  // namespace moe
