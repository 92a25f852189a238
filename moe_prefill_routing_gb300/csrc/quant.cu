// Expert weights in 8-bit floating point (E4M3) with one fp32 scale per
// expert and output feature.
//
// "Round 4 Track C: Prefill MoE Plan ...", section 2, runs the experts from
// quantized weight packs (8-, 4- and 2-bit block formats); the GEMMs here
// are bound by streaming the weights from HBM, so storing them in 8 bits
// halves the dominant traffic.  The packed form is the OCP E4M3 format (the
// one GB300 converts in hardware) with a per-(expert, output feature)
// scale, applied in the GEMM epilogue:
//   scale[e][m] = max_k |W[e][k][m]| / 448   (1 when that is 0)
//   q[e][k][m]  = E4M3 nearest to W[e][k][m] / scale[e][m], saturated at 448
// Both divisions are IEEE fp32 round-to-nearest, so the codes are a pure
// function of the weights.  This is a one-time preparation, not part of
// the layer's hot path.
#include "../../include/moe_prefill.h"
#include "internal.h"

#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace moe {
namespace {

constexpr int kQuantThreads = 256;

// One thread per output feature m of one expert: a pass over K for the
// largest magnitude, then a pass writing the codes.  Adjacent threads take
// adjacent features, so every row access of a warp is contiguous.
__global__ void __launch_bounds__(kQuantThreads)
    k_quantize_e4m3(const __nv_bfloat16 *__restrict__ W, int K, int M, uint8_t *__restrict__ q,
                    float *__restrict__ scale)
{
    const int m = blockIdx.x * kQuantThreads + threadIdx.x;
    const int64_t e = blockIdx.y;
    if (m >= M)
        return;
    const __nv_bfloat16 *col = W + e * K * int64_t(M) + m;
    float amax = 0.0f;
    for (int k = 0; k < K; ++k)
        amax = fmaxf(amax, fabsf(__bfloat162float(col[int64_t(k) * M])));
    float s = __fdiv_rn(amax, 448.0f);
    if (s == 0.0f)
        s = 1.0f;
    scale[e * M + m] = s;
    uint8_t *qc = q + e * K * int64_t(M) + m;
    for (int k = 0; k < K; ++k) {
        const float v = __fdiv_rn(__bfloat162float(col[int64_t(k) * M]), s);
        qc[int64_t(k) * M] = __nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
    }
}

}  // namespace

cudaError_t launch_quantize_e4m3(const void *W, int E, int K, int M, uint8_t *q, float *scale,
                                 cudaStream_t stream)
{
    const dim3 grid(unsigned((M + kQuantThreads - 1) / kQuantThreads), unsigned(E));
    k_quantize_e4m3<<<grid, kQuantThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(W), K, M, q, scale);
    return cudaGetLastError();
}

}  // namespace moe
