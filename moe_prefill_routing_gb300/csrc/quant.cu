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
constexpr int kTile = 64;  // K-major codes: 64 x 64 tiles transposed through shared memory

// One thread per output feature m of one expert: the largest magnitude
// over K, then the scale.  Adjacent threads take adjacent features, so
// every row access of a warp is contiguous.
__global__ void __launch_bounds__(kQuantThreads)
    k_quant_scales(const __nv_bfloat16 *__restrict__ W, int K, int M, float *__restrict__ scale)
{
    const int m = blockIdx.x * kQuantThreads + threadIdx.x;
    const int64_t e = blockIdx.y;
    if (m >= M)
        return;
    const __nv_bfloat16 *col = W + e * K * int64_t(M) + m;
    float amax = 0.0f;
    for (int k = 0; k < K; ++k)
        amax = fmaxf(amax, fabsf(__bfloat162float(col[int64_t(k) * M])));
    const float s = __fdiv_rn(amax, 448.0f);
    scale[e * M + m] = s == 0.0f ? 1.0f : s;
}

__device__ __forceinline__ uint8_t e4m3_code(__nv_bfloat16 w, float s)
{
    return __nv_cvt_float_to_fp8(__fdiv_rn(__bfloat162float(w), s), __NV_SATFINITE, __NV_E4M3);
}

// Codes in the weights' own layout [E, K, M].
__global__ void __launch_bounds__(kQuantThreads)
    k_quant_codes_mn(const __nv_bfloat16 *__restrict__ W, int K, int M,
                     const float *__restrict__ scale, uint8_t *__restrict__ q)
{
    const int m = blockIdx.x * kQuantThreads + threadIdx.x;
    const int64_t e = blockIdx.y;
    if (m >= M)
        return;
    const float s = scale[e * M + m];
    const int64_t base = e * K * int64_t(M) + m;
    for (int k = 0; k < K; ++k)
        q[base + int64_t(k) * M] = e4m3_code(W[base + int64_t(k) * M], s);
}

// Codes transposed to [E, M, K] (K contiguous): block (m-tile, k-tile, e)
// reads a 64 x 64 tile along M, writes it along K.
__global__ void __launch_bounds__(kQuantThreads)
    k_quant_codes_km(const __nv_bfloat16 *__restrict__ W, int K, int M,
                     const float *__restrict__ scale, uint8_t *__restrict__ q)
{
    __shared__ uint8_t tile[kTile][kTile + 4];
    const int m0 = blockIdx.x * kTile, k0 = blockIdx.y * kTile;
    const int64_t e = blockIdx.z;
    const int tx = threadIdx.x & (kTile - 1), ty = threadIdx.x / kTile;  // 64 x 4
    const float s = scale[e * M + m0 + tx];
    for (int r = ty; r < kTile; r += kQuantThreads / kTile) {
        const int64_t i = (e * K + k0 + r) * int64_t(M) + m0 + tx;
        tile[tx][r] = e4m3_code(W[i], s);
    }
    __syncthreads();
    for (int r = ty; r < kTile; r += kQuantThreads / kTile)
        q[(e * M + m0 + r) * int64_t(K) + k0 + tx] = tile[r][tx];
}

}  // namespace

cudaError_t launch_quantize_e4m3(const void *W, int E, int K, int M, uint8_t *q, float *scale,
                                 bool kmajor, cudaStream_t stream)
{
    const __nv_bfloat16 *w = static_cast<const __nv_bfloat16 *>(W);
    const dim3 grid(unsigned((M + kQuantThreads - 1) / kQuantThreads), unsigned(E));
    k_quant_scales<<<grid, kQuantThreads, 0, stream>>>(w, K, M, scale);
    if (kmajor)
        k_quant_codes_km<<<dim3(unsigned(M / kTile), unsigned(K / kTile), unsigned(E)),
                           kQuantThreads, 0, stream>>>(w, K, M, scale, q);
    else
        k_quant_codes_mn<<<grid, kQuantThreads, 0, stream>>>(w, K, M, scale, q);
    return cudaGetLastError();
}

}  // namespace moe
