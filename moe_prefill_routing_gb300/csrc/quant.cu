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

// ---- MXFP4 (OCP Microscaling, 4-bit E2M1 elements) ---------------------------------
//
// Blocks of 32 consecutive weights along K (the reduction axis) per expert
// and output feature share one power-of-two scale 2^x, stored as the byte
// S = x + 127:
//   x = floor(log2(max |W| over the block)) - 2   (2: the exponent of E2M1's
//       largest value, 6 = 1.5 x 2^2), clamped to [-127, 127]; -127 for a
//       block of zeros
//   code = the E2M1 value nearest to W / 2^x, ties to the even code (mantissa
//       bit 0), past 6 saturated, the sign kept
// Codes are stored along K ([E, M, K/2] bytes: each output feature's codes
// contiguous, 16 bytes a block), eight to a 32-bit word (little-endian): the
// word of k = 8i .. 8i + 7 holds k = 8i + 2j in bits 4j .. 4j + 3 and
// k = 8i + 2j + 1 in bits 16 + 4j .. 19 + 4j (j = 0..3), the order in which
// the GEMMs' decode takes them apart with one mask each.

namespace {

// E2M1 code of a = |W / 2^x| (the magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 are
// codes 0..7): the count of decision points a lies above; a point that is a
// tie between two codes belongs to the even one, so it counts as passed only
// when the upper code is even (>=) and not when it is odd (>).
__device__ __forceinline__ uint32_t e2m1_code(float a)
{
    return uint32_t(a > 0.25f) + uint32_t(a >= 0.75f) + uint32_t(a > 1.25f) +
           uint32_t(a >= 1.75f) + uint32_t(a > 2.5f) + uint32_t(a >= 3.5f) + uint32_t(a > 5.0f);
}

// One thread per (expert, block of 32 k, output feature m): the block's 32
// weights (stride M, coalesced across the threads), its exponent, its 32
// codes as one 16-byte store.
__global__ void __launch_bounds__(kQuantThreads)
    k_quant_mxfp4(const __nv_bfloat16 *__restrict__ W, int K, int M,
                  uint8_t *__restrict__ codes, uint8_t *__restrict__ scales)
{
    const int m = blockIdx.x * kQuantThreads + threadIdx.x;  // output feature
    const int b = blockIdx.y;                                // block along K
    const int64_t e = blockIdx.z;
    if (m >= M)
        return;
    const __nv_bfloat16 *src = W + (e * K + int64_t(b) * 32) * M + m;
    float v[32];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v[i] = __bfloat162float(src[int64_t(i) * M]);
        amax = fmaxf(amax, fabsf(v[i]));
    }
    // x from the exponent field of the block maximum (a subnormal or zero
    // maximum clamps to -127)
    const int f = int((__float_as_uint(amax) >> 23) & 0xffu);
    const int x = f == 0 ? -127 : max(-127, min(127, f - 127 - 2));
    const float r = __uint_as_float(uint32_t(127 - x) << 23);  // 2^-x, exact (x <= 125 here)
    uint32_t word[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t c = e2m1_code(fabsf(v[i]) * r) | (signbit(v[i]) ? 8u : 0u);
        word[i >> 3] |= c << (4 * ((i & 7) >> 1) + 16 * (i & 1));
    }
    *reinterpret_cast<uint4 *>(codes + (e * M + m) * int64_t(K / 2) + 16 * b) =
        make_uint4(word[0], word[1], word[2], word[3]);
    scales[(e * (K / 32) + b) * int64_t(M) + m] = uint8_t(x + 127);
}

}  // namespace

cudaError_t launch_quantize_mxfp4(const void *W, int E, int K, int M, uint8_t *codes,
                                  uint8_t *scales, cudaStream_t stream)
{
    const dim3 grid(unsigned((M + kQuantThreads - 1) / kQuantThreads), unsigned(K / 32),
                    unsigned(E));
    k_quant_mxfp4<<<grid, kQuantThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(W), K, M,
                                                      codes, scales);
    return cudaGetLastError();
}

}  // namespace moe
