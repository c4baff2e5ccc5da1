// Per-token FP8 (E4M3) quantisation on sm_103a: the indexer's input step.
//
// The indexer runs in FP8 with one scale per token ("AMD Instinct MI355X GPUs
// Power DeepSeek-V3.2-Exp", section "DeepSeek Sparse Attention (DSA)", item 1;
// release summary "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency with
// DeepSeek Sparse Attention", section "Method"); the gist page's indexer test
// script casts along chosen dimensions to E4M3 with an option for power-of-two
// (UE8M0) scales.  For each row of `cols` fp32 values:
//     mode 0   scale = amax / 448                 (1 for an all-zero row)
//     mode 1   scale = smallest power of two >= amax / 448   (1 for zero rows)
//     code     E4M3 nearest to x / scale, ties to even, saturated to +-448
// Both divisions are IEEE single precision (correctly rounded), so the codes
// are a function of the fp32 inputs alone.
//
// HBM-bound: 4 bytes read and 1 byte written per value.  A thread group (one
// warp for rows shorter than 1024 values, else the whole CTA) owns a row: one
// pass takes the amax with 16-byte loads, a second pass re-reads the row (now
// in L1/L2), divides, and converts pairs with cvt.rn.satfinite.e4m3x2.f32.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

constexpr int kQThreads = 256;

// Smallest power of two not below a positive finite fp32 r (exact, bit level).
__device__ __forceinline__ float pow2_ceil(float r)
{
    const uint32_t u = __float_as_uint(r);
    const uint32_t ex = u & 0x7F800000u, man = u & 0x007FFFFFu;
    if (ex != 0u) // normal: r itself when the mantissa is zero, else the next exponent
        return man == 0u ? r : __uint_as_float(ex + 0x00800000u);
    // subnormal r = man * 2^-149: the next power of two of man, in the same units
    const uint32_t p = (man & (man - 1u)) == 0u ? man : (1u << (32 - __clz(man - 1u)));
    return __uint_as_float(p);
}

// Two fp32 -> two E4M3 codes (round to nearest even, saturating), lo in byte 0.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int GROUP>
__global__ void __launch_bounds__(kQThreads)
    quantize_kernel(const float *__restrict__ x, int64_t rows, int64_t cols, int mode, uint8_t *__restrict__ codes,
                    float *__restrict__ scale)
{
    constexpr int kRowsPerCta = kQThreads / GROUP;
    __shared__ float red[kQThreads / 32];
    grid_dep_wait();
    grid_dep_launch();
    const int g = threadIdx.x % GROUP;
    const int64_t stride = (int64_t)gridDim.x * kRowsPerCta;
    // GROUP == kQThreads: the whole CTA walks the same rows, so the loop and the
    // barriers inside it are uniform.
    for (int64_t row = (int64_t)blockIdx.x * kRowsPerCta + threadIdx.x / GROUP; row < rows; row += stride) {
        const float *xr = x + row * cols;
        uint8_t *cr = codes + row * cols;
        const bool vec = ((reinterpret_cast<uintptr_t>(xr) & 15u) == 0) && ((reinterpret_cast<uintptr_t>(cr) & 3u) == 0);
        const int64_t n4 = vec ? cols / 4 : 0;
        float m = 0.f;
        for (int64_t i = g; i < n4; i += GROUP) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(xr) + i);
            m = fmaxf(fmaxf(fmaxf(m, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
        }
        for (int64_t i = 4 * n4 + g; i < cols; i += GROUP)
            m = fmaxf(m, fabsf(__ldg(xr + i)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (GROUP > 32) {
            if ((threadIdx.x & 31) == 0)
                red[threadIdx.x >> 5] = m;
            __syncthreads();
            m = red[0];
#pragma unroll
            for (int w = 1; w < GROUP / 32; ++w)
                m = fmaxf(m, red[w]);
            __syncthreads(); // red is reused by the next row
        }
        float s = 1.f;
        if (m > 0.f) {
            const float ratio = m / 448.f;
            s = mode == 0 ? ratio : pow2_ceil(ratio);
        }
        if (g == 0)
            scale[row] = s;
        for (int64_t i = g; i < n4; i += GROUP) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(xr) + i);
            const uint32_t lo = e4m3x2(v.x / s, v.y / s), hi = e4m3x2(v.z / s, v.w / s);
            reinterpret_cast<uint32_t *>(cr)[i] = lo | (hi << 16);
        }
        for (int64_t i = 4 * n4 + g; i < cols; i += GROUP)
            cr[i] = static_cast<uint8_t>(e4m3x2(__ldg(xr + i) / s, 0.f) & 0xFFu);
    }
}

} // namespace

int launch_quantize(const QuantizeArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    if (a.rows == 0)
        return DSA_OK;
    const int sms = num_sms();
    cudaError_t e;
    if (a.cols < 1024) {
        constexpr int kRows = kQThreads / 32;
        int64_t grid = (a.rows + kRows - 1) / kRows;
        if (grid > 64LL * sms)
            grid = 64LL * sms;
        e = launch_pdl(quantize_kernel<32>, dim3((unsigned)grid), dim3(kQThreads), 0, stream, 1, a.x, a.rows, a.cols,
                       a.mode, a.codes, a.scale);
    } else {
        int64_t grid = a.rows;
        if (grid > 64LL * sms)
            grid = 64LL * sms;
        e = launch_pdl(quantize_kernel<kQThreads>, dim3((unsigned)grid), dim3(kQThreads), 0, stream, 1, a.x, a.rows,
                       a.cols, a.mode, a.codes, a.scale);
    }
    if (e != cudaSuccess) {
        snprintf(err, errlen, "quantize launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

} // namespace dsa
