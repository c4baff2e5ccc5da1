// Top-k token selection on sm_103a: radix select over fp32 logits.
//
// Defines ("AMD Instinct MI355X GPUs Power DeepSeek-V3.2-Exp", section "DeepSeek
// Sparse Attention (DSA)", item 2, fine-grained top-2048 selection): for each
// query row, the k candidates with the highest index score, ranked by (score
// descending, index ascending), written in ascending index order and padded
// with -1 when the row has fewer than k candidates.
//
// Method.  Each fp32 score maps to a 32-bit key whose unsigned order is the
// float order (-0 is first mapped to +0, so the two tie).  Three histogram
// passes over the row fix the key of the k-th largest candidate, tau, one
// digit at a time (12 + 12 + 8 bits).  A last pass walks the row in index
// order and keeps every key > tau plus the first (k - #greater) keys == tau;
// a block-wide prefix count gives each kept index its output slot directly,
// so the output comes out sorted without a sort.  One CTA owns one row; the
// first pass reads the row from HBM, the later ones mostly hit L2.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t order_key(float x)
{
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u)
        u = 0u; // -0 ties with +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the block in thread order; returns the prefix and
// writes the block total to *total.  `scratch` holds kWarps + 1 ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int *scratch, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        if (lane < kWarps)
            scratch[lane] = w; // inclusive over warps
        if (lane == kWarps - 1)
            scratch[kWarps] = w;
    }
    __syncthreads();
    const int prefix = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
    *total = scratch[kWarps];
    __syncthreads(); // scratch reusable afterwards
    return prefix;
}

template <bool kVec, typename F>
__device__ __forceinline__ void for_each_key(const float *row, int n, F &&f)
{
    if (kVec) {
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        const int n4 = n >> 2;
        for (int i = threadIdx.x; i < n4; i += kThreads) {
            const float4 v = __ldg(r4 + i);
            f(4 * i + 0, order_key(v.x));
            f(4 * i + 1, order_key(v.y));
            f(4 * i + 2, order_key(v.z));
            f(4 * i + 3, order_key(v.w));
        }
        for (int i = 4 * n4 + threadIdx.x; i < n; i += kThreads)
            f(i, order_key(__ldg(row + i)));
    } else {
        for (int i = threadIdx.x; i < n; i += kThreads)
            f(i, order_key(__ldg(row + i)));
    }
}

// Given a histogram of `nbins` bins, finds the bin b holding the k_rem-th
// largest element: count(bins > b) < k_rem <= count(bins >= b).  Writes b and
// count(bins > b) to out[0], out[1].
__device__ __forceinline__ void select_bin(const int *hist, int nbins, int k_rem, int *scratch, int *out)
{
    const int per = nbins / kThreads > 0 ? nbins / kThreads : 1;
    const int hi = nbins - threadIdx.x * per; // this thread owns bins [hi - per, hi), highest first
    int sum = 0;
    if (hi > 0)
        for (int b = hi - 1; b >= hi - per && b >= 0; --b)
            sum += hist[b];
    int total;
    int above = block_exclusive_scan(sum, scratch, &total);
    if (hi > 0) {
        for (int b = hi - 1; b >= hi - per && b >= 0; --b) {
            const int c = hist[b];
            if (above < k_rem && above + c >= k_rem) {
                out[0] = b;
                out[1] = above;
            }
            above += c;
        }
    }
    __syncthreads();
}

template <bool kVec>
__device__ void topk_row(const float *row, int n, int k, int32_t *out, int *hist, int *scratch, int *sel)
{
    // pass 1: top 12 bits
    for (int b = threadIdx.x; b < 4096; b += kThreads)
        hist[b] = 0;
    __syncthreads();
    for_each_key<kVec>(row, n, [&](int, uint32_t key) { atomicAdd(&hist[key >> 20], 1); });
    __syncthreads();
    select_bin(hist, 4096, k, scratch, sel);
    const uint32_t d0 = sel[0];
    int k_rem = k - sel[1];
    __syncthreads();

    // pass 2: next 12 bits among keys with the chosen top digit
    for (int b = threadIdx.x; b < 4096; b += kThreads)
        hist[b] = 0;
    __syncthreads();
    for_each_key<kVec>(row, n, [&](int, uint32_t key) {
        if ((key >> 20) == d0)
            atomicAdd(&hist[(key >> 8) & 0xFFFu], 1);
    });
    __syncthreads();
    select_bin(hist, 4096, k_rem, scratch, sel);
    const uint32_t p1 = (d0 << 12) | static_cast<uint32_t>(sel[0]);
    k_rem -= sel[1];
    __syncthreads();

    // pass 3: last 8 bits
    for (int b = threadIdx.x; b < 256; b += kThreads)
        hist[b] = 0;
    __syncthreads();
    for_each_key<kVec>(row, n, [&](int, uint32_t key) {
        if ((key >> 8) == p1)
            atomicAdd(&hist[key & 0xFFu], 1);
    });
    __syncthreads();
    select_bin(hist, 256, k_rem, scratch, sel);
    const uint32_t tau = (p1 << 8) | static_cast<uint32_t>(sel[0]);
    k_rem -= sel[1];
    // k_rem = how many keys equal to tau are kept (the first ones in index order)
    const int need_eq = k_rem;
    __syncthreads();

    // pass 4: ordered compaction.  Thread i handles elements [4i, 4i+4) of
    // each 4*kThreads chunk; gt/eq counts are packed (gt << 16 | eq).
    int gt_base = 0, eq_base = 0;
    for (int c0 = 0; c0 < n; c0 += 4 * kThreads) {
        const int i0 = c0 + 4 * threadIdx.x;
        uint32_t keys[4];
        int valid = 0;
        if (kVec && i0 + 3 < n) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(row + i0));
            keys[0] = order_key(v.x);
            keys[1] = order_key(v.y);
            keys[2] = order_key(v.z);
            keys[3] = order_key(v.w);
            valid = 4;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (i0 + j < n) {
                    keys[j] = order_key(__ldg(row + i0 + j));
                    valid = j + 1;
                } else {
                    keys[j] = 0u;
                }
            }
        }
        int gt = 0, eq = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < valid) {
                gt += keys[j] > tau;
                eq += keys[j] == tau;
            }
        }
        int total;
        const int pre = block_exclusive_scan((gt << 16) | eq, scratch, &total);
        int g_before = gt_base + (pre >> 16);
        int e_before = eq_base + (pre & 0xFFFF);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < valid) {
                if (keys[j] > tau) {
                    const int slot = g_before + (e_before < need_eq ? e_before : need_eq);
                    if (slot < k)
                        out[slot] = i0 + j;
                    ++g_before;
                } else if (keys[j] == tau) {
                    if (e_before < need_eq && g_before + e_before < k)
                        out[g_before + e_before] = i0 + j;
                    ++e_before;
                }
            }
        }
        gt_base += total >> 16;
        eq_base += total & 0xFFFF;
        if (gt_base + (eq_base < need_eq ? eq_base : need_eq) >= k)
            break; // block-uniform: every kept index has been written
    }
}

__global__ void __launch_bounds__(kThreads, 2)
    topk_kernel(const float *__restrict__ logits, int64_t ld, int T, const int32_t *__restrict__ valid_len, int k,
                int32_t *__restrict__ idx, unsigned *status)
{
    __shared__ int hist[4096];
    __shared__ int scratch[kWarps + 1];
    __shared__ int sel[2];
    for (int row = blockIdx.x; row < T; row += gridDim.x) {
        int n = valid_len[row];
        if (n < 0)
            n = 0;
        if (n > ld) {
            if (threadIdx.x == 0)
                atomicOr(status, DSA_DEV_BAD_POSITION);
            n = static_cast<int>(ld);
        }
        int32_t *out = idx + static_cast<int64_t>(row) * k;
        if (n <= k) {
            for (int j = threadIdx.x; j < k; j += kThreads)
                out[j] = j < n ? j : -1;
            continue;
        }
        const float *r = logits + static_cast<int64_t>(row) * ld;
        if ((reinterpret_cast<uintptr_t>(r) & 15u) == 0)
            topk_row<true>(r, n, k, out, hist, scratch, sel);
        else
            topk_row<false>(r, n, k, out, hist, scratch, sel);
        __syncthreads();
    }
}

} // namespace

int launch_topk(const TopkArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    unsigned *status = device_status_ptr();
    if (!status) {
        snprintf(err, errlen, "device status word unavailable");
        return DSA_ERR_CUDA;
    }
    const int grid = a.T < 65535 * 4 ? a.T : 65535 * 4;
    topk_kernel<<<grid, kThreads, 0, stream>>>(a.logits, a.ld, a.T, a.valid_len, a.k, a.idx, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, errlen, "topk launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

} // namespace dsa
