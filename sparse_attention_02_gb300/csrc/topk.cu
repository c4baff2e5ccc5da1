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
// so the output comes out sorted without a sort.
//
// Fast path (every row it can take; the passes above are its fallback).  Four
// passes over a long row cost more than they need to: (1) rows longer than
// kCand draw kSamples keys at a fixed stride, and a radix select over those
// samples gives the key at sample rank ~ (1.5 k + 512) / n from the top, the
// threshold (shorter rows use none); (2) one streaming pass keeps every key at
// or above it: warp w scans its own contiguous segment of the row and appends
// (key, index) to its own region of shared memory with warp-level prefix
// counts, so the regions taken in warp order list the candidates in index
// order; (3) the exact radix select runs on those few thousand candidates;
// (4) one block-wide prefix count over the ordered candidates writes the kept
// indices in ascending order, as the compaction above does.  A row whose
// candidates miss [k, capacity] (tie-heavy or adversarial rows) takes the four
// passes instead; either way the output is the same.  The fast path runs only
// when the grid is at most one resident wave (decode batches): with many rows
// in flight the four-pass kernel, whose footprint is 16 KB of shared memory
// rather than 80 KB, keeps more rows per SM and finishes the batch sooner.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSeg = 512;               // candidates one warp's segment may keep
constexpr int kCand = kWarps * kSeg;    // 8192
constexpr int kSamples = 4 * kThreads;  // 2048 threshold samples
constexpr int kSmemTopk = (2 * kCand + 4096) * 4; // candidate keys, indices, histogram

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

// Fast path for one row with k < n; returns false (writing nothing) when the
// row must take the four passes.  wc: kWarps + 1 ints of shared memory.
template <bool kVec>
__device__ bool topk_row_fast(const float *row, int n, int k, int32_t *out, uint32_t *ckey, int32_t *cidx,
                              int *hist, int *scratch, int *sel, int *wc)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1. threshold: the r-th largest of kSamples keys drawn at a fixed stride
    uint32_t thr = 0u;
    if (n > kCand) {
        uint32_t sk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sk[e] = order_key(__ldg(row + (int64_t)(threadIdx.x + e * kThreads) * n / kSamples));
        int r = (int)((int64_t)(3 * k / 2 + 512) * kSamples / n);
        r = r < 1 ? 1 : (r > kSamples ? kSamples : r);
        for (int b = threadIdx.x; b < 4096; b += kThreads)
            hist[b] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e)
            atomicAdd(&hist[sk[e] >> 20], 1);
        __syncthreads();
        select_bin(hist, 4096, r, scratch, sel);
        const uint32_t d0 = sel[0];
        r -= sel[1];
        __syncthreads();
        for (int b = threadIdx.x; b < 4096; b += kThreads)
            hist[b] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((sk[e] >> 20) == d0)
                atomicAdd(&hist[(sk[e] >> 8) & 0xFFFu], 1);
        __syncthreads();
        select_bin(hist, 4096, r, scratch, sel);
        const uint32_t p1 = (d0 << 12) | static_cast<uint32_t>(sel[0]);
        r -= sel[1];
        __syncthreads();
        for (int b = threadIdx.x; b < 256; b += kThreads)
            hist[b] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((sk[e] >> 8) == p1)
                atomicAdd(&hist[sk[e] & 0xFFu], 1);
        __syncthreads();
        select_bin(hist, 256, r, scratch, sel);
        thr = (p1 << 8) | static_cast<uint32_t>(sel[0]);
        __syncthreads();
    }
    // 2. warp w keeps the keys >= thr of its segment [s0, s1), in order
    const int seg = (((n + kWarps - 1) / kWarps) + 3) & ~3;
    const int s0 = warp * seg;
    const int s1 = s0 + seg < n ? s0 + seg : n;
    uint32_t *wk = ckey + warp * kSeg;
    int32_t *wi = cidx + warp * kSeg;
    int cnt = 0; // warp-uniform
    if (kVec) {
        for (int base = s0; base < s1; base += 128) {
            const int i = base + 4 * lane;
            uint32_t kk[4];
            bool f[4];
            if (i + 3 < s1) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(row + i));
                kk[0] = order_key(v.x);
                kk[1] = order_key(v.y);
                kk[2] = order_key(v.z);
                kk[3] = order_key(v.w);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    f[e] = kk[e] >= thr;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kk[e] = i + e < s1 ? order_key(__ldg(row + i + e)) : 0u;
                    f[e] = i + e < s1 && kk[e] >= thr;
                }
            }
            const int c = (int)f[0] + (int)f[1] + (int)f[2] + (int)f[3];
            int x = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o)
                    x += y;
            }
            int slot = cnt + x - c;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (f[e]) {
                    if (slot < kSeg) {
                        wk[slot] = kk[e];
                        wi[slot] = i + e;
                    }
                    ++slot;
                }
            }
            cnt += __shfl_sync(0xffffffffu, x, 31);
        }
    } else {
        for (int base = s0; base < s1; base += 32) {
            const int i = base + lane;
            const uint32_t key = i < s1 ? order_key(__ldg(row + i)) : 0u;
            const bool f = i < s1 && key >= thr;
            const unsigned m = __ballot_sync(0xffffffffu, f);
            const int slot = cnt + __popc(m & ((1u << lane) - 1u));
            if (f && slot < kSeg) {
                wk[slot] = key;
                wi[slot] = i;
            }
            cnt += __popc(m);
        }
    }
    if (lane == 0)
        wc[warp] = cnt;
    __syncthreads();
    // candidate count, overflow, and the exclusive prefix of the regions (in place)
    if (threadIdx.x == 0) {
        int tot = 0, over = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int c = wc[w];
            over |= c > kSeg;
            wc[w] = tot;
            tot += c;
        }
        wc[kWarps] = over ? -1 : tot;
    }
    __syncthreads();
    const int nc = wc[kWarps];
    if (nc < k) // overflow (-1) or too few
        return false;
    // flat candidate f lives in region w (wc[w] <= f < wc[w + 1]) at offset f - wc[w]
    auto at = [&](int f) -> int {
        int w = 0;
#pragma unroll
        for (int q = 1; q < kWarps; ++q)
            w = wc[q] <= f ? q : w;
        return w * kSeg + (f - wc[w]);
    };
    // 3. exact radix select among the candidates on (key - kmin): the range of
    //    candidate keys spans at most 4096 bins per pass, so close scores spread
    //    out instead of piling into a few bins of the raw top digit
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int f = threadIdx.x; f < nc; f += kThreads) {
        const uint32_t key = ckey[at(f)];
        lo = key < lo ? key : lo;
        hi = key > hi ? key : hi;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint32_t l2 = __shfl_xor_sync(0xffffffffu, lo, o), h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        lo = l2 < lo ? l2 : lo;
        hi = h2 > hi ? h2 : hi;
    }
    if (lane == 0) {
        hist[2 * warp] = static_cast<int>(lo);
        hist[2 * warp + 1] = static_cast<int>(hi);
    }
    __syncthreads();
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t l2 = static_cast<uint32_t>(hist[2 * w]), h2 = static_cast<uint32_t>(hist[2 * w + 1]);
        kmin = l2 < kmin ? l2 : kmin;
        kmax = h2 > kmax ? h2 : kmax;
    }
    __syncthreads();
    const uint32_t range = kmax - kmin;
    const int bits = range == 0u ? 0 : 32 - __clz(range); // d = key - kmin has `bits` significant bits
    int shift = bits > 12 ? bits - 12 : 0;  // this pass sorts d into bins of d >> shift ...
    int nbins = 1 << (bits - shift);        // ... of which there are nbins (at most 4096)
    int prev = 32;                          // bits of d at and above `prev` are fixed to `prefix`
    uint32_t prefix = 0u;
    int k_rem = k;
    for (;;) {
        for (int q = threadIdx.x; q < nbins; q += kThreads)
            hist[q] = 0;
        __syncthreads();
        for (int f = threadIdx.x; f < nc; f += kThreads) {
            const uint32_t d = ckey[at(f)] - kmin;
            if (prev == 32 || (d >> prev) == prefix)
                atomicAdd(&hist[(d >> shift) & static_cast<uint32_t>(nbins - 1)], 1);
        }
        __syncthreads();
        select_bin(hist, nbins, k_rem, scratch, sel);
        const uint32_t bsel = static_cast<uint32_t>(sel[0]);
        k_rem -= sel[1];
        __syncthreads();
        prefix = prev == 32 ? bsel : ((prefix << (prev - shift)) | bsel); // = d >> shift of the chosen keys
        if (shift == 0)
            break;
        prev = shift;
        shift = shift > 12 ? shift - 12 : 0;
        nbins = 1 << (prev - shift);
    }
    const uint32_t tau = kmin + prefix; // every bit of d fixed: the k-th largest candidate key
    const int need_eq = k_rem;          // keys equal to tau to keep (the smallest indices)
    __syncthreads();
    // 4. ordered output: thread t walks flat candidates [t*per, t*per + per)
    const int per = (nc + kThreads - 1) / kThreads;
    const int f0 = threadIdx.x * per;
    const int f1 = f0 + per < nc ? f0 + per : nc;
    int gt = 0, eq = 0;
    for (int f = f0; f < f1; ++f) {
        const uint32_t key = ckey[at(f)];
        gt += key > tau;
        eq += key == tau;
    }
    int total;
    const int pre = block_exclusive_scan((gt << 16) | eq, scratch, &total);
    int g_before = pre >> 16, e_before = pre & 0xFFFF;
    for (int f = f0; f < f1; ++f) {
        const int a = at(f);
        const uint32_t key = ckey[a];
        if (key > tau) {
            out[g_before + (e_before < need_eq ? e_before : need_eq)] = cidx[a];
            ++g_before;
        } else if (key == tau) {
            if (e_before < need_eq)
                out[g_before + e_before] = cidx[a];
            ++e_before;
        }
    }
    return true;
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

__global__ void __launch_bounds__(kThreads, 2)
    topk_fast_kernel(const float *__restrict__ logits, int64_t ld, int T, const int32_t *__restrict__ valid_len, int k,
                int32_t *__restrict__ idx, unsigned *status)
{
    extern __shared__ __align__(16) uint32_t dsm[];
    uint32_t *ckey = dsm;
    int32_t *cidx = reinterpret_cast<int32_t *>(dsm + kCand);
    int *hist = reinterpret_cast<int *>(dsm + 2 * kCand);
    __shared__ int scratch[kWarps + 1];
    __shared__ int sel[2];
    __shared__ int wc[kWarps + 1];
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
        const bool vec = (reinterpret_cast<uintptr_t>(r) & 15u) == 0;
        const bool done = vec ? topk_row_fast<true>(r, n, k, out, ckey, cidx, hist, scratch, sel, wc)
                              : topk_row_fast<false>(r, n, k, out, ckey, cidx, hist, scratch, sel, wc);
        __syncthreads();
        if (!done) {
            if (vec)
                topk_row<true>(r, n, k, out, hist, scratch, sel);
            else
                topk_row<false>(r, n, k, out, hist, scratch, sel);
        }
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
    // Few rows (decode, one resident wave at most): each row's latency is the
    // cost, so the candidate fast path takes them.  Many rows (prefill): the
    // four-pass kernel's small footprint keeps more rows in flight per SM and
    // wins on throughput.
    if (a.T <= 2 * num_sms()) {
        static bool attr_set[64] = {};
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 64 && !attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(topk_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kSmemTopk);
            if (e != cudaSuccess) {
                snprintf(err, errlen, "cudaFuncSetAttribute(topk): %s", cudaGetErrorString(e));
                return DSA_ERR_CUDA;
            }
            attr_set[dev] = true;
        }
        topk_fast_kernel<<<a.T, kThreads, kSmemTopk, stream>>>(a.logits, a.ld, a.T, a.valid_len, a.k, a.idx,
                                                                status);
    } else {
        const int grid = a.T < 65535 * 4 ? a.T : 65535 * 4;
        topk_kernel<<<grid, kThreads, 0, stream>>>(a.logits, a.ld, a.T, a.valid_len, a.k, a.idx, status);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, errlen, "topk launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

} // namespace dsa
