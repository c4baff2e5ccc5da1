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
// The four passes are the fallback of two candidate kernels, which read a row
// once or twice and select among a few thousand of its keys.
//
// Decode-sized batches (at most two rows per SM): each row runs on a cluster
// of cs CTAs (cs = 1, 2, 4 or 8, as many as the SMs allow): (1) rows longer
// than kGather draw kSamples keys at a fixed stride, and one 11-bit histogram
// over the samples' key range gives a threshold near sample rank
// (1.25 k + 256) / n from the top (row_threshold; every CTA of the cluster
// draws the same samples and gets the same value; shorter rows use none);
// (2) CTA c streams its own 1/cs of the row once, kUnroll 16-byte loads per
// lane in flight, and keeps every key at or above the threshold: warp w
// scans a contiguous segment and appends (score bits, index) to its own
// region of shared memory with ballot prefix counts, so the regions taken in
// warp order list the CTA's candidates in index order; (3) each CTA pushes its candidates,
// in order, into CTA 0's list through distributed shared memory; (4) CTA 0
// runs the exact radix select on those few thousand candidates and one
// block-wide prefix count over the ordered list writes the kept indices in
// ascending order, as the compaction above does.  A row whose candidates miss
// [k, kGather] (tie-heavy or adversarial rows) takes the four passes in CTA 0
// instead; either way the output is the same.  Prefill-sized batches use the
// one-CTA-per-row kernel described before topk_rows_kernel.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSeg = 512;               // candidates one warp's segment may keep
constexpr int kCand = kWarps * kSeg;    // 8192: a CTA's own candidates
constexpr int kGather = 8192;           // a cluster's candidates, gathered in CTA 0
constexpr int kSamples = 4 * kThreads;  // 2048 threshold samples
constexpr int kUnroll = 4;              // 16-byte loads per lane in flight in the filter (8: 1.4 % slower, 16: 46 %)
// candidate keys and indices (own, then gathered), histogram
constexpr int kSmemTopk = (2 * kCand + 2 * kGather + 4096) * 4;

__device__ __forceinline__ uint32_t order_key_bits(uint32_t u)
{
    if (u == 0x80000000u)
        u = 0u; // -0 ties with +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t order_key(float x) { return order_key_bits(__float_as_uint(x)); }

// The float whose key is `key` (order_key's inverse; -0 for the key between
// the negatives and +0).  For finite x, order_key(x) >= key  <=>  x >= key_float(key),
// so the filters below compare floats and form keys only for the keys they keep.
__device__ __forceinline__ float key_float(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Exclusive prefix sum over the block in thread order; returns the prefix and
// writes the block total to *total.  `scratch` holds kWarps + 1 ints.
template <int NT>
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
        int w = lane < (NT / 32) ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        if (lane < (NT / 32))
            scratch[lane] = w; // inclusive over warps
        if (lane == (NT / 32) - 1)
            scratch[(NT / 32)] = w;
    }
    __syncthreads();
    const int prefix = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
    *total = scratch[(NT / 32)];
    __syncthreads(); // scratch reusable afterwards
    return prefix;
}

template <int NT, bool kVec, typename F>
__device__ __forceinline__ void for_each_key(const float *row, int n, F &&f)
{
    if (kVec) {
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        const int n4 = n >> 2;
        for (int i = threadIdx.x; i < n4; i += NT) {
            const float4 v = __ldg(r4 + i);
            f(4 * i + 0, order_key(v.x));
            f(4 * i + 1, order_key(v.y));
            f(4 * i + 2, order_key(v.z));
            f(4 * i + 3, order_key(v.w));
        }
        for (int i = 4 * n4 + threadIdx.x; i < n; i += NT)
            f(i, order_key(__ldg(row + i)));
    } else {
        for (int i = threadIdx.x; i < n; i += NT)
            f(i, order_key(__ldg(row + i)));
    }
}

// Given a histogram of `nbins` bins (a power of two, 16-byte aligned), finds
// the bin b holding the k_rem-th largest element: count(bins > b) < k_rem <=
// count(bins >= b).  Writes b and count(bins > b) to out[0], out[1].  Thread t
// owns the contiguous bins [nbins - (t + 1) per, nbins - t per), read with
// 16-byte loads when per >= 4 so the warp's reads do not collide on banks.
template <int NT>
__device__ __forceinline__ void select_bin(const int *hist, int nbins, int k_rem, int *scratch, int *out)
{
    constexpr int kMaxPer = 4096 / NT; // histograms hold at most 4096 bins
    const int per = nbins / NT > 0 ? nbins / NT : 1;
    const int hi = nbins - threadIdx.x * per; // this thread owns bins [hi - per, hi), highest first
    int c[kMaxPer];                           // c[j]: count of bin hi - 1 - j
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j)
        c[j] = 0;
    if (hi > 0) {
        if (per >= 4) {
#pragma unroll
            for (int q = 0; q < kMaxPer / 4; ++q) {
                if (4 * q < per) {
                    const int4 b = *reinterpret_cast<const int4 *>(hist + hi - 4 * (q + 1));
                    c[4 * q] = b.w;
                    c[4 * q + 1] = b.z;
                    c[4 * q + 2] = b.y;
                    c[4 * q + 3] = b.x;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
                if (j < per)
                    c[j] = hist[hi - 1 - j];
        }
    }
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j)
        sum += c[j];
    int total;
    int above = block_exclusive_scan<NT>(sum, scratch, &total);
    if (hi > 0) {
#pragma unroll
        for (int j = 0; j < kMaxPer; ++j) {
            if (j < per) {
                if (above < k_rem && above + c[j] >= k_rem) {
                    out[0] = hi - 1 - j;
                    out[1] = above;
                }
                above += c[j];
            }
        }
    }
    __syncthreads();
}

// The key of the k-th largest of row[0, n) (1 <= k <= n), digit by digit in
// three histogram passes (12 + 12 + 8 bits); *k_eq receives how many keys
// equal to it are among the k largest (the rest of them rank below).
template <int NT, bool kVec>
__device__ uint32_t kth_key(const float *row, int n, int k, int *hist, int *scratch, int *sel, int *k_eq)
{
    // pass 1: top 12 bits
    for (int b = threadIdx.x; b < 4096; b += NT)
        hist[b] = 0;
    __syncthreads();
    for_each_key<NT, kVec>(row, n, [&](int, uint32_t key) { atomicAdd(&hist[key >> 20], 1); });
    __syncthreads();
    select_bin<NT>(hist, 4096, k, scratch, sel);
    const uint32_t d0 = sel[0];
    int k_rem = k - sel[1];
    __syncthreads();

    // pass 2: next 12 bits among keys with the chosen top digit
    for (int b = threadIdx.x; b < 4096; b += NT)
        hist[b] = 0;
    __syncthreads();
    for_each_key<NT, kVec>(row, n, [&](int, uint32_t key) {
        if ((key >> 20) == d0)
            atomicAdd(&hist[(key >> 8) & 0xFFFu], 1);
    });
    __syncthreads();
    select_bin<NT>(hist, 4096, k_rem, scratch, sel);
    const uint32_t p1 = (d0 << 12) | static_cast<uint32_t>(sel[0]);
    k_rem -= sel[1];
    __syncthreads();

    // pass 3: last 8 bits
    for (int b = threadIdx.x; b < 256; b += NT)
        hist[b] = 0;
    __syncthreads();
    for_each_key<NT, kVec>(row, n, [&](int, uint32_t key) {
        if ((key >> 8) == p1)
            atomicAdd(&hist[key & 0xFFu], 1);
    });
    __syncthreads();
    select_bin<NT>(hist, 256, k_rem, scratch, sel);
    const uint32_t tau = (p1 << 8) | static_cast<uint32_t>(sel[0]);
    k_rem -= sel[1];
    *k_eq = k_rem;
    __syncthreads();
    return tau;
}

template <int NT, bool kVec>
__device__ void topk_row(const float *row, int n, int k, int32_t *out, int *hist, int *scratch, int *sel)
{
    // k_rem = how many keys equal to tau are kept (the first ones in index order)
    int need_eq;
    const uint32_t tau = kth_key<NT, kVec>(row, n, k, hist, scratch, sel, &need_eq);

    // pass 4: ordered compaction.  Thread i handles elements [4i, 4i+4) of
    // each 4*NT chunk; gt/eq counts are packed (gt << 16 | eq).
    int gt_base = 0, eq_base = 0;
    for (int c0 = 0; c0 < n; c0 += 4 * NT) {
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
        const int pre = block_exclusive_scan<NT>((gt << 16) | eq, scratch, &total);
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
// Keeps the keys >= thr (kAll: every key) of row[c0, c1) in index order,
// comparing floats (key_float) and forming keys only for the kept ones.  The
// first `head` keys (row + c0 + head is 16-byte aligned) go through warp 0 one per lane;
// then warp w scans its own contiguous segment of the rest, kUnroll 16-byte
// loads per lane in flight.  Keys are appended as (score bits, index) to the warp's
// region ck/ci[w * kSeg, +kSeg) with ballot prefix counts.  Leaves in wc[w]
// the offset of warp w's region in the CTA's flat candidate list and in
// wc[kWarps] the CTA's count, or -1 if a region overflowed.
template <int NT, bool kAll>
__device__ void filter_segment(const float *row, int c0, int c1, int head, uint32_t thr, uint32_t *ck, int32_t *ci,
                               int *wc)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    const int v0 = c0 + head;
    const int seg = (((c1 - v0 + (NT / 32) - 1) / (NT / 32)) + 3) & ~3;
    const int s0 = v0 + warp * seg < c1 ? v0 + warp * seg : c1;
    const int s1 = s0 + seg < c1 ? s0 + seg : c1;
    uint32_t *wk = ck + warp * kSeg;
    int32_t *wi = ci + warp * kSeg;
    const float thr_f = key_float(thr);
    int cnt = 0; // warp-uniform
    if (warp == 0 && head > 0) {
        const int i = c0 + lane;
        const float x = lane < head ? __ldg(row + i) : 0.f;
        const bool f = lane < head && (kAll || x >= thr_f);
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (f) {
            wk[__popc(m & lt)] = __float_as_uint(x);
            wi[__popc(m & lt)] = i;
        }
        cnt = __popc(m);
    }
    for (int base = s0; base < s1; base += 128 * kUnroll) {
        float xx[kUnroll][4];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + 128 * u + 4 * lane;
            if (i + 3 < s1) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(row + i));
                xx[u][0] = v.x;
                xx[u][1] = v.y;
                xx[u][2] = v.z;
                xx[u][3] = v.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    xx[u][e] = i + e < s1 ? __ldg(row + i + e) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + 128 * u + 4 * lane;
            bool f[4];
            int pre = 0, tot = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[e] = i + e < s1 && (kAll || xx[u][e] >= thr_f);
                const unsigned m = __ballot_sync(0xffffffffu, f[e]);
                pre += __popc(m & lt);
                tot += __popc(m);
            }
            int slot = cnt + pre; // keys of lower lanes come first, then this lane's in order
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (f[e]) {
                    if (slot < kSeg) {
                        wk[slot] = __float_as_uint(xx[u][e]);
                        wi[slot] = i + e;
                    }
                    ++slot;
                }
            }
            cnt += tot;
        }
    }
    if (lane == 0)
        wc[warp] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
        int tot = 0, over = 0;
        for (int w = 0; w < (NT / 32); ++w) {
            const int c = wc[w];
            over |= c > kSeg;
            wc[w] = tot;
            tot += c;
        }
        wc[(NT / 32)] = over ? -1 : tot;
    }
    __syncthreads();
}

// Slot of flat candidate f: region w (wc[w] <= f < wc[w + 1]) at offset f - wc[w].
__device__ __forceinline__ int cand_slot(const int *wc, int f)
{
    int w = 0;
#pragma unroll
    for (int q = 1; q < kWarps; ++q)
        w = wc[q] <= f ? q : w;
    return w * kSeg + (f - wc[w]);
}

// Key tau of the k-th largest of nc >= k candidates ck (raw fp32 score bits;
// the keys are formed as they are read), in any order; *need_eq receives how
// many candidates equal to tau are among the k largest.
template <int NT>
__device__ uint32_t select_tau(const uint32_t *ck, int nc, int k, int *hist, int *sel, int *need_eq)
{
    constexpr int NW = NT / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // hist: two 1024-bin histograms that alternate between passes (the next one
    // is cleared while warp 0 picks the bin in the current one), then NW ints
    // left to the caller and the per-warp minima and maxima.
    int *mm = hist + 2048 + NW;
    for (int q = threadIdx.x; q < 1024; q += NT)
        hist[q] = 0;
    // Radix select on d = key - kmin: the candidates span a narrow key range,
    // so passes of at most 10 bits over d spread close scores over the bins
    // instead of piling them into a few bins of the raw top digit.
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int f = threadIdx.x; f < nc; f += NT) {
        const uint32_t key = order_key_bits(ck[f]);
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
        mm[2 * warp] = static_cast<int>(lo);
        mm[2 * warp + 1] = static_cast<int>(hi);
    }
    __syncthreads();
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t l2 = static_cast<uint32_t>(mm[2 * w]), h2 = static_cast<uint32_t>(mm[2 * w + 1]);
        kmin = l2 < kmin ? l2 : kmin;
        kmax = h2 > kmax ? h2 : kmax;
    }
    const uint32_t range = kmax - kmin;
    const int bits = range == 0u ? 0 : 32 - __clz(range); // d has `bits` significant bits
    int shift = bits > 10 ? bits - 10 : 0;  // this pass sorts d into bins of d >> shift ...
    int nbins = 1 << (bits - shift);        // ... of which there are nbins (at most 1024)
    int prev = 32;                          // bits of d at and above `prev` are fixed to `prefix`
    uint32_t prefix = 0u;
    int k_rem = k;
    for (int pass = 0;; ++pass) {
        int *cur = hist + 1024 * (pass & 1);
        int *nxt = hist + 1024 * ((pass & 1) ^ 1);
        for (int f = threadIdx.x; f < nc; f += NT) {
            const uint32_t d = order_key_bits(ck[f]) - kmin;
            if (prev == 32 || (d >> prev) == prefix)
                atomicAdd(&cur[(d >> shift) & static_cast<uint32_t>(nbins - 1)], 1);
        }
        __syncthreads();
        if (warp == 0) {
            // the bin with (keys above it) < k_rem <= (keys at or above it); lane l
            // reads bins 32 l .. 32 l + 31 (bins past nbins are empty)
            const int4 *b4 = reinterpret_cast<const int4 *>(cur + 32 * lane);
            int sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int4 v = b4[q];
                sum += v.x + v.y + v.z + v.w;
            }
            int incl = sum; // keys in the bins of this lane and of the lanes above it
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32)
                    incl += y;
            }
            const int excl = incl - sum;
            const unsigned m = __ballot_sync(0xffffffffu, excl < k_rem && incl >= k_rem);
            // within the chosen lane's 32 bins, highest first: lane i takes bin
            // 32 L + 31 - i, a prefix count over the lanes finds the bin
            const int L = m ? __ffs(m) - 1 : 0;
            const int above_L = __shfl_sync(0xffffffffu, excl, L);
            const int c = cur[32 * L + 31 - lane];
            int pre = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, pre, o);
                if (lane >= o)
                    pre += y;
            }
            const unsigned m2 = __ballot_sync(0xffffffffu, above_L + pre >= k_rem);
            if (m2 && lane == __ffs(m2) - 1) {
                sel[0] = 32 * L + 31 - lane;
                sel[1] = above_L + pre - c;
            }
        } else {
            for (int q = threadIdx.x - 32; q < 1024; q += NT - 32)
                nxt[q] = 0;
        }
        __syncthreads();
        const uint32_t bsel = static_cast<uint32_t>(sel[0]);
        k_rem -= sel[1];
        prefix = prev == 32 ? bsel : ((prefix << (prev - shift)) | bsel); // = d >> shift of the chosen keys
        if (shift == 0)
            break;
        prev = shift;
        shift = shift > 10 ? shift - 10 : 0;
        nbins = 1 << (prev - shift);
    }
    *need_eq = k_rem; // keys equal to tau to keep (the smallest indices)
    return kmin + prefix; // every bit of d fixed: the k-th largest candidate key
}

// Exact top-k of nc >= k candidates ck/ci listed in ascending index order (ck
// holds the raw fp32 score bits); writes the kept indices to out in that order.
template <int NT>
__device__ void select_candidates(const uint32_t *ck, const int32_t *ci, int nc, int k, int32_t *out, int *hist,
                                  int *sel)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *wsum = hist + 2048; // per-warp totals of the ordered output
    int need_eq;
    const uint32_t tau = select_tau<NT>(ck, nc, k, hist, sel, &need_eq);
    // ordered output: thread t walks candidates [t * per, t * per + per); one
    // prefix count over threads of (#greater << 16 | #equal) gives its slots
    const int per = (nc + NT - 1) / NT;
    const int f0 = threadIdx.x * per < nc ? threadIdx.x * per : nc;
    const int f1 = f0 + per < nc ? f0 + per : nc;
    int gt = 0, eq = 0;
    for (int f = f0; f < f1; ++f) {
        const uint32_t key = order_key_bits(ck[f]);
        gt += key > tau;
        eq += key == tau;
    }
    const int v = (gt << 16) | eq;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        wsum[warp] = x;
    __syncthreads();
    int pre = x - v;
    for (int w = 0; w < warp; ++w)
        pre += wsum[w];
    int g_before = pre >> 16, e_before = pre & 0xFFFF;
    for (int f = f0; f < f1; ++f) {
        const uint32_t key = order_key_bits(ck[f]);
        if (key > tau) {
            out[g_before + (e_before < need_eq ? e_before : need_eq)] = ci[f];
            ++g_before;
        } else if (key == tau) {
            if (e_before < need_eq)
                out[g_before + e_before] = ci[f];
            ++e_before;
        }
    }
}

// ---------------------------------------------------------------------------
// Prefill-sized batches: one 256-thread CTA per row, four rows in flight per
// SM (the phases below are short and end in barriers, so rows in flight, not
// bytes, set the rate); the row is read twice.
// (1) Rows longer than kRowCap draw kSamples keys at a fixed stride; one
//     11-bit histogram of (sample key - smallest sample key), scaled to the
//     samples' range, gives a threshold at or below the sample of rank
//     ~ (1.25 k + 256) / n from the top.  (2) A counting pass over the row
//     (warp w scans its own contiguous segment, ballot counts) and a block
//     scan place every warp's keys at or above the threshold; a second pass
//     (L1/L2 hits) writes (score bits, index) there, so the list is in index order.
//     (3) The exact radix select over those candidates and the ordered
//     compaction of select_candidates.  A row whose count misses [k, kRowCap]
//     takes the four passes instead; the result is the same.
constexpr int kRowThreads = 256;                       // four rows in flight per SM
constexpr int kRowCap = 4096;                          // candidates of one row
constexpr int kRowSmem = (2 * kRowCap + 4096) * 4;     // keys, indices, histogram

template <int NT>
__device__ uint32_t row_threshold(const float *row, int n, int k, int *hist, int *scratch, int *sel)
{
    constexpr int kPer = kSamples / NT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t sk[kPer];
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        sk[e] = order_key(__ldg(row + (int64_t)(threadIdx.x + e * NT) * n / kSamples));
        lo = sk[e] < lo ? sk[e] : lo;
        hi = sk[e] > hi ? sk[e] : hi;
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
    uint32_t smin = 0xFFFFFFFFu, smax = 0u;
    for (int w = 0; w < (NT / 32); ++w) {
        const uint32_t l2 = static_cast<uint32_t>(hist[2 * w]), h2 = static_cast<uint32_t>(hist[2 * w + 1]);
        smin = l2 < smin ? l2 : smin;
        smax = h2 > smax ? h2 : smax;
    }
    __syncthreads();
    const uint32_t range = smax - smin;
    const int bits = range == 0u ? 0 : 32 - __clz(range);
    const int shift = bits > 11 ? bits - 11 : 0;
    for (int b = threadIdx.x; b < 2048; b += NT)
        hist[b] = 0;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kPer; ++e)
        atomicAdd(&hist[(sk[e] - smin) >> shift], 1);
    __syncthreads();
    int r = (int)((int64_t)(5 * k / 4 + 256) * kSamples / n);
    r = r < 1 ? 1 : (r > kSamples ? kSamples : r);
    select_bin<NT>(hist, 2048, r, scratch, sel);
    const uint32_t thr = smin + (static_cast<uint32_t>(sel[0]) << shift);
    __syncthreads();
    return thr;
}

// One pass over warp w's segment of row[c0 + head, c1) (16-byte aligned from
// there; the `head` keys before it go to warp 0 first): counts the keys >= thr
// (kWrite = false), or writes them as (score bits, index) from slot base on (kWrite;
// kAll: every key, no compare).  Returns the warp's count (warp-uniform).
template <int NT, bool kWrite, bool kAll = false>
__device__ int row_pass(const float *row, int c0, int c1, int head, uint32_t thr, int base, uint32_t *ck,
                        int32_t *ci)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    const float thr_f = key_float(thr);
    const int v0 = c0 + head;
    const int seg = (((c1 - v0 + (NT / 32) - 1) / (NT / 32)) + 3) & ~3;
    const int s0 = v0 + warp * seg < c1 ? v0 + warp * seg : c1;
    const int s1 = s0 + seg < c1 ? s0 + seg : c1;
    int cnt = 0;  // kWrite: the warp's count so far; else this lane's
    if (warp == 0 && head > 0) {
        const int i = c0 + lane;
        const float x = lane < head ? __ldg(row + i) : 0.f;
        const bool f = lane < head && (kAll || x >= thr_f);
        if (kWrite) {
            const unsigned m = __ballot_sync(0xffffffffu, f);
            if (f) {
                ck[base + __popc(m & lt)] = __float_as_uint(x);
                ci[base + __popc(m & lt)] = i;
            }
            cnt = __popc(m);
        } else {
            cnt = f ? 1 : 0;
        }
    }
    for (int b0 = s0; b0 < s1; b0 += 128 * kUnroll) {
        float xx[kUnroll][4];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = b0 + 128 * u + 4 * lane;
            if (i + 3 < s1) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(row + i));
                xx[u][0] = v.x;
                xx[u][1] = v.y;
                xx[u][2] = v.z;
                xx[u][3] = v.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    xx[u][e] = i + e < s1 ? __ldg(row + i + e) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = b0 + 128 * u + 4 * lane;
            bool f[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                f[e] = i + e < s1 && (kAll || xx[u][e] >= thr_f);
            if (kWrite) {
                int pre = 0, tot = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const unsigned m = __ballot_sync(0xffffffffu, f[e]);
                    pre += __popc(m & lt);
                    tot += __popc(m);
                }
                int slot = base + cnt + pre;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (f[e]) {
                        ck[slot] = __float_as_uint(xx[u][e]);
                        ci[slot] = i + e;
                        ++slot;
                    }
                }
                cnt += tot;
            } else {
                cnt += (f[0] ? 1 : 0) + (f[1] ? 1 : 0) + (f[2] ? 1 : 0) + (f[3] ? 1 : 0);
            }
        }
    }
    if (!kWrite)
        cnt = __reduce_add_sync(0xffffffffu, cnt);
    return cnt;
}

// Candidate path for one row with k < n; false (nothing written) when the row
// must take the four passes.  wc: kWarps + 1 ints of shared memory.
template <int NT>
__device__ bool topk_row_candidates(const float *row, int n, int k, int32_t *out, uint32_t *ck, int32_t *ci,
                                    int *hist, int *scratch, int *sel, int *wc)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int h = static_cast<int>((4u - ((reinterpret_cast<uintptr_t>(row) >> 2) & 3u)) & 3u);
    h = h < n ? h : n;
    int nc, base;
    if (n <= kRowCap) {
        // every key is a candidate: warp w's slots start after the keys of the
        // segments before it (the segment split of row_pass), no counting pass
        const int seg = (((n - h + (NT / 32) - 1) / (NT / 32)) + 3) & ~3;
        const int s0 = h + warp * seg < n ? h + warp * seg : n;
        base = warp == 0 ? 0 : s0;
        nc = n;
        row_pass<NT, true, true>(row, 0, n, h, 0u, base, ck, ci);
    } else {
        const uint32_t thr = row_threshold<NT>(row, n, k, hist, scratch, sel);
        const int c = row_pass<NT, false>(row, 0, n, h, thr, 0, ck, ci);
        if (lane == 0)
            wc[warp] = c;
        __syncthreads();
        if (threadIdx.x == 0) {
            int tot = 0;
            for (int w = 0; w < (NT / 32); ++w) {
                const int x = wc[w];
                wc[w] = tot;
                tot += x;
            }
            wc[(NT / 32)] = tot;
        }
        __syncthreads();
        nc = wc[(NT / 32)];
        if (nc < k || nc > kRowCap)
            return false;
        row_pass<NT, true>(row, 0, n, h, thr, wc[warp], ck, ci);
    }
    __syncthreads();
    select_candidates<NT>(ck, ci, nc, k, out, hist, sel);
    return true;
}

__global__ void __launch_bounds__(kRowThreads, 4)
    topk_rows_kernel(const float *__restrict__ logits, int64_t ld, int T, const int32_t *__restrict__ valid_len, int k,
                     int32_t *__restrict__ idx, unsigned *status, const int32_t *__restrict__ row_flag)
{
    extern __shared__ __align__(16) uint32_t dsm[];
    uint32_t *ck = dsm;
    int32_t *ci = reinterpret_cast<int32_t *>(dsm + kRowCap);
    int *hist = reinterpret_cast<int *>(dsm + 2 * kRowCap);
    __shared__ int scratch[kRowThreads / 32 + 1];
    __shared__ int sel[2];
    __shared__ int wc[kRowThreads / 32 + 1];
    grid_dep_wait();
    grid_dep_launch();
    for (int row = blockIdx.x; row < T; row += gridDim.x) {
        if (row_flag && !row_flag[row])
            continue; // not one of the rows asked for (uniform)
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
            for (int j = threadIdx.x; j < k; j += kRowThreads)
                out[j] = j < n ? j : -1;
            continue;
        }
        const float *r = logits + static_cast<int64_t>(row) * ld;
        const bool done = topk_row_candidates<kRowThreads>(r, n, k, out, ck, ci, hist, scratch, sel, wc);
        __syncthreads();
        if (!done) {
            if ((reinterpret_cast<uintptr_t>(r) & 15u) == 0)
                topk_row<kRowThreads, true>(r, n, k, out, hist, scratch, sel);
            else
                topk_row<kRowThreads, false>(r, n, k, out, hist, scratch, sel);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Top-k from the candidate lists of the fused indexer (no logits in memory).
//
// Threshold.  Row t holds n = min(q_pos[t] + 1, S) keys.  A row with n <= cap
// keeps every key (threshold -inf).  Otherwise its m valid samples samp[t, 0, m)
// (scores of keys at a fixed stride over the keys) give thr[t] = the exact
// r-th largest sample, r = ceil((1.25 k + 256) m / n), found digit by digit
// (kth_key): about 1.25 k + 256 keys of the row score at or above it, so its k
// largest are among them unless the row is far from what its samples show
// (then its candidate count misses [k, cap] and the row is redone from full
// logits; the result is the same).  A single coarse histogram over the
// samples' whole key range is not enough here: near the threshold one of its
// bins can span a score interval holding a thousand keys of a 32K-key row.
__global__ void __launch_bounds__(kRowThreads)
    topk_threshold_kernel(const float *__restrict__ samp, int ld_s, int T, const int32_t *__restrict__ q_pos,
                          const int32_t *__restrict__ qpos_s, int S, int k, int cap, float *__restrict__ thr)
{
    __shared__ __align__(16) int hist[4096];
    __shared__ int scratch[kRowThreads / 32 + 1];
    __shared__ int sel[2];
    grid_dep_wait();
    grid_dep_launch();
    for (int row = blockIdx.x; row < T; row += gridDim.x) {
        int64_t n = static_cast<int64_t>(q_pos[row]) + 1;
        n = n < 0 ? 0 : (n > S ? S : n);
        int m = qpos_s[row] + 1;
        m = m < 0 ? 0 : (m > ld_s ? ld_s : m);
        if (n <= cap || m == 0) {
            if (threadIdx.x == 0)
                thr[row] = -INFINITY;
            continue;
        }
        int64_t r = (static_cast<int64_t>(5 * k / 4 + 256) * m + n - 1) / n;
        r = r < 1 ? 1 : (r > m ? m : r);
        const float *srow = samp + static_cast<int64_t>(row) * ld_s;
        int k_eq;
        const uint32_t tau = (reinterpret_cast<uintptr_t>(srow) & 15u) == 0
                                 ? kth_key<kRowThreads, true>(srow, m, static_cast<int>(r), hist, scratch, sel, &k_eq)
                                 : kth_key<kRowThreads, false>(srow, m, static_cast<int>(r), hist, scratch, sel, &k_eq);
        if (threadIdx.x == 0)
            thr[row] = key_float(tau);
        __syncthreads();
    }
}

// Select.  One CTA per row: a row with n <= k keeps keys 0 .. n-1; a row whose
// candidate count c is in [k, cap], with no region of its list overflowed (the
// list is kCandRegions regions of cap / 64 entries, one per indexer epilogue
// lane), loads its candidates (any order), finds the
// key tau of the k-th largest and how many keys equal to tau rank among the k
// (select_tau), marks the keys above tau and those equal to it in two bitmaps
// over the row's positions and walks the bitmaps in position order: every key
// > tau is kept, and of the keys == tau the first need_eq; a block-wide
// prefix count gives each kept position its output slot, so the output is in
// ascending order and the tie rule is (score desc, position asc).  A row whose
// count misses [k, cap] or overflowed a region is flagged (flag[t] = 1) for
// the full path and left untouched; every other row gets flag[t] = 0.
constexpr int kCandHistInts = 2048 + 3 * (kRowThreads / 32); // select_tau's scratch
constexpr int kCandRegions = 128;                            // regions of a row's candidate list
constexpr int kCandSmemMax = 232448 - 2048;                  // dynamic bytes, beside the kernel's static ones

__global__ void __launch_bounds__(kRowThreads)
    topk_candidates_kernel(const uint2 *__restrict__ cand, const int32_t *__restrict__ cand_cnt, int cap, int T,
                           const int32_t *__restrict__ q_pos, int S, int k, int32_t *__restrict__ idx,
                           int32_t *__restrict__ flag)
{
    extern __shared__ __align__(16) uint32_t dsm[];
    const int nw_max = (S + 31) / 32;
    uint32_t *ck = dsm;
    int32_t *ci = reinterpret_cast<int32_t *>(dsm + cap);
    int *hist = reinterpret_cast<int *>(dsm + 2 * cap);
    uint32_t *bgt = dsm + 2 * cap + kCandHistInts;
    uint32_t *beq = bgt + nw_max;
    __shared__ int scratch[kRowThreads / 32 + 1];
    __shared__ int sel[2];
    __shared__ int reg_off[kCandRegions];
    grid_dep_wait();
    grid_dep_launch();
    for (int row = blockIdx.x; row < T; row += gridDim.x) {
        int64_t n64 = static_cast<int64_t>(q_pos[row]) + 1;
        const int n = static_cast<int>(n64 < 0 ? 0 : (n64 > S ? S : n64));
        int32_t *out = idx + static_cast<int64_t>(row) * k;
        if (n <= k) {
            for (int j = threadIdx.x; j < k; j += kRowThreads)
                out[j] = j < n ? j : -1;
            if (threadIdx.x == 0)
                flag[row] = 0;
            continue;
        }
        // the row's list: kCandRegions regions of rcap entries, region q holding cq
        const int rcap = cap / 64;
        const int q = threadIdx.x;
        const int cq = q < kCandRegions ? __ldg(cand_cnt + static_cast<int64_t>(row) * kCandRegions + q) : 0;
        int c;
        const int off = block_exclusive_scan<kRowThreads>(cq, scratch, &c);
        if (__syncthreads_or(cq > rcap) || c < k || c > cap) {
            if (threadIdx.x == 0)
                flag[row] = 1;
            continue;
        }
        // entry f of the concatenated list lies in the last region whose offset is <= f
        // (binary search over the offsets): every load is independent of the others
        if (q < kCandRegions)
            reg_off[q] = off;
        __syncthreads();
        for (int f = threadIdx.x; f < c; f += kRowThreads) {
            int lo = 0, hi = kCandRegions - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (reg_off[mid] <= f)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            const uint2 v = __ldg(cand + (static_cast<int64_t>(row) * kCandRegions + lo) * rcap + (f - reg_off[lo]));
            ck[f] = v.x;
            ci[f] = static_cast<int32_t>(v.y);
        }
        const int nw = (n + 31) / 32;
        for (int w = threadIdx.x; w < nw; w += kRowThreads) {
            bgt[w] = 0u;
            beq[w] = 0u;
        }
        __syncthreads();
        int need_eq;
        const uint32_t tau = select_tau<kRowThreads>(ck, c, k, hist, sel, &need_eq);
        for (int f = threadIdx.x; f < c; f += kRowThreads) {
            const uint32_t key = order_key_bits(ck[f]);
            const int i = ci[f];
            if (key > tau)
                atomicOr(&bgt[i >> 5], 1u << (i & 31));
            else if (key == tau)
                atomicOr(&beq[i >> 5], 1u << (i & 31));
        }
        __syncthreads();
        const int per = (nw + kRowThreads - 1) / kRowThreads;
        const int w0 = threadIdx.x * per < nw ? threadIdx.x * per : nw;
        const int w1 = w0 + per < nw ? w0 + per : nw;
        int gt = 0, eq = 0;
        for (int w = w0; w < w1; ++w) {
            gt += __popc(bgt[w]);
            eq += __popc(beq[w]);
        }
        int total;
        const int pre = block_exclusive_scan<kRowThreads>((gt << 16) | eq, scratch, &total);
        int g_before = pre >> 16, e_before = pre & 0xFFFF;
        for (int w = w0; w < w1; ++w) {
            const uint32_t g = bgt[w];
            uint32_t m = g | beq[w];
            while (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1u;
                const int i = 32 * w + b;
                if ((g >> b) & 1u) {
                    out[g_before + (e_before < need_eq ? e_before : need_eq)] = i;
                    ++g_before;
                } else {
                    if (e_before < need_eq)
                        out[g_before + e_before] = i;
                    ++e_before;
                }
            }
        }
        if (threadIdx.x == 0)
            flag[row] = 0;
        __syncthreads();
    }
}

// Candidate path: one cluster of cs CTAs per row (cs from the launch).
__global__ void __launch_bounds__(kThreads, 1)
    topk_cluster_kernel(const float *__restrict__ logits, int64_t ld, int T, const int32_t *__restrict__ valid_len,
                        int k, int32_t *__restrict__ idx, unsigned *status)
{
    extern __shared__ __align__(16) uint32_t dsm[];
    uint32_t *lkey = dsm;
    int32_t *lidx = reinterpret_cast<int32_t *>(dsm + kCand);
    uint32_t *gkey = dsm + 2 * kCand;
    int32_t *gidx = reinterpret_cast<int32_t *>(dsm + 2 * kCand + kGather);
    int *hist = reinterpret_cast<int *>(dsm + 2 * kCand + 2 * kGather);
    __shared__ int scratch[kWarps + 1];
    __shared__ int sel[2];
    __shared__ int wc[kWarps + 1];
    __shared__ int cinfo[2]; // this CTA's offset in CTA 0's list; the cluster's count, or -1
    const int cs = static_cast<int>(cluster_nctarank());
    const int cr = static_cast<int>(cluster_ctarank());
    const int ncl = gridDim.x / cs;
    const uint32_t gk0 = mapa_shared(smem_u32(gkey), 0), gi0 = mapa_shared(smem_u32(gidx), 0);
    const uint32_t cnt_local = smem_u32(&wc[kWarps]);
    grid_dep_wait();
    grid_dep_launch();
    for (int row = blockIdx.x / cs; row < T; row += ncl) { // the same rows in every CTA of the cluster
        int n = valid_len[row];
        if (n < 0)
            n = 0;
        if (n > ld) {
            if (cr == 0 && threadIdx.x == 0)
                atomicOr(status, DSA_DEV_BAD_POSITION);
            n = static_cast<int>(ld);
        }
        int32_t *out = idx + static_cast<int64_t>(row) * k;
        if (n <= k) {
            if (cr == 0)
                for (int j = threadIdx.x; j < k; j += kThreads)
                    out[j] = j < n ? j : -1;
            continue;
        }
        const float *r = logits + static_cast<int64_t>(row) * ld;
        const bool vec = (reinterpret_cast<uintptr_t>(r) & 15u) == 0;
        const uint32_t thr = n > kGather ? row_threshold<kThreads>(r, n, k, hist, scratch, sel) : 0u;
        // keys before the row's first 16-byte boundary, then chunks of a multiple
        // of 4 keys from there (fp32 rows are 4-byte aligned)
        int h = static_cast<int>((4u - ((reinterpret_cast<uintptr_t>(r) >> 2) & 3u)) & 3u);
        h = h < n ? h : n;
        const int chunk = ((n - h + cs - 1) / cs + 3) & ~3;
        const int c0 = cr == 0 ? 0 : (h + cr * chunk < n ? h + cr * chunk : n);
        const int c1 = h + (cr + 1) * chunk < n ? h + (cr + 1) * chunk : n;
        if (thr == 0u) // rows that fit the gathered list: every key is a candidate
            filter_segment<kThreads, true>(r, c0, c1, cr == 0 ? h : 0, thr, lkey, lidx, wc);
        else
            filter_segment<kThreads, false>(r, c0, c1, cr == 0 ? h : 0, thr, lkey, lidx, wc);
        cluster_sync_all(); // every CTA's count is in its wc[kWarps]
        if (threadIdx.x == 0) {
            int off = 0, tot = 0;
            bool bad = false;
            for (int q = 0; q < cs; ++q) {
                const int c = static_cast<int>(ld_cluster_u32(mapa_shared(cnt_local, q)));
                bad |= c < 0;
                off += q < cr ? c : 0;
                tot += c;
            }
            cinfo[0] = off;
            cinfo[1] = (bad || tot < k || tot > kGather) ? -1 : tot;
        }
        __syncthreads();
        const int nc = cinfo[1];
        if (nc >= 0) {
            const int off = cinfo[0], mine = wc[kWarps];
            for (int f = threadIdx.x; f < mine; f += kThreads) {
                const int a = cand_slot(wc, f);
                st_cluster_u32(gk0 + 4u * (off + f), lkey[a]);
                st_cluster_u32(gi0 + 4u * (off + f), static_cast<uint32_t>(lidx[a]));
            }
        }
        cluster_sync_all(); // CTA 0's list is complete; nothing of a peer is touched after this
        if (cr == 0) {
            if (nc >= 0)
                select_candidates<kThreads>(gkey, gidx, nc, k, out, hist, sel);
            else if (vec)
                topk_row<kThreads, true>(r, n, k, out, hist, scratch, sel);
            else
                topk_row<kThreads, false>(r, n, k, out, hist, scratch, sel);
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
    const int sms = num_sms();
    cudaError_t e;
    if (a.T <= 2 * sms && !a.row_flag) {
        // Few rows (decode): each row's latency is the cost, so a row gets as
        // many CTAs as the SMs allow and is read once.  Many rows (prefill): one
        // small CTA per row keeps four rows in flight per SM.
        static std::atomic<bool> attr_set[64];
        if (cudaError_t e_attr = raise_smem_limit_once(topk_cluster_kernel, kSmemTopk, attr_set);
            e_attr != cudaSuccess) {
            snprintf(err, errlen, "cudaFuncSetAttribute(topk): %s", cudaGetErrorString(e_attr));
            return DSA_ERR_CUDA;
        }
        int cs = 1;
        while (cs < 8 && a.T * cs * 2 <= sms)
            cs *= 2;
        const int clusters = a.T < sms / cs ? a.T : sms / cs;
        e = launch_pdl(topk_cluster_kernel, dim3(static_cast<unsigned>(clusters * cs)), dim3(kThreads), kSmemTopk,
                       stream, static_cast<unsigned>(cs), a.logits, a.ld, a.T, a.valid_len, a.k, a.idx, status);
    } else {
        static std::atomic<bool> rows_attr[64];
        if (cudaError_t e_attr = raise_smem_limit_once(topk_rows_kernel, kRowSmem, rows_attr); e_attr != cudaSuccess) {
            snprintf(err, errlen, "cudaFuncSetAttribute(topk rows): %s", cudaGetErrorString(e_attr));
            return DSA_ERR_CUDA;
        }
        // (with a row filter, few rows are expected: one CTA per SM walks the flags)
        const int cap_grid = a.row_flag ? sms : 65535 * 4;
        const int grid = a.T < cap_grid ? a.T : cap_grid;
        e = launch_pdl(topk_rows_kernel, dim3(grid), dim3(kRowThreads), kRowSmem, stream, 1, a.logits, a.ld, a.T,
                       a.valid_len, a.k, a.idx, status, a.row_flag);
    }
    if (e != cudaSuccess) {
        snprintf(err, errlen, "topk launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}


size_t topk_candidates_smem(int S, int cap)
{
    return (static_cast<size_t>(2) * cap + kCandHistInts + 2 * static_cast<size_t>((S + 31) / 32)) * 4;
}

int launch_topk_threshold(const float *samp, int ld_s, int T, const int32_t *q_pos, const int32_t *qpos_s, int S,
                          int k, int cap, float *thr, cudaStream_t stream, char *err, size_t errlen)
{
    const int grid = T < 4 * num_sms() ? T : 4 * num_sms();
    cudaError_t e = launch_pdl(topk_threshold_kernel, dim3(grid), dim3(kRowThreads), 0, stream, 1, samp, ld_s, T,
                               q_pos, qpos_s, S, k, cap, thr);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "topk threshold launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

int launch_topk_candidates(const uint2 *cand, const int32_t *cand_cnt, int cap, int T, const int32_t *q_pos, int S,
                           int k, int32_t *idx, int32_t *flag, cudaStream_t stream, char *err, size_t errlen)
{
    const size_t smem = topk_candidates_smem(S, cap);
    if (smem > kCandSmemMax) {
        snprintf(err, errlen, "topk candidates: %zu bytes of shared memory needed", smem);
        return DSA_ERR_UNSUPPORTED;
    }
    // the attribute is set once per device to the largest size any call may ask for
    static std::atomic<bool> attr_set[64];
    if (cudaError_t e_attr = raise_smem_limit_once(topk_candidates_kernel, kCandSmemMax, attr_set);
        e_attr != cudaSuccess) {
        snprintf(err, errlen, "cudaFuncSetAttribute(topk candidates): %s", cudaGetErrorString(e_attr));
        return DSA_ERR_CUDA;
    }
    // as many rows in flight per SM as shared memory allows (4 at most: the phases of a row end in barriers)
    int per_sm = static_cast<int>(232448 / (smem + 2048));
    per_sm = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
    const int grid = T < per_sm * num_sms() ? T : per_sm * num_sms();
    cudaError_t e = launch_pdl(topk_candidates_kernel, dim3(grid), dim3(kRowThreads), smem, stream, 1, cand, cand_cnt,
                               cap, T, q_pos, S, k, idx, flag);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "topk candidates launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

} // namespace dsa
