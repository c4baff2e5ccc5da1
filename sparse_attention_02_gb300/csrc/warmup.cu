// Indexer warm-up (training path) on sm_103a: the KL loss of the lightning
// indexer against the main attention and its gradients.
//
// Defines (release summary "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency
// with DeepSeek Sparse Attention", section "Method": a dense warm-up trains only
// the indexer, against a KL-divergence-to-main-attention target), for query row
// t at position q_pos[t] over keys s <= q_pos[t]:
//     p[t,s]   = mean over heads h of softmax_s(sm_scale * <Q[t,h], KV[s]>)
//     I[t,s]   = sum_j w[t,j] ReLU(a[t,j,s]),  a[t,j,s] = <q[t,j], k[s]>
//     L[t]     = sum_s p (ln p - ln softmax(I)_s)
//     g[t,s]   = softmax(I)_s - p[t,s]                       (dL/dI)
//     dw[t,j]  = sum_s g ReLU(a),  dq[t,j] = sum_s g w[t,j] [a > 0] k[s],
//     dk[s]    = sum_t sum_j g w[t,j] [a > 0] q[t,j]
// with q, k the dequantised FP8 indexer inputs (code * scale; the quantiser
// passes gradients straight through).
//
// Kernels, in order:
//   attn_target_kernel  tcgen05 BF16, one query token per CTA, its 128 heads x
//                       576 columns resident in shared memory, key tiles of 128
//                       streamed in 64-column chunks.  Pass 0: D = Q K^T with
//                       heads on TMEM lanes, each thread a head's running max
//                       and sum over the keys -> the head's LSE.  Pass 1: the
//                       same operands with the roles swapped, D = K Q^T, keys
//                       on lanes, each thread a key's sum over heads of
//                       exp(S - LSE) / H -> p.
//   (the FP8 indexer)   I, as dsa_indexer_logits computes it.
//   kl_grad_kernel      one CTA per row: LSE of I, the loss, g over I in place.
//   codes_kernel        the FP8 codes as bf16 (exact) and the bounds of the
//                       exact ReLU decision.
//   bwd_tc_kernel<0>    tcgen05 BF16, one CTA per tile of 128 (t, j) rows:
//                       a = Q K^T per 128-key tile, c = g ks [a > 0] as a bf16
//                       hi + lo pair in TMEM, dq += C K; dw on the way.
//   bwd_tc_kernel<1>    the same per (128-key tile, chunk of row tiles) with
//                       the roles swapped: dk += C^T Q, chunks meeting in atomics.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

// ------------------------------------------------------------------ target
constexpr int kTD = 576;
constexpr int kTChunks = kTD / 64;             // 64-column (128-byte) chunks of a latent row
constexpr int kTTile = 128;                    // keys per tile
constexpr int kTStages = 4;
constexpr int kTChunkBytes = 128 * 128;        // 128 rows x 64 bf16
constexpr int kTOffQ = 0;
constexpr int kTOffKV = kTOffQ + kTChunks * kTChunkBytes;   // 144 KB
constexpr int kTOffLse = kTOffKV + kTStages * kTChunkBytes; // 208 KB
constexpr int kTOffMl = kTOffLse + 128 * 4;                  // the second key half's (max, sum) per head
constexpr int kTOffBar = kTOffMl + 128 * 8;
constexpr int kTNBar = 2 * kTStages + 4 + 4;
constexpr int kTOffMisc = kTOffBar + kTNBar * 8;
constexpr int kTSmem = kTOffMisc + 64 + 1024;
constexpr int kTThreads = 10 * 32;             // producer, MMA, eight epilogue warps (two per TMEM quadrant)
static_assert(kTSmem <= 232448, "target kernel shared memory");

struct TargetParams {
    const int32_t *q_pos;
    int T, S, H;
    float scale_log2;
    float *p;
    int64_t ld;
    unsigned *status;
};

__global__ void __launch_bounds__(kTThreads, 1)
    attn_target_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                       TargetParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    float *lse2 = reinterpret_cast<float *>(smem + kTOffLse);
    const uint32_t bar0 = sbase + kTOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kTStages + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * kTStages + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * kTStages + 2 + a); };
    const uint32_t q_bar = bar0 + 8u * (2 * kTStages + 4);
    const uint32_t done_bar = bar0 + 8u * (2 * kTStages + 5);
    const uint32_t ml_bar = bar0 + 8u * (2 * kTStages + 6);  // the second halves' (max, sum) are in shared memory
    const uint32_t lse_bar = bar0 + 8u * (2 * kTStages + 7); // every head's LSE is in shared memory
    float *mls = reinterpret_cast<float *>(smem + kTOffMl);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + kTOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kTOffMisc + 4);
    int *pos_s = reinterpret_cast<int *>(smem + kTOffMisc + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = gridDim.x - 1 - blockIdx.x; // long rows first

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 8);
        }
        mbar_init(q_bar, 1);
        mbar_init(done_bar, 1);
        mbar_init(ml_bar, 4);
        mbar_init(lse_bar, 4);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1)
        tmem_alloc(sbase + kTOffMisc, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    grid_dep_wait();
    grid_dep_launch();
    if (threadIdx.x == 0) {
        int64_t qp = p.q_pos[t];
        if (qp > p.S - 1) {
            atomicOr(p.status, DSA_DEV_BAD_POSITION);
            qp = p.S - 1;
        }
        *pos_s = qp < 0 ? -1 : static_cast<int>(qp);
    }
    __syncthreads();
    const int pos = *pos_s;
    const int ntiles = pos < 0 ? 0 : pos / kTTile + 1;
    const int items = 2 * ntiles; // pass 0 tiles, then pass 1 tiles
    // p's row is summed from the two head halves of pass 1
    for (int s = threadIdx.x; s <= pos; s += kTThreads)
        p.p[(int64_t)t * p.ld + s] = 0.f;
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int issued = 0;
        if (lane == 0 && ntiles > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_kv);
            mbar_arrive_expect_tx(q_bar, kTChunks * kTChunkBytes);
            for (int c = 0; c < kTChunks; ++c)
                tma_load_2d(sbase + kTOffQ + c * kTChunkBytes, &tm_q, q_bar, 64 * c, t * p.H);
            for (int it = 0; it < items; ++it) {
                const int kt = it % ntiles;
                bool ok = true;
                for (int c = 0; c < kTChunks; ++c, ++issued) {
                    const int s = issued % kTStages;
                    if (issued >= kTStages &&
                        !mbar_wait(empty_bar(s), ((issued / kTStages) - 1) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), kTChunkBytes);
                    tma_load_2d(sbase + kTOffKV + s * kTChunkBytes, &tm_kv, full_bar(s), 64 * c, kt * kTTile);
                }
                if (!ok)
                    break;
            }
            // every load issued has landed before the CTA exits
            mbar_drain(q_bar, 0);
            for (int i = issued - kTStages > 0 ? issued - kTStages : 0; i < issued; ++i)
                mbar_drain(full_bar(i % kTStages), (i / kTStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_f32acc(128, 128, 1u, false, false);
        bool ok = ntiles == 0 || mbar_wait_warp(q_bar, 0, abort_flag, p.status);
        int chunk = 0;
        for (int it = 0; ok && it < items; ++it) {
            const int a = it & 1, use = it >> 1;
            const bool pass1 = it >= ntiles;
            if (use >= 1 && !mbar_wait_warp(acce_bar(a), (use - 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int c = 0; c < kTChunks; ++c, ++chunk) {
                const int s = chunk % kTStages;
                if (!mbar_wait_warp(full_bar(s), (chunk / kTStages) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t qa = sbase + kTOffQ + c * kTChunkBytes;
                    const uint32_t ka = sbase + kTOffKV + s * kTChunkBytes;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // pass 0: A = Q (M = heads), B = keys; pass 1: A = keys (M = keys), B = Q
                        const uint64_t qd = sdesc(qa + 32 * k, 16, 1024, 2);
                        const uint64_t kd = sdesc(ka + 32 * k, 16, 1024, 2);
                        umma_f16_ss(tmem + 128 * a, pass1 ? kd : qd, pass1 ? qd : kd, idesc,
                                    (c > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(empty_bar(s));
                    if (c == kTChunks - 1)
                        umma_commit(accf_bar(a));
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            umma_commit(done_bar);
            mbar_drain(done_bar, 0);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- epilogue
        // Two warps per TMEM lane quadrant: half hh takes columns 64 hh .. 64 hh + 63 of
        // each accumulator (pass 0: keys of the tile; pass 1: heads).
        const int quad = warp & 3, hh = (warp - 2) >> 2;
        const int row = quad * 32 + lane; // pass 0: head; pass 1: key within the tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        float m = -INFINITY, l = 0.f;
        for (int it = 0; it < items; ++it) {
            const int a = it & 1, use = it >> 1;
            const bool pass1 = it >= ntiles;
            const int kt = it % ntiles;
            if (it == ntiles) {
                // pass 0 done: the halves' (max, sum) of each head meet, its LSE (log2 units)
                // goes to shared memory, and every warp waits for all of them
                if (hh == 1) {
                    mls[2 * row] = m;
                    mls[2 * row + 1] = l;
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(ml_bar);
                } else {
                    if (!mbar_wait_warp(ml_bar, 0, abort_flag, p.status))
                        break;
                    const float m1 = mls[2 * row], l1 = mls[2 * row + 1];
                    const float mm = fmaxf(m, m1);
                    const float ll = (m == -INFINITY ? 0.f : l * exp2f(m - mm)) + (m1 == -INFINITY ? 0.f : l1 * exp2f(m1 - mm));
                    lse2[row] = ll > 0.f ? mm + __log2f(ll) : INFINITY;
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(lse_bar);
                }
                if (!mbar_wait_warp(lse_bar, 0, abort_flag, p.status))
                    break;
            }
            if (!mbar_wait_warp(accf_bar(a), use & 1, abort_flag, p.status))
                break;
            tc_fence_after();
            float bsum = 0.f; // pass 1: this key's sum over the half's heads
#pragma unroll 1
            for (int c0 = 64 * hh; c0 < 64 * hh + 64; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_base + 128 * a + c0, r);
                tmem_ld_wait();
                if (c0 == 64 * hh + 32) {
                    // this warp's columns of the accumulator are in registers: release it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(acce_bar(a));
                }
                if (!pass1) {
                    // thread = head: online max and sum over these 32 keys (the valid ones)
                    float bm = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (kt * kTTile + c0 + c <= pos)
                            bm = fmaxf(bm, __uint_as_float(r[c]) * p.scale_log2);
                    if (bm > m) {
                        l *= exp2f(m - bm);
                        m = bm;
                    }
                    float ls = 0.f;
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (kt * kTTile + c0 + c <= pos)
                            ls += exp2f(__uint_as_float(r[c]) * p.scale_log2 - m);
                    l += ls;
                } else {
                    // thread = key: exp(S - LSE) of heads c0 .. c0 + 31 (those below H)
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (c0 + c < p.H)
                            bsum += exp2f(__uint_as_float(r[c]) * p.scale_log2 - lse2[c0 + c]);
                }
            }
            if (pass1) {
                const int s = kt * kTTile + row;
                if (s <= pos) // two additions onto 0: the same sum in either order
                    atomicAdd(p.p + (int64_t)t * p.ld + s, bsum / static_cast<float>(p.H));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------- KL, g in place
// One CTA per row: m = max I, lse = m + ln sum exp(I - m), L = sum p (ln p -
// I + lse) over p > 0, g = exp(I - lse) - p written over I.
__global__ void __launch_bounds__(256)
    kl_grad_kernel(float *__restrict__ ig, const float *__restrict__ p, int64_t ld, const int32_t *__restrict__ q_pos,
                   int T, int S, float *__restrict__ loss)
{
    __shared__ float red[8];
    grid_dep_wait();
    grid_dep_launch();
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        int64_t n64 = static_cast<int64_t>(q_pos[t]) + 1;
        const int n = static_cast<int>(n64 < 0 ? 0 : (n64 > S ? S : n64));
        float *row = ig + (int64_t)t * ld;
        const float *pr = p + (int64_t)t * ld;
        auto block_sum = [&](float v, bool is_max) -> float {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float y = __shfl_xor_sync(0xffffffffu, v, o);
                v = is_max ? fmaxf(v, y) : v + y;
            }
            if ((threadIdx.x & 31) == 0)
                red[threadIdx.x >> 5] = v;
            __syncthreads();
            float x = red[0];
            for (int w = 1; w < 8; ++w)
                x = is_max ? fmaxf(x, red[w]) : x + red[w];
            __syncthreads();
            return x;
        };
        float m = -INFINITY;
        for (int s = threadIdx.x; s < n; s += 256)
            m = fmaxf(m, row[s]);
        m = block_sum(m, true);
        float z = 0.f;
        for (int s = threadIdx.x; s < n; s += 256)
            z += expf(row[s] - m);
        z = block_sum(z, false);
        const float lse = m + logf(z);
        float L = 0.f;
        for (int s = threadIdx.x; s < n; s += 256) {
            const float x = row[s], ps = pr[s];
            if (ps > 0.f)
                L += ps * (logf(ps) - (x - lse));
            row[s] = expf(x - lse) - ps;
        }
        L = block_sum(L, false);
        if (threadIdx.x == 0)
            loss[t] = n > 0 ? L : 0.f;
    }
}

// ------------------------------------------------------------ FP8 decoding
// E4M3 ("fn") code -> float from the format's definition: bias 7, three
// mantissa bits, subnormals at exponent field 0.
__device__ __forceinline__ float e4m3_to_float(uint32_t c)
{
    const uint32_t sign = (c & 0x80u) << 24;
    const uint32_t e = (c >> 3) & 15u, man = c & 7u;
    if (e == 0)
        return __uint_as_float(sign | __float_as_uint(static_cast<float>(man) * 0.001953125f)); // man * 2^-9
    return __uint_as_float(sign | ((e + 120u) << 23) | (man << 20));
}

// ------------------------------------------------- backward on tensor cores
// Both gradient contractions run on BF16 tensor cores, in two kernels of one
// shape.  The operands are the FP8 codes as bf16 (exact); the scales are
// positive, so they multiply out of a and of the ReLU decision:
//   rows (KEYS = false): one CTA per tile of 128 (t, j) rows, walking the key
//     tiles its rows see.  D1 = Qc Kc^T (rows x keys, fp32 in TMEM); per
//     element c = g ks [a > 0] and dw += g ks a; D2 += C Kc.  Then
//     dq[t,j,:] = w[t,j] D2 and dw[t,j] = q_scale[t] sum.
//   keys (KEYS = true): one CTA per (128-key tile, chunk of row tiles).
//     D1 = Kc Qc^T (keys x rows); c = g w q_scale [a > 0]; D2 += C Qc, and D2
//     is added to dk (chunks meet in the atomics; dk is zeroed first).
// C reaches the tensor cores as a bf16 pair hi + lo (c to ~2^-17 relative), so
// D2 is an fp32 sum of exact products.  The streamed code tile serves both
// MMAs: K-major as D1's B operand, MN-major as D2's.
// ReLU decision, exact: the tensor cores sum exact products in fp32, whose
// error is below 2^-16 sum_d |q_d k_d| for 128 terms (127 additions at most
// 2^-23 relative each); that sum is bounded by the q row's L1 norm times the
// key row's largest code.  Where |a| is within that bound (and the element
// contributes), the warp forms the exact sum of the code products as a 64-bit
// integer (codes times 2^9 are integers, products below 2^36, 128 of them
// below 2^43) and takes its sign.
constexpr int kGThreads = 320;             // producer, MMA issuer, eight epilogue warps (two per TMEM quadrant)
constexpr int kGStages = 3;                // streamed code tiles
constexpr int kGAtom = 128 * 128;          // one 64-column SW128 atom of a 128-row bf16 tile
constexpr int kGTileBytes = 2 * kGAtom;    // 128 rows x 128 codes
constexpr int kGAux = 6 * 128 * 4;         // per-stage column data (floats)
constexpr int kGRowChunk = 64;             // row tiles per CTA of the keys kernel
constexpr int kGOffRes = 0;                                   // the CTA's own tile
constexpr int kGOffSt = kGOffRes + kGTileBytes;               // streamed tiles
constexpr int kGOffAux = kGOffSt + kGStages * kGTileBytes;
constexpr int kGOffList = kGOffAux + kGStages * kGAux;        // active row tiles (keys kernel)
constexpr int kGOffBar = kGOffList + kGRowChunk * 4;
constexpr int kGNBar = 18;
constexpr int kGOffMisc = kGOffBar + kGNBar * 8;
constexpr int kGSmem = kGOffMisc + 64 + 1024;
static_assert(kGSmem <= 232448, "backward kernel shared memory");
// barriers
constexpr int G_RES = 0, G_SF = 1, G_SE = 4, G_DF = 7, G_DE = 9, G_CF = 11, G_CE = 13, G_D2 = 15, G_DONE = 16,
              G_DW = 17; // the second key half's dw partial sums are in shared memory
// TMEM columns: D1 (two buffers), D2, C (two slots of 64 keys: hi then lo bf16 pairs)
constexpr uint32_t GT_D1 = 0, GT_D2 = 256, GT_C = 384;

struct BwdParams {
    const uint8_t *q8, *k8;  // FP8 codes (exact decisions)
    const float *q_scale, *w, *k_scale;
    const float *qb;         // [T * HI] 2^-16 x the q code row's L1 norm (rounded up)
    const float *wq;         // [T * HI] w[t,j] q_scale[t]
    const float *kinf;       // [S] largest |code| of the key row
    const int32_t *q_pos;
    const float *g;          // [T, ldg] dL/dI
    int64_t ldg;
    int T, S, HI;
    float *dw, *dq, *dk;
    unsigned *status;
};

// E4M3 ("fn") code times 2^9 as an integer: (8 + mantissa) << (exponent - 1), or
// the mantissa itself for subnormals.
__device__ __forceinline__ int e4m3_q9(uint32_t c)
{
    const int e = static_cast<int>((c >> 3) & 15u), m = static_cast<int>(c & 7u);
    const int mag = e ? (8 | m) << (e - 1) : m;
    return (c & 0x80u) ? -mag : mag;
}

// Exact sign test of <q code row, k code row> (128 codes each), by the whole warp.
__device__ __forceinline__ bool exact_dot_positive(const uint8_t *qr, const uint8_t *kr, int lane)
{
    const uint32_t qw = __ldg(reinterpret_cast<const uint32_t *>(qr) + lane);
    const uint32_t kw = __ldg(reinterpret_cast<const uint32_t *>(kr) + lane);
    long long acc = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b)
        acc += static_cast<long long>(e4m3_q9((qw >> (8 * b)) & 255u)) * e4m3_q9((kw >> (8 * b)) & 255u);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc > 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ int clamp_pos(const BwdParams &p, int t)
{
    if (t >= p.T)
        return -1;
    const int qp = p.q_pos[t];
    return qp > p.S - 1 ? p.S - 1 : qp;
}

// Largest clamped position among the tokens of row tile rt (-1: none sees a key).
__device__ __forceinline__ int tile_maxpos(const BwdParams &p, int rt, int tpt)
{
    int m = -1;
    for (int tl = 0; tl < tpt; ++tl) {
        const int q = clamp_pos(p, rt * tpt + tl);
        m = q > m ? q : m;
    }
    return m;
}

template <bool KEYS>
__global__ void __launch_bounds__(kGThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_str, BwdParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + kGOffBar + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + kGOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kGOffMisc + 4);
    int *n_items_s = reinterpret_cast<int *>(smem + kGOffMisc + 8);
    int *list = reinterpret_cast<int *>(smem + kGOffList);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tpt = 128 / p.HI; // tokens per row tile
    const int nrt = (p.T * p.HI + 127) / 128;
    // this CTA's own tile: a row tile (rows kernel) or a key tile (keys kernel)
    const int own = KEYS ? static_cast<int>(blockIdx.x) : nrt - 1 - static_cast<int>(blockIdx.x);

    if (threadIdx.x == 0) {
        mbar_init(bar(G_RES), 1);
        for (int i = 0; i < kGStages; ++i) {
            mbar_init(bar(G_SF + i), 1);
            mbar_init(bar(G_SE + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(G_DF + i), 1);
            mbar_init(bar(G_DE + i), 8);
            mbar_init(bar(G_CF + i), 4);
            mbar_init(bar(G_CE + i), 1);
        }
        mbar_init(bar(G_D2), 1);
        mbar_init(bar(G_DONE), 1);
        mbar_init(bar(G_DW), 4);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1)
        tmem_alloc(sbase + kGOffMisc, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    grid_dep_wait(); // no global memory before this: the previous kernel may still be running
    grid_dep_launch();
    // ---- the work list: key tiles 0 .. (rows kernel), active row tiles of the chunk (keys kernel)
    if (warp == 0) {
        if (!KEYS) {
            if (lane == 0) {
                const int mp = tile_maxpos(p, own, tpt);
                *n_items_s = mp < 0 ? 0 : mp / 128 + 1;
            }
        } else {
            const int r0 = static_cast<int>(blockIdx.y) * kGRowChunk, s0 = own * 128;
            int n = 0;
            for (int b = 0; b < kGRowChunk; b += 32) {
                const int rt = r0 + b + lane;
                const bool act = rt < nrt && tile_maxpos(p, rt, tpt) >= s0;
                const unsigned m = __ballot_sync(0xffffffffu, act);
                if (act)
                    list[n + __popc(m & ((1u << lane) - 1u))] = rt;
                n += __popc(m);
            }
            if (lane == 0)
                *n_items_s = n;
        }
    }
    __syncthreads();
    const int n_items = *n_items_s;
    bool ok = true;

    if (warp == 0) {
        // --------------------------------------------- producer: tiles by TMA, column data
        int pos[4];
#pragma unroll
        for (int tl = 0; tl < 4; ++tl)
            pos[tl] = (!KEYS && tl < tpt) ? clamp_pos(p, own * tpt + tl) : -1;
        if (lane == 0 && n_items > 0) {
            tma_prefetch_desc(&tm_res);
            tma_prefetch_desc(&tm_str);
            mbar_arrive_expect_tx(bar(G_RES), kGTileBytes);
            tma_load_2d(sbase + kGOffRes, &tm_res, bar(G_RES), 0, own * 128);
            tma_load_2d(sbase + kGOffRes + kGAtom, &tm_res, bar(G_RES), 64, own * 128);
        }
        int issued = 0; // streamed tiles whose loads were issued (all n_items unless a wait gave up)
        for (int i = 0; i < n_items; ++i) {
            const int st = i % kGStages;
            if (i >= kGStages && !mbar_wait_warp(bar(G_SE + st), ((i / kGStages) - 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            float *aux = reinterpret_cast<float *>(smem + kGOffAux + st * kGAux);
            const int str = KEYS ? list[i] : i; // streamed tile: row tile / key tile
            if (!KEYS) {
                // [tl][key]: g ks of token tl (0 where the token does not see the key); [4][key]: max |k code|
                float v[4][4], kv[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int s = str * 128 + 32 * m + lane;
                    kv[m] = s < p.S ? p.kinf[s] : 0.f;
#pragma unroll
                    for (int tl = 0; tl < 4; ++tl)
                        v[tl][m] = (tl < tpt && s <= pos[tl])
                                       ? p.g[(int64_t)(own * tpt + tl) * p.ldg + s] * p.k_scale[s] : 0.f;
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int tl = 0; tl < 4; ++tl)
                        aux[tl * 128 + 32 * m + lane] = v[tl][m];
                    aux[4 * 128 + 32 * m + lane] = kv[m];
                }
            } else {
                // [tl][key]: g of token tl of the row tile at this CTA's keys; [4][row]: w q_scale; [5][row]: q bound
                int pt[4];
#pragma unroll
                for (int tl = 0; tl < 4; ++tl)
                    pt[tl] = tl < tpt ? clamp_pos(p, str * tpt + tl) : -1;
                float v[4][4], wv[4], bv[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int s = own * 128 + 32 * m + lane, r = str * 128 + 32 * m + lane;
                    const bool rv = r < p.T * p.HI;
                    wv[m] = rv ? p.wq[r] : 0.f;
                    bv[m] = rv ? p.qb[r] : 0.f;
#pragma unroll
                    for (int tl = 0; tl < 4; ++tl)
                        v[tl][m] = s <= pt[tl] ? p.g[(int64_t)(str * tpt + tl) * p.ldg + s] : 0.f;
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int tl = 0; tl < 4; ++tl)
                        aux[tl * 128 + 32 * m + lane] = v[tl][m];
                    aux[4 * 128 + 32 * m + lane] = wv[m];
                    aux[5 * 128 + 32 * m + lane] = bv[m];
                }
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t dst = sbase + kGOffSt + st * kGTileBytes;
                mbar_arrive_expect_tx(bar(G_SF + st), kGTileBytes);
                tma_load_2d(dst, &tm_str, bar(G_SF + st), 0, str * 128);
                tma_load_2d(dst + kGAtom, &tm_str, bar(G_SF + st), 64, str * 128);
            }
            ++issued;
        }
        // every load issued has landed before the CTA exits
        if (lane == 0 && n_items > 0) {
            mbar_drain(bar(G_RES), 0);
            for (int i = issued > kGStages ? issued - kGStages : 0; i < issued; ++i)
                mbar_drain(bar(G_SF + i % kGStages), (i / kGStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t id1 = idesc_f32acc(128, 128, 1u, false, false);
        constexpr uint32_t id2 = idesc_f32acc(128, 128, 1u, false, true);
        // D2 += C(it) . tile(it): keys (rows kernel) / rows (keys kernel) 64 h .. 64 h + 63 of the
        // streamed tile are K, its 128 columns N (MN-major); C's hi then lo pairs are A (TMEM)
        auto mma2 = [&](int it) -> bool {
            const int st = it % kGStages;
            const uint32_t stg = sbase + kGOffSt + st * kGTileBytes;
            for (int h = 0; h < 2; ++h) {
                if (!mbar_wait_warp(bar(G_CF + h), it & 1, abort_flag, p.status))
                    return false;
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = sdesc(stg + (64 * h + 16 * kk) * 128, kGAtom, 1024, 2);
                        const uint32_t ca = tmem + GT_C + 64 * h + 8 * kk;
                        umma_f16_ts(tmem + GT_D2, ca, bd, id2, (it > 0 || h > 0 || kk > 0) ? 1u : 0u);
                        umma_f16_ts(tmem + GT_D2, ca + 32, bd, id2, 1u);
                    }
                    umma_commit(bar(G_CE + h));
                    if (h == 1)
                        umma_commit(bar(G_SE + st));
                }
                __syncwarp();
            }
            return true;
        };
        if (n_items > 0 && !mbar_wait_warp(bar(G_RES), 0, abort_flag, p.status))
            ok = false;
        for (int i = 0; ok && i < n_items; ++i) {
            const int st = i % kGStages, b = i & 1;
            if (!mbar_wait_warp(bar(G_SF + st), (i / kGStages) & 1, abort_flag, p.status) ||
                (i >= 2 && !mbar_wait_warp(bar(G_DE + b), ((i >> 1) - 1) & 1, abort_flag, p.status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t stg = sbase + kGOffSt + st * kGTileBytes, res = sbase + kGOffRes;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kGAtom + 32 * (k & 3);
                    umma_f16_ss(tmem + GT_D1 + 128 * b, sdesc(res + off, 16, 1024, 2), sdesc(stg + off, 16, 1024, 2),
                                id1, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(G_DF + b));
            }
            __syncwarp();
            if (i >= 1 && !mma2(i - 1))
                ok = false;
        }
        if (ok && n_items > 0 && !mma2(n_items - 1))
            ok = false;
        if (lane == 0) {
            if (ok && n_items > 0)
                umma_commit(bar(G_D2));
            umma_commit(bar(G_DONE));
            mbar_drain(bar(G_DONE), 0);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- epilogue
        // Two warps per TMEM lane quadrant: half hh takes keys (rows kernel) / rows (keys
        // kernel) 64 hh .. 64 hh + 63 of each streamed tile, i.e. C slot hh, and D2's
        // columns 64 hh .. 64 hh + 63.
        const int quad = warp & 3, hh = (warp - 2) >> 2;
        const int row = quad * 32 + lane; // TMEM lane: (t, j) row (rows kernel) / key (keys kernel)
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const int rrow = own * 128 + row; // rows kernel: global (t, j) row; keys kernel: key
        const int tl_own = row / p.HI;    // rows kernel: token of this row within the tile (warp-uniform)
        const bool valid = KEYS ? rrow < p.S : rrow < p.T * p.HI;
        const float qb_own = (!KEYS && valid) ? p.qb[rrow] : 0.f;
        const float kinf_own = (KEYS && valid) ? p.kinf[rrow] : 0.f;
        float dw_acc = 0.f;
        for (int i = 0; i < n_items; ++i) {
            const int b = i & 1, st = i % kGStages;
            const int str = KEYS ? list[i] : i;
            // the stage's column data (the producer's stores) and D1
            if (!mbar_wait_warp(bar(G_SF + st), (i / kGStages) & 1, abort_flag, p.status) ||
                !mbar_wait_warp(bar(G_DF + b), (i >> 1) & 1, abort_flag, p.status) ||
                (i >= 1 && !mbar_wait_warp(bar(G_CE + hh), (i - 1) & 1, abort_flag, p.status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *aux = reinterpret_cast<const float *>(smem + kGOffAux + st * kGAux);
            float gt[4] = {0.f, 0.f, 0.f, 0.f}; // keys kernel: this key's g for each token of the row tile
            if (KEYS)
#pragma unroll
                for (int tl = 0; tl < 4; ++tl)
                    gt[tl] = aux[tl * 128 + row];
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * hh + cc;
                uint32_t r[32];
                tmem_ld32(lane_base + GT_D1 + 128 * b + 32 * c, r);
                tmem_ld_wait();
                if (cc == 1) { // this warp's part of D1 is in registers: release it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar(G_DE + b));
                }
                // per column: the coefficient if a > 0, and whether the fp32 sign can be trusted
                float cv[32];
                uint32_t posm = 0u, ambm = 0u;
                const int tlc = (32 * c) / p.HI; // keys kernel: token of these columns (uniform)
                const float gc = tlc == 0 ? gt[0] : tlc == 1 ? gt[1] : tlc == 2 ? gt[2] : gt[3];
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const int col = 32 * c + 4 * e4;
                    float4 v4, b4;
                    if (!KEYS) {
                        v4 = *reinterpret_cast<const float4 *>(aux + tl_own * 128 + col);
                        b4 = *reinterpret_cast<const float4 *>(aux + 4 * 128 + col);
                    } else {
                        v4 = *reinterpret_cast<const float4 *>(aux + 4 * 128 + col);
                        b4 = *reinterpret_cast<const float4 *>(aux + 5 * 128 + col);
                    }
                    const float vv[4] = {v4.x, v4.y, v4.z, v4.w}, bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int e = 4 * e4 + q;
                        const float a = __uint_as_float(r[e]);
                        const float v = KEYS ? gc * vv[q] : vv[q];
                        const float bnd = KEYS ? bb[q] * kinf_own : qb_own * bb[q];
                        cv[e] = v;
                        posm |= (a > 0.f ? 1u : 0u) << e;
                        ambm |= ((v != 0.f && fabsf(a) <= bnd) ? 1u : 0u) << e;
                    }
                }
                // exact decisions where the fp32 sum is within its error bound of 0
                unsigned todo = __ballot_sync(0xffffffffu, ambm != 0u);
                while (todo) {
                    const int L = __ffs(todo) - 1;
                    const uint32_t mL = __shfl_sync(0xffffffffu, ambm, L);
                    const int e = __ffs(mL) - 1;
                    const int qrow = KEYS ? str * 128 + 32 * c + e : own * 128 + quad * 32 + L;
                    const int key = KEYS ? own * 128 + quad * 32 + L : str * 128 + 32 * c + e;
                    const bool pos = exact_dot_positive(p.q8 + (int64_t)qrow * 128, p.k8 + (int64_t)key * 128, lane);
                    if (lane == L) {
                        ambm &= ~(1u << e);
                        posm = pos ? (posm | (1u << e)) : (posm & ~(1u << e));
                    }
                    todo = __ballot_sync(0xffffffffu, ambm != 0u);
                }
                // C = coefficient where a > 0, as hi + lo bf16 pairs
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) {
                    const int e0 = 2 * e2, e1 = e0 + 1;
                    const float c0 = ((posm >> e0) & 1u) ? cv[e0] : 0.f;
                    const float c1 = ((posm >> e1) & 1u) ? cv[e1] : 0.f;
                    if (!KEYS)
                        dw_acc += c0 * __uint_as_float(r[e0]) + c1 * __uint_as_float(r[e1]);
                    const uint32_t hp = pack_bf16x2(c0, c1);
                    hi[e2] = hp;
                    lo[e2] = pack_bf16x2(c0 - __uint_as_float(hp << 16), c1 - __uint_as_float(hp & 0xFFFF0000u));
                }
                tmem_st16(lane_base + GT_C + 64 * hh + 16 * cc, hi);
                tmem_st16(lane_base + GT_C + 64 * hh + 32 + 16 * cc, lo);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(G_CF + hh));
        }
        // ---- D2 out: dq and dw (rows kernel), dk partial sums (keys kernel); D2 columns 64 hh ..
        const bool have = ok && n_items > 0;
        if (have && !mbar_wait_warp(bar(G_D2), 0, abort_flag, p.status))
            ok = false;
        tc_fence_after();
        if (!KEYS) {
            const float wr = valid ? p.w[rrow] : 0.f;
#pragma unroll 1
            for (int c0 = 64 * hh; c0 < 64 * hh + 64; c0 += 32) {
                uint32_t r[32];
                if (have && ok) {
                    tmem_ld32(lane_base + GT_D2 + c0, r);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        r[e] = 0u;
                }
                if (valid) {
                    float4 *dst = reinterpret_cast<float4 *>(p.dq + (int64_t)rrow * 128 + c0);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(wr * __uint_as_float(r[4 * e]), wr * __uint_as_float(r[4 * e + 1]),
                                             wr * __uint_as_float(r[4 * e + 2]), wr * __uint_as_float(r[4 * e + 3]));
                }
            }
            // dw: the second half's partial sums meet the first's in shared memory
            float *dwp = reinterpret_cast<float *>(smem + kGOffAux); // the stages' column data are no longer read
            if (hh == 1) {
                if (have && ok)
                    dwp[row] = dw_acc;
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(G_DW));
            } else {
                const bool got = !(have && ok) || mbar_wait_warp(bar(G_DW), 0, abort_flag, p.status);
                if (valid)
                    p.dw[rrow] = p.q_scale[rrow / p.HI] * (dw_acc + (have && ok && got ? dwp[row] : 0.f));
            }
        } else if (have && ok) { // warp-uniform: the TMEM loads are warp-collective
#pragma unroll 1
            for (int c0 = 64 * hh; c0 < 64 * hh + 64; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_base + GT_D2 + c0, r);
                tmem_ld_wait();
                if (valid) {
                    float *dst = p.dk + (int64_t)rrow * 128 + c0;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        atomicAdd(dst + e, __uint_as_float(r[e]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// The codes as bf16 (exact) for the tensor cores, the decision bounds (qb[row]
// = 2^-16 x L1 norm of a q code row, rounded up; kinf[s] = largest |code| of
// key s) and wq[row] = w q_scale.  One warp per row; rows [0, nq) are q rows
// (nq = T H_I), then key rows.
__global__ void __launch_bounds__(256)
    codes_kernel(const uint8_t *__restrict__ q8, int nq, const uint8_t *__restrict__ k8, int nk,
                 const float *__restrict__ w, const float *__restrict__ q_scale, int HI,
                 __nv_bfloat16 *__restrict__ qc, float *__restrict__ qb, float *__restrict__ wq,
                 __nv_bfloat16 *__restrict__ kc, float *__restrict__ kinf)
{
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int r = static_cast<int>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (r >= nq + nk)
        return;
    const bool isq = r < nq;
    const uint8_t *src = isq ? q8 + (int64_t)r * 128 : k8 + (int64_t)(r - nq) * 128;
    const uint32_t wv = reinterpret_cast<const uint32_t *>(src)[lane];
    float v[4];
    float l1 = 0.f, mx = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        v[b] = e4m3_to_float((wv >> (8 * b)) & 255u);
        l1 += fabsf(v[b]);
        mx = fmaxf(mx, fabsf(v[b]));
    }
    __nv_bfloat16 *dst = isq ? qc + (int64_t)r * 128 : kc + (int64_t)(r - nq) * 128;
    const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16(v[0]))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16(v[1]))) << 16);
    const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16(v[2]))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16(v[3]))) << 16);
    reinterpret_cast<uint2 *>(dst)[lane] = make_uint2(lo, hi);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
        if (isq) {
            qb[r] = l1 * (1.52587890625e-05f * 1.00390625f); // 2^-16 (1 + 2^-8): margin for this sum's rounding
            wq[r] = w[r] * q_scale[r / HI];
        } else {
            kinf[r - nq] = mx;
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WLayout {
    size_t p, ig, qc, kc, qb, wq, kinf, total;
};

WLayout wlayout(int T, int S, int HI)
{
    WLayout l;
    size_t o = 0;
    l.p = o;
    o += align256(static_cast<size_t>(T) * S * 4);
    l.ig = o;
    o += align256(static_cast<size_t>(T) * S * 4);
    l.qc = o;
    o += align256(static_cast<size_t>(T) * HI * 128 * 2);
    l.kc = o;
    o += align256(static_cast<size_t>(S) * 128 * 2);
    l.qb = o;
    o += align256(static_cast<size_t>(T) * HI * 4);
    l.wq = o;
    o += align256(static_cast<size_t>(T) * HI * 4);
    l.kinf = o;
    o += align256(static_cast<size_t>(S) * 4);
    l.total = o;
    return l;
}

int launch_backward(const WarmupArgs &a, const WLayout &l, char *ws, const float *ig, unsigned *status,
                    cudaStream_t stream, char *err, size_t errlen)
{
    __nv_bfloat16 *qc = reinterpret_cast<__nv_bfloat16 *>(ws + l.qc);
    __nv_bfloat16 *kc = reinterpret_cast<__nv_bfloat16 *>(ws + l.kc);
    float *qb = reinterpret_cast<float *>(ws + l.qb);
    float *wq = reinterpret_cast<float *>(ws + l.wq);
    float *kinf = reinterpret_cast<float *>(ws + l.kinf);
    const int nq = a.T * a.HI;
    cudaError_t e = launch_pdl(codes_kernel, dim3(static_cast<unsigned>((nq + a.S + 7) / 8)), dim3(256), 0, stream, 1,
                               static_cast<const uint8_t *>(a.q8), nq, static_cast<const uint8_t *>(a.k8), a.S, a.w,
                               a.q_scale, a.HI, qc, qb, wq, kc, kinf);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "warm-up codes launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    static std::atomic<bool> rows_attr[64], keys_attr[64];
    if (cudaError_t ea = raise_smem_limit_once(bwd_tc_kernel<false>, kGSmem, rows_attr); ea != cudaSuccess) {
        snprintf(err, errlen, "cudaFuncSetAttribute(warm-up rows): %s", cudaGetErrorString(ea));
        return DSA_ERR_CUDA;
    }
    if (cudaError_t ea = raise_smem_limit_once(bwd_tc_kernel<true>, kGSmem, keys_attr); ea != cudaSuccess) {
        snprintf(err, errlen, "cudaFuncSetAttribute(warm-up keys): %s", cudaGetErrorString(ea));
        return DSA_ERR_CUDA;
    }
    CUtensorMap tq, tk;
    if (!encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qc, 128, (uint64_t)nq, 256, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B, err, errlen) ||
        !encode_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kc, 128, (uint64_t)a.S, 256, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B, err, errlen))
        return DSA_ERR_CUDA;
    BwdParams bp{static_cast<const uint8_t *>(a.q8), static_cast<const uint8_t *>(a.k8), a.q_scale, a.w, a.k_scale,
                 qb, wq, kinf, a.q_pos, ig, (int64_t)a.S, a.T, a.S, a.HI, a.dw, a.dq, a.dk, status};
    const int nrt = (nq + 127) / 128, nkt = (a.S + 127) / 128;
    e = launch_pdl(bwd_tc_kernel<false>, dim3(static_cast<unsigned>(nrt)), dim3(kGThreads), kGSmem, stream, 1, tq, tk,
                   bp);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "warm-up rows launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    e = cudaMemsetAsync(a.dk, 0, static_cast<size_t>(a.S) * 128 * 4, stream);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "zeroing dk: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    const dim3 grid(static_cast<unsigned>(nkt), static_cast<unsigned>((nrt + kGRowChunk - 1) / kGRowChunk));
    e = launch_pdl(bwd_tc_kernel<true>, grid, dim3(kGThreads), kGSmem, stream, 1, tk, tq, bp);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "warm-up keys launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

} // namespace

size_t warmup_workspace_bytes(int T, int S, int HI) { return wlayout(T, S, HI).total; }

int launch_warmup(const WarmupArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    const WLayout l = wlayout(a.T, a.S, a.HI);
    if (!a.workspace || a.workspace_bytes < l.total) {
        snprintf(err, errlen, "workspace too small for the warm-up path (%zu bytes needed)", l.total);
        return DSA_ERR_WORKSPACE;
    }
    unsigned *status = device_status_ptr();
    if (!status) {
        snprintf(err, errlen, "device status word unavailable");
        return DSA_ERR_CUDA;
    }
    char *ws = static_cast<char *>(a.workspace);
    float *pt = reinterpret_cast<float *>(ws + l.p);
    float *ig = reinterpret_cast<float *>(ws + l.ig);

    // 1. target p
    static std::atomic<bool> target_attr[64];
    if (cudaError_t e = raise_smem_limit_once(attn_target_kernel, kTSmem, target_attr); e != cudaSuccess) {
        snprintf(err, errlen, "cudaFuncSetAttribute(warm-up target): %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    CUtensorMap tq, tkv;
    if (!encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kTD, (uint64_t)a.T * a.H, kTD * 2, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B, err, errlen) ||
        !encode_tmap_2d(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.kv, kTD, (uint64_t)a.S, kTD * 2, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B, err, errlen))
        return DSA_ERR_CUDA;
    TargetParams tp{a.q_pos, a.T, a.S, a.H, a.sm_scale * 1.4426950408889634f, pt, (int64_t)a.S, status};
    cudaError_t e = launch_pdl(attn_target_kernel, dim3(a.T), dim3(kTThreads), kTSmem, stream, 1, tq, tkv, tp);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "warm-up target launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    // 2. index scores
    IndexerArgs ia{a.q8, a.q_scale, a.w, a.T, a.HI, a.dI, a.k8, a.k_scale, a.S, nullptr, 0, 0, 0, a.q_pos, ig, a.S};
    int rc = launch_indexer(ia, stream, err, errlen);
    if (rc != DSA_OK)
        return rc;
    // 3. loss and g
    const int grid = a.T < 8 * num_sms() ? a.T : 8 * num_sms();
    e = launch_pdl(kl_grad_kernel, dim3(grid), dim3(256), 0, stream, 1, ig, static_cast<const float *>(pt),
                   (int64_t)a.S, a.q_pos, a.T, a.S, a.loss);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "warm-up loss launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    // 4. gradients
    return launch_backward(a, l, ws, ig, status, stream, err, errlen);
}

} // namespace dsa
