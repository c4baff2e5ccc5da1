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
//   bwd_rows_kernel     one CTA per query row, FP32 on the CUDA cores, 64-key
//                       tiles in shared memory: a, dw, dq, and the coefficients
//                       c[t,j,s] = g w [a > 0] for dk.
//   bwd_keys_kernel     one CTA per (64-key tile, 256-row chunk): dk from c and
//                       q, added to dk with atomics (dk is zeroed first).
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
constexpr int kTOffBar = kTOffLse + 128 * 4;
constexpr int kTNBar = 2 * kTStages + 4 + 2;
constexpr int kTOffMisc = kTOffBar + kTNBar * 8;
constexpr int kTSmem = kTOffMisc + 64 + 1024;
constexpr int kTThreads = 6 * 32;              // producer, MMA, four epilogue warps
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
            mbar_init(acce_bar(a), 4);
        }
        mbar_init(q_bar, 1);
        mbar_init(done_bar, 1);
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
        const int quad = warp & 3;
        const int row = quad * 32 + lane; // pass 0: head; pass 1: key within the tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        float m = -INFINITY, l = 0.f;
        for (int it = 0; it < items; ++it) {
            const int a = it & 1, use = it >> 1;
            const bool pass1 = it >= ntiles;
            const int kt = it % ntiles;
            if (it == ntiles) {
                // pass 0 done: every head's LSE (log2 units) into shared memory
                lse2[row] = l > 0.f ? m + __log2f(l) : INFINITY;
                named_bar_sync(1, 128);
            }
            if (!mbar_wait_warp(accf_bar(a), use & 1, abort_flag, p.status))
                break;
            tc_fence_after();
            float bsum = 0.f; // pass 1: this key's sum over the heads
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_base + 128 * a + c0, r);
                tmem_ld_wait();
                if (c0 == 96) {
                    // every column of the accumulator is in registers: release it
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
                if (s <= pos)
                    p.p[(int64_t)t * p.ld + s] = bsum / static_cast<float>(p.H);
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

// ---------------------------------------------------------- backward: rows
// One CTA of 256 threads per query row t.  Per 64-key tile: the tile's
// dequantised keys kd[64][128] and g; a[j][s] for the 64 heads x 64 keys
// (thread: 4 heads x keys sg, sg + 16, sg + 32, sg + 48, float4 loads along d);
// dw partials; c = g w [a>0] into shared memory and to the global c[t][j][s];
// then dq[j][d] += sum_s c[j][s] kd[s][d] (thread: 4 heads x columns
// 4 dd .. +4 and 64 + 4 dd .. +4).  Neighbouring threads read neighbouring key
// rows and neighbouring column groups: with keys 4 rows apart (4 x 132 floats
// = 16 banks) sixteen threads' rows fell on two bank groups, and 8-column
// groups on four, and the kernel ran at the shared-memory pipe's limit.
constexpr int kBTile = 64;
constexpr int kBD = 128;
constexpr int kBKdPitch = kBD + 4;   // floats per key row in shared memory (16-byte aligned, banks spread)
constexpr int kBCPitch = kBTile + 4; // floats per head row of c

template <int HI>
__global__ void __launch_bounds__(256)
    bwd_rows_kernel(const uint8_t *__restrict__ q8, const float *__restrict__ q_scale, const float *__restrict__ w,
                    const uint8_t *__restrict__ k8, const float *__restrict__ k_scale, const int32_t *__restrict__ q_pos,
                    int T, int S, const float *__restrict__ g, int64_t ldg, float *__restrict__ cbuf, int64_t ldc,
                    float *__restrict__ dw, float *__restrict__ dq)
{
    static_assert(HI == 64 || HI == 32, "heads");
    constexpr int JT = HI / 16; // heads per thread in the a phase (16 head groups)
    extern __shared__ __align__(16) float bsm[];
    float *qd = bsm;                             // [HI][kBD]
    float *kd = qd + HI * kBD;                   // [kBTile][kBKdPitch]
    float *cs = kd + kBTile * kBKdPitch;         // [HI][kBCPitch]
    float *gt = cs + HI * kBCPitch;              // [kBTile]
    float *dws = gt + kBTile;                    // [HI]
    grid_dep_wait();
    grid_dep_launch();
    const int t = gridDim.x - 1 - blockIdx.x;
    int64_t qp = q_pos[t];
    qp = qp > S - 1 ? S - 1 : qp;
    const int pos = qp < 0 ? -1 : static_cast<int>(qp);
    const float qs = q_scale[t];
    for (int i = threadIdx.x; i < HI * kBD; i += 256)
        qd[i] = e4m3_to_float(q8[(int64_t)t * HI * kBD + i]) * qs;
    for (int i = threadIdx.x; i < HI; i += 256)
        dws[i] = 0.f;
    // a phase: thread (jg, sg) = heads jg * JT .. +JT, keys sg + 16 e (e < 4)
    const int jg = threadIdx.x >> 4, sg = threadIdx.x & 15;
    // dq phase: thread (jd, dd) = heads jd * JD .. +JD, columns 4 dd .. +4 and 64 + 4 dd .. +4
    constexpr int JD = HI / 16;
    const int jd = threadIdx.x >> 4, dd = threadIdx.x & 15;
    float acc_dq[JD][8];
#pragma unroll
    for (int i = 0; i < JD; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc_dq[i][e] = 0.f;
    float acc_dw[JT];
#pragma unroll
    for (int i = 0; i < JT; ++i)
        acc_dw[i] = 0.f;
    float wj[JT];
#pragma unroll
    for (int i = 0; i < JT; ++i)
        wj[i] = w[(int64_t)t * HI + jg * JT + i];
    const int ntiles = pos < 0 ? 0 : pos / kBTile + 1;
    for (int kt = 0; kt < ntiles; ++kt) {
        const int s0 = kt * kBTile;
        __syncthreads(); // previous tile's kd, cs, gt fully used
        for (int i = threadIdx.x; i < kBTile * kBD; i += 256) {
            const int s = i / kBD, d = i % kBD;
            const int sk = s0 + s;
            kd[s * kBKdPitch + d] = sk <= pos ? e4m3_to_float(k8[(int64_t)sk * kBD + d]) * k_scale[sk] : 0.f;
        }
        for (int i = threadIdx.x; i < kBTile; i += 256)
            gt[i] = s0 + i <= pos ? g[(int64_t)t * ldg + s0 + i] : 0.f;
        __syncthreads();
        float a[JT][4];
#pragma unroll
        for (int i = 0; i < JT; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                a[i][e] = 0.f;
#pragma unroll 4
        for (int d = 0; d < kBD; d += 4) {
            float4 qv[JT], kv[4];
#pragma unroll
            for (int i = 0; i < JT; ++i)
                qv[i] = *reinterpret_cast<const float4 *>(qd + (jg * JT + i) * kBD + d);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                kv[e] = *reinterpret_cast<const float4 *>(kd + (sg + 16 * e) * kBKdPitch + d);
#pragma unroll
            for (int i = 0; i < JT; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    a[i][e] = fmaf(qv[i].x, kv[e].x,
                                   fmaf(qv[i].y, kv[e].y, fmaf(qv[i].z, kv[e].z, fmaf(qv[i].w, kv[e].w, a[i][e]))));
        }
#pragma unroll
        for (int i = 0; i < JT; ++i) {
            const int j = jg * JT + i;
            float *crow = cbuf + ((int64_t)t * HI + j) * ldc + s0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int sl = sg + 16 * e;
                const float ge = gt[sl];
                acc_dw[i] += a[i][e] > 0.f ? ge * a[i][e] : 0.f;
                const float c = a[i][e] > 0.f ? ge * wj[i] : 0.f;
                cs[j * kBCPitch + sl] = c;
                if (s0 + sl < S)
                    crow[sl] = c; // sixteen threads: 64 contiguous bytes
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int s = 0; s < kBTile; ++s) {
            const float4 k0 = *reinterpret_cast<const float4 *>(kd + s * kBKdPitch + dd * 4);
            const float4 k1 = *reinterpret_cast<const float4 *>(kd + s * kBKdPitch + 64 + dd * 4);
#pragma unroll
            for (int i = 0; i < JD; ++i) {
                const float c = cs[(jd * JD + i) * kBCPitch + s];
                acc_dq[i][0] = fmaf(c, k0.x, acc_dq[i][0]);
                acc_dq[i][1] = fmaf(c, k0.y, acc_dq[i][1]);
                acc_dq[i][2] = fmaf(c, k0.z, acc_dq[i][2]);
                acc_dq[i][3] = fmaf(c, k0.w, acc_dq[i][3]);
                acc_dq[i][4] = fmaf(c, k1.x, acc_dq[i][4]);
                acc_dq[i][5] = fmaf(c, k1.y, acc_dq[i][5]);
                acc_dq[i][6] = fmaf(c, k1.z, acc_dq[i][6]);
                acc_dq[i][7] = fmaf(c, k1.w, acc_dq[i][7]);
            }
        }
    }
    // dw: the 16 key groups of a head group meet in shared memory
#pragma unroll
    for (int i = 0; i < JT; ++i)
        atomicAdd(&dws[jg * JT + i], acc_dw[i]);
    __syncthreads();
    for (int i = threadIdx.x; i < HI; i += 256)
        dw[(int64_t)t * HI + i] = dws[i];
#pragma unroll
    for (int i = 0; i < JD; ++i) {
        float *dst = dq + ((int64_t)t * HI + jd * JD + i) * kBD + dd * 4;
        *reinterpret_cast<float4 *>(dst) = make_float4(acc_dq[i][0], acc_dq[i][1], acc_dq[i][2], acc_dq[i][3]);
        *reinterpret_cast<float4 *>(dst + 64) = make_float4(acc_dq[i][4], acc_dq[i][5], acc_dq[i][6], acc_dq[i][7]);
    }
}

template <int HI>
size_t bwd_rows_smem()
{
    return (static_cast<size_t>(HI) * kBD + kBTile * kBKdPitch + HI * kBCPitch + kBTile + HI) * 4;
}

// ---------------------------------------------------------- backward: keys
// One CTA of 256 threads per (64-key tile kt, chunk of 256 query rows): for
// each row t of the chunk that sees the tile, dk[s][d] += sum_j c[t][j][s]
// q[t][j][d] (thread: 4 keys x columns 4 dd .. +4 and 64 + 4 dd .. +4, so the
// sixteen column groups of a row are 256 contiguous bytes); the partial sums
// are added to dk with atomics.
constexpr int kBRowChunk = 256;

template <int HI>
__global__ void __launch_bounds__(256)
    bwd_keys_kernel(const uint8_t *__restrict__ q8, const float *__restrict__ q_scale,
                    const int32_t *__restrict__ q_pos, int T, int S, const float *__restrict__ cbuf, int64_t ldc,
                    float *__restrict__ dk)
{
    extern __shared__ __align__(16) float ksm[];
    float *qd = ksm;                        // [HI][kBD]
    float *ct = qd + HI * kBD;              // [HI][kBCPitch]: c[t][j][s0 .. s0 + 64)
    grid_dep_wait();
    grid_dep_launch();
    const int s0 = blockIdx.x * kBTile;
    const int t0 = blockIdx.y * kBRowChunk;
    const int t1 = t0 + kBRowChunk < T ? t0 + kBRowChunk : T;
    const int sg = threadIdx.x >> 4, dd = threadIdx.x & 15; // keys sg * 4 .. +4, columns 4 dd .. +4, 64 + 4 dd .. +4
    float acc[4][8];
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int c = 0; c < 8; ++c)
            acc[e][c] = 0.f;
    bool any = false;
    for (int t = t0; t < t1; ++t) {
        int64_t qp = q_pos[t];
        qp = qp > S - 1 ? S - 1 : qp;
        if (qp < s0)
            continue; // uniform: this row sees none of the tile
        any = true;
        const int nvalid = static_cast<int>(qp - s0 + 1 < kBTile ? qp - s0 + 1 : kBTile);
        __syncthreads();
        const float qs = q_scale[t];
        for (int i = threadIdx.x; i < HI * kBD; i += 256)
            qd[i] = e4m3_to_float(q8[(int64_t)t * HI * kBD + i]) * qs;
        for (int i = threadIdx.x; i < HI * kBTile; i += 256) {
            const int j = i / kBTile, s = i % kBTile;
            ct[j * kBCPitch + s] = s < nvalid ? cbuf[((int64_t)t * HI + j) * ldc + s0 + s] : 0.f;
        }
        __syncthreads();
#pragma unroll 2
        for (int j = 0; j < HI; ++j) {
            const float4 q0 = *reinterpret_cast<const float4 *>(qd + j * kBD + dd * 4);
            const float4 q1 = *reinterpret_cast<const float4 *>(qd + j * kBD + 64 + dd * 4);
            const float4 cv = *reinterpret_cast<const float4 *>(ct + j * kBCPitch + sg * 4);
            const float cc[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[e][0] = fmaf(cc[e], q0.x, acc[e][0]);
                acc[e][1] = fmaf(cc[e], q0.y, acc[e][1]);
                acc[e][2] = fmaf(cc[e], q0.z, acc[e][2]);
                acc[e][3] = fmaf(cc[e], q0.w, acc[e][3]);
                acc[e][4] = fmaf(cc[e], q1.x, acc[e][4]);
                acc[e][5] = fmaf(cc[e], q1.y, acc[e][5]);
                acc[e][6] = fmaf(cc[e], q1.z, acc[e][6]);
                acc[e][7] = fmaf(cc[e], q1.w, acc[e][7]);
            }
        }
    }
    if (!any)
        return;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int s = s0 + sg * 4 + e;
        if (s < S)
#pragma unroll
            for (int c = 0; c < 8; ++c)
                atomicAdd(dk + (int64_t)s * kBD + (c < 4 ? dd * 4 + c : 64 + dd * 4 + c - 4), acc[e][c]);
    }
}

template <int HI>
size_t bwd_keys_smem()
{
    return (static_cast<size_t>(HI) * kBD + HI * kBCPitch) * 4;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WLayout {
    size_t p, ig, c, total;
    int64_t ldc; // row pitch of c, a multiple of 4 floats
};

WLayout wlayout(int T, int S, int HI)
{
    WLayout l;
    size_t o = 0;
    l.p = o;
    o += align256(static_cast<size_t>(T) * S * 4);
    l.ig = o;
    o += align256(static_cast<size_t>(T) * S * 4);
    l.ldc = (S + 3) & ~3;
    l.c = o;
    o += align256(static_cast<size_t>(T) * HI * l.ldc * 4);
    l.total = o;
    return l;
}

template <int HI>
int launch_backward(const WarmupArgs &a, float *ig, float *cbuf, int64_t ldc, cudaStream_t stream, char *err,
                    size_t errlen)
{
    static std::atomic<bool> rows_attr[64], keys_attr[64];
    if (cudaError_t e = raise_smem_limit_once(bwd_rows_kernel<HI>, static_cast<int>(bwd_rows_smem<HI>()), rows_attr);
        e != cudaSuccess) {
        snprintf(err, errlen, "cudaFuncSetAttribute(warm-up rows): %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    if (cudaError_t e = raise_smem_limit_once(bwd_keys_kernel<HI>, static_cast<int>(bwd_keys_smem<HI>()), keys_attr);
        e != cudaSuccess) {
        snprintf(err, errlen, "cudaFuncSetAttribute(warm-up keys): %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    cudaError_t e = launch_pdl(bwd_rows_kernel<HI>, dim3(a.T), dim3(256), bwd_rows_smem<HI>(), stream, 1,
                               static_cast<const uint8_t *>(a.q8), a.q_scale, a.w, static_cast<const uint8_t *>(a.k8),
                               a.k_scale, a.q_pos, a.T, a.S, static_cast<const float *>(ig), (int64_t)a.S, cbuf,
                               ldc, a.dw, a.dq);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "warm-up rows launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    e = cudaMemsetAsync(a.dk, 0, static_cast<size_t>(a.S) * kBD * 4, stream);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "zeroing dk: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    dim3 grid((a.S + kBTile - 1) / kBTile, (a.T + kBRowChunk - 1) / kBRowChunk);
    e = launch_pdl(bwd_keys_kernel<HI>, grid, dim3(256), bwd_keys_smem<HI>(), stream, 1,
                   static_cast<const uint8_t *>(a.q8), a.q_scale, a.q_pos, a.T, a.S, static_cast<const float *>(cbuf),
                   ldc, a.dk);
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
    float *cbuf = reinterpret_cast<float *>(ws + l.c);

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
    return a.HI == 64 ? launch_backward<64>(a, ig, cbuf, l.ldc, stream, err, errlen)
                      : launch_backward<32>(a, ig, cbuf, l.ldc, stream, err, errlen);
}

} // namespace dsa
