// Sparse MLA in MQA mode on sm_103a: gather the selected latent rows, QK^T and
// PV on tcgen05 BF16 tensor cores, online softmax with LSE.
//
// Defines (release summary "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency
// with DeepSeek Sparse Attention", section "Method"): the main attention of a
// query token reads only its top-k selected entries, in MLA's MQA mode, so one
// 576-wide latent row (512 + 64 RoPE columns) serves as the key of every query
// head and its first 512 columns serve as the value:
//     S[h,i] = sm_scale * <Q[t,h,:576], KV[s_i,:576]>
//     O[t,h] = sum_i softmax_i(S[h,:]) * KV[s_i,:512],  LSE[t,h] = ln sum_i exp S[h,i]
//
// On-chip budget.  O for 128 heads x 512 columns in fp32 is 256 KB: all of one
// SM's TMEM.  Each token therefore runs on a cluster of two CTAs (two SMs):
//   CTA r keeps O[:, 256r : 256r+256) in TMEM and gathers latent columns
//   [256r, 256r+320) of every selected row (five 64-column swizzle atoms);
//   it computes the PARTIAL scores over latent columns [288r, 288r+288) (K-split
//   of QK^T, no duplicated MMA work), the two CTAs swap their 128 x 64 fp32
//   partial-score tiles through distributed shared memory, and each adds the
//   other's half.  Both then hold the same full scores, run the same softmax
//   (so both see identical P, m and l), and apply P to their own V half.
//
// Per 64-key block j (double-buffered S, P and KV stage):
//   producer warp   cp.async gather of 64 rows x 640 B into the SW128 layout,
//                   zero-filling invalid entries, then publish the stage;
//   MMA warp        S_j = Q_half . KV_j^T   (M=128 heads, N=64, K=288; A and B
//                   K-major in smem) issued one block ahead of
//                   O += P_j . V_j          (M=128, N=256, K=64; A = P from
//                   TMEM, B = the same KV stage read MN-major);
//   softmax warps   thread = head: partial S from TMEM, DSMEM swap, mask, max,
//                   exp2, running sum; P (bf16) back into TMEM.  The running
//                   max is only moved when a block exceeds it by more than
//                   2^8 (then O is rescaled in TMEM), so P stays <= 256.
// At the end the softmax warps normalise O by 1/l, round to bf16 and store it;
// CTA 0 stores the LSE.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kBN = 64;        // keys per block
constexpr int kAtoms = 5;      // 64-column atoms gathered per CTA
constexpr int kRowBytes = kAtoms * 128;
constexpr int kQAtom = 128 * 128;       // bytes of one Q atom (128 rows)
constexpr int kKVAtom = kBN * 128;      // bytes of one KV atom (64 rows)
constexpr int kStage = kAtoms * kKVAtom; // 40 KB
constexpr int kNStage = 2;
constexpr int kXStride = 68;           // floats per row of the swap buffer (pad: no bank conflicts)
constexpr int kThreads = 192;          // producer, MMA, 4 softmax warps
constexpr float kRescaleLog2 = 8.f;    // move the running max only when exceeded by this

constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + kAtoms * kQAtom;          // 80 KB
constexpr int OFF_X = OFF_KV + kNStage * kStage;         // 160 KB
constexpr int OFF_BAR = OFF_X + 128 * kXStride * 4;      // + 34 KB
constexpr int NBAR = 2 * kNStage + 2 + 2 + 2 + 2 + 2;    // kv f/e, s f/e, p f/e, x f/e, q, done
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int kSmem = OFF_MISC + 64 + 1024;

// TMEM columns
constexpr uint32_t TM_O = 0;
constexpr uint32_t TM_S = 256;  // two buffers of 64
constexpr uint32_t TM_P = 384;  // two buffers of 32 (bf16 pairs)
constexpr uint32_t kTmemCols = 512;

struct Params {
    const __nv_bfloat16 *kv;   // [S, 576] or pool [num_pages * page_size, 576]
    const int32_t *idx;        // [T, k]
    int S, T, H, k;
    float scale_log2;          // sm_scale * log2(e)
    __nv_bfloat16 *out;        // [T, H, 512]
    float *lse;                // [T, H]
    const int32_t *block_table;
    int max_pages, num_pages, page_size;
    const int32_t *ctx_len;
    unsigned *status;
};

// Latent row of a selected entry, or -1 if the entry is to be skipped.
template <bool PAGED>
__device__ __forceinline__ int64_t latent_row(const Params &p, int t, int32_t s, int ctx)
{
    if (!PAGED)
        return (s >= 0 && s < p.S) ? (int64_t)s : -1;
    if (s < 0 || s >= ctx)
        return -1;
    const int lp = s / p.page_size;
    if (lp >= p.max_pages)
        return -1;
    const int page = p.block_table[(int64_t)t * p.max_pages + lp];
    if (page < 0 || page >= p.num_pages)
        return -2; // flagged by the caller
    return (int64_t)page * p.page_size + s % p.page_size;
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q, Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    auto kvf_bar = [&](int s) { return bar0 + 8u * s; };
    auto kve_bar = [&](int s) { return bar0 + 8u * (kNStage + s); };
    auto sf_bar = [&](int b) { return bar0 + 8u * (2 * kNStage + b); };
    auto se_bar = [&](int b) { return bar0 + 8u * (2 * kNStage + 2 + b); };
    auto pf_bar = [&](int b) { return bar0 + 8u * (2 * kNStage + 4 + b); };
    auto pe_bar = [&](int b) { return bar0 + 8u * (2 * kNStage + 6 + b); };
    const uint32_t xf_bar = bar0 + 8u * (2 * kNStage + 8);
    const uint32_t xe_bar = bar0 + 8u * (2 * kNStage + 9);
    const uint32_t q_bar = bar0 + 8u * (2 * kNStage + 10);
    const uint32_t done_bar = bar0 + 8u * (2 * kNStage + 11);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    int *nblk_s = reinterpret_cast<int *>(smem + OFF_MISC + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int t = blockIdx.x >> 1;
    const int ctx = PAGED ? p.ctx_len[t] : 0;
    const int32_t *idx_row = p.idx + (int64_t)t * p.k;

    // ---- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < kNStage; ++s) {
            mbar_init(kvf_bar(s), 32);
            mbar_init(kve_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sf_bar(b), 1);
            mbar_init(se_bar(b), 128);
            mbar_init(pf_bar(b), 128);
            mbar_init(pe_bar(b), 1);
        }
        mbar_init(xf_bar, 128);
        mbar_init(xe_bar, 128);
        mbar_init(q_bar, 1);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        *nblk_s = 0;
        fence_mbar_init();
    }
    // Q rows >= H stay zero (their scores are computed but never stored).
    if (p.H < 128) {
        for (int i = threadIdx.x; i < kAtoms * (128 - p.H) * 8; i += kThreads) {
            const int a = i / ((128 - p.H) * 8), rem = i % ((128 - p.H) * 8);
            const int row = p.H + rem / 8, c = rem % 8;
            *reinterpret_cast<uint4 *>(smem + OFF_Q + a * kQAtom + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    // number of 64-key blocks up to the last valid entry (same in both CTAs)
    {
        int last = -1;
        for (int i = threadIdx.x; i < p.k; i += kThreads) {
            const int64_t row = latent_row<PAGED>(p, t, idx_row[i], ctx);
            if (row >= 0)
                last = i;
        }
        for (int o = 16; o > 0; o >>= 1) {
            const int y = __shfl_xor_sync(0xffffffffu, last, o);
            last = y > last ? y : last;
        }
        if (lane == 0 && last >= 0)
            atomicMax(nblk_s, last / kBN + 1);
    }
    if (warp == 1)
        tmem_alloc(sbase + OFF_MISC, kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all(); // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int nb = *nblk_s;

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0 && nb > 0) {
            tma_prefetch_desc(&tm_q);
            mbar_arrive_expect_tx(q_bar, kAtoms * p.H * 128);
            for (int a = 0; a < kAtoms; ++a)
                tma_load_2d(sbase + OFF_Q + a * kQAtom, &tm_q, q_bar, (int)(256 * rank) + 64 * a, t * p.H);
        }
        const __nv_bfloat16 *kv_cols = p.kv + 256 * rank;
        for (int j = 0; j < nb; ++j) {
            const int st = j % kNStage;
            if (j >= kNStage && !mbar_wait_warp(kve_bar(st), ((j / kNStage) - 1) & 1, abort_flag, p.status))
                break;
            // rows of this block: lane l resolves entries l and l + 32
            int64_t r_lo, r_hi;
            {
                const int i0 = j * kBN + lane, i1 = i0 + 32;
                r_lo = i0 < p.k ? latent_row<PAGED>(p, t, idx_row[i0], ctx) : -1;
                r_hi = i1 < p.k ? latent_row<PAGED>(p, t, idx_row[i1], ctx) : -1;
                if (PAGED && (r_lo == -2 || r_hi == -2))
                    atomicOr(p.status, DSA_DEV_BAD_PAGE);
            }
            const uint32_t stage = sbase + OFF_KV + st * kStage;
#pragma unroll 4
            for (int c = lane; c < kBN * kAtoms * 8; c += 32) {
                const int i = c / (kAtoms * 8);
                const int q = c % (kAtoms * 8);
                const int a = q >> 3, cc = q & 7;
                const int64_t rlo = __shfl_sync(0xffffffffu, r_lo, i & 31);
                const int64_t rhi = __shfl_sync(0xffffffffu, r_hi, i & 31);
                const int64_t row = i < 32 ? rlo : rhi;
                const uint32_t dst = stage + a * kKVAtom + i * 128 + ((cc ^ (i & 7)) << 4);
                const __nv_bfloat16 *src = row >= 0 ? kv_cols + row * kD + a * 64 + cc * 8 : p.kv;
                const uint32_t bytes = row >= 0 ? 16u : 0u; // 0: zero-fill, nothing read
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
                             : "memory");
            }
            cp_async_commit();
            cp_async_wait_group<0>();
            fence_proxy_async_smem();
            mbar_arrive(kvf_bar(st));
        }
        cp_async_wait_group<0>();
        if (lane == 0 && nb > 0)
            mbar_drain(q_bar, 0);
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc_qk = idesc_f32acc(128, kBN, 1u, false, false);
        constexpr uint32_t idesc_pv = idesc_f32acc(128, 256, 1u, false, true);
        const int ks0 = 2 * (int)rank; // first 16-column k-step of this CTA's score half
        bool ok = nb > 0 && mbar_wait_warp(q_bar, 0, abort_flag, p.status);
        auto issue_qk = [&](int j) -> bool {
            const int st = j % kNStage, b = j & 1;
            if (!mbar_wait_warp(kvf_bar(st), (j / kNStage) & 1, abort_flag, p.status))
                return false;
            if (j >= 2 && !mbar_wait_warp(se_bar(b), ((j - 2) >> 1) & 1, abort_flag, p.status))
                return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t stage = sbase + OFF_KV + st * kStage;
#pragma unroll
                for (int kk = 0; kk < 18; ++kk) {
                    const int ks = ks0 + kk, a = ks >> 2, w = ks & 3;
                    const uint64_t ad = sdesc(sbase + OFF_Q + a * kQAtom + w * 32, 16, 1024, 2);
                    const uint64_t bd = sdesc(stage + a * kKVAtom + w * 32, 16, 1024, 2);
                    umma_f16_ss(tmem + TM_S + 64 * b, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                }
                umma_commit(sf_bar(b));
            }
            __syncwarp();
            return true;
        };
        if (ok)
            ok = issue_qk(0);
        for (int j = 0; ok && j < nb; ++j) {
            if (j + 1 < nb && !issue_qk(j + 1)) {
                ok = false;
                break;
            }
            const int b = j & 1, st = j % kNStage;
            if (!mbar_wait_warp(pf_bar(b), (j >> 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t stage = sbase + OFF_KV + st * kStage;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t bd = sdesc(stage + kk * 16 * 128, kKVAtom, 1024, 2);
                    umma_f16_ts(tmem + TM_O, tmem + TM_P + 32 * b + 8 * kk, bd, idesc_pv,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(pe_bar(b));
                umma_commit(kve_bar(st));
            }
            __syncwarp();
        }
        if (lane == 0) {
            umma_commit(done_bar);
            mbar_drain(done_bar, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax + epilogue
        const int quad = warp & 3;
        const int h = quad * 32 + lane;                  // head = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        float *xrow = reinterpret_cast<float *>(smem + OFF_X) + h * kXStride;
        const uint32_t x_remote = mapa_shared(smem_u32(xrow), peer);
        const uint32_t xf_remote = mapa_shared(xf_bar, peer);
        const uint32_t xe_remote = mapa_shared(xe_bar, peer);
        float m_run = -INFINITY; // running max, log2 domain
        float l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            const int b = j & 1;
            // validity of the 64 entries of this block
            uint32_t vm_lo, vm_hi;
            {
                const int i0 = j * kBN + lane, i1 = i0 + 32;
                const bool v0 = i0 < p.k && latent_row<PAGED>(p, t, idx_row[i0], ctx) >= 0;
                const bool v1 = i1 < p.k && latent_row<PAGED>(p, t, idx_row[i1], ctx) >= 0;
                vm_lo = __ballot_sync(0xffffffffu, v0);
                vm_hi = __ballot_sync(0xffffffffu, v1);
            }
            // 1. partial scores of this CTA
            if (!mbar_wait_warp(sf_bar(b), (j >> 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float sc[kBN];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_off + TM_S + 64 * b, r0);
                tmem_ld32(tmem + lane_off + TM_S + 64 * b + 32, r1);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    sc[c] = __uint_as_float(r0[c]);
                    sc[c + 32] = __uint_as_float(r1[c]);
                }
            }
            tc_fence_before();
            mbar_arrive(se_bar(b));
            // 2. swap partial scores with the peer CTA
            if (j >= 1 && !mbar_wait<true>(xe_bar, (j - 1) & 1, abort_flag, p.status)) {
                ok = false;
            }
            if (!__all_sync(0xffffffffu, ok))
                break;
#pragma unroll
            for (int c = 0; c < kBN; c += 4)
                st_cluster_v4(x_remote + c * 4, sc[c], sc[c + 1], sc[c + 2], sc[c + 3]);
            mbar_arrive_remote(xf_remote);
            if (!mbar_wait_warp<true>(xf_bar, j & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int c = 0; c < kBN; c += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(xrow + c);
                sc[c] += x.x;
                sc[c + 1] += x.y;
                sc[c + 2] += x.z;
                sc[c + 3] += x.w;
            }
            mbar_arrive_remote(xe_remote);
            // 3. mask, block max (log2 domain)
            float bmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                const bool v = ((c < 32 ? vm_lo : vm_hi) >> (c & 31)) & 1u;
                sc[c] = v ? sc[c] * p.scale_log2 : -INFINITY;
                bmax = fmaxf(bmax, sc[c]);
            }
            // 4. move the running max only when it is exceeded by more than 2^8
            //    (per head; the TMEM rescale below is warp-collective)
            float alpha = 1.f;
            bool scale_o = false;
            if (bmax > m_run + kRescaleLog2) {
                if (m_run != -INFINITY) {
                    alpha = fast_exp2(m_run - bmax);
                    scale_o = true;
                }
                m_run = bmax;
            }
            l_run *= alpha;
            if (__any_sync(0xffffffffu, scale_o)) {
                // O holds blocks < j (j >= 1 here): wait for PV_{j-1}, then scale the rows
                if (!mbar_wait(pe_bar((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag, p.status))
                    ok = false;
                if (!__all_sync(0xffffffffu, ok))
                    break;
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_off + TM_O + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
                    tmem_st32(tmem + lane_off + TM_O + c0, r);
                }
                tmem_st_wait();
            }
            const float m_use = m_run == -INFINITY ? 0.f : m_run;
            // 5. P = exp2(S - m), running sum, bf16 pairs into TMEM
            uint32_t pk[32];
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
                const float p0 = fast_exp2(sc[c] - m_use);
                const float p1 = fast_exp2(sc[c + 1] - m_use);
                lsum += p0 + p1;
                pk[c >> 1] = pack_bf16x2(p0, p1);
            }
            l_run += lsum;
            if (j >= 2 && !mbar_wait(pe_bar(b), ((j - 2) >> 1) & 1, abort_flag, p.status))
                ok = false;
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after();
            tmem_st32(tmem + lane_off + TM_P + 32 * b, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(pf_bar(b));
        }
        // ---- epilogue: O / l -> bf16, LSE
        if (ok && nb > 0) {
            ok = mbar_wait_warp(pe_bar((nb - 1) & 1), ((nb - 1) >> 1) & 1, abort_flag, p.status);
        }
        const bool store = h < p.H;
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        __nv_bfloat16 *orow = p.out + ((int64_t)t * p.H + h) * kDv + 256 * rank;
        if (ok && nb > 0) {
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < 256; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + TM_O + c0, r);
                tmem_ld_wait();
                uint32_t o[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    o[c] = pack_bf16x2(__uint_as_float(r[2 * c]) * inv_l, __uint_as_float(r[2 * c + 1]) * inv_l);
                if (store) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                }
            }
        } else if (ok && store) {
            // nothing valid: O = 0
            uint4 *dst = reinterpret_cast<uint4 *>(orow);
            for (int c = 0; c < 256 / 8; ++c)
                dst[c] = make_uint4(0, 0, 0, 0);
        }
        if (ok && store && rank == 0)
            p.lse[(int64_t)t * p.H + h] = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all(); // no CTA leaves while its peer may still touch its smem
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool PAGED>
int launch(const MlaArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel<PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmem);
        if (e != cudaSuccess) {
            snprintf(err, errlen, "cudaFuncSetAttribute(sparse_mla): %s", cudaGetErrorString(e));
            return DSA_ERR_CUDA;
        }
        attr_set[dev] = true;
    }
    CUtensorMap tq;
    if (!encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kD, (uint64_t)a.T * a.H, kD * 2, 64, a.H,
                        CU_TENSOR_MAP_SWIZZLE_128B, err, errlen))
        return DSA_ERR_CUDA;
    Params p;
    p.kv = static_cast<const __nv_bfloat16 *>(a.kv);
    p.idx = a.idx;
    p.S = a.S;
    p.T = a.T;
    p.H = a.H;
    p.k = a.k;
    p.scale_log2 = a.sm_scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    p.block_table = a.block_table;
    p.max_pages = a.max_pages;
    p.num_pages = a.num_pages;
    p.page_size = a.page_size;
    p.ctx_len = a.ctx_len;
    p.status = device_status_ptr();
    if (!p.status) {
        snprintf(err, errlen, "device status word unavailable");
        return DSA_ERR_CUDA;
    }
    if ((int64_t)a.T * 2 > (int64_t)INT32_MAX) {
        snprintf(err, errlen, "sparse_mla: T too large");
        return DSA_ERR_UNSUPPORTED;
    }
    sparse_mla_kernel<PAGED><<<dim3(2 * a.T), kThreads, kSmem, stream>>>(tq, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, errlen, "sparse_mla launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

} // namespace

int launch_mla_prefill(const MlaArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    return launch<false>(a, stream, err, errlen);
}

int launch_mla_decode(const MlaArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    return launch<true>(a, stream, err, errlen);
}

size_t mla_decode_workspace_bytes(int, int, int) { return 0; }

} // namespace dsa
