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
//   producer warp   resolves the 64 selected rows and gathers them with TMA
//                   gather4 (4 rows x 128 B per instruction, 16 lanes x 5 atoms);
//                   an invalid entry re-reads the token's first valid row (an
//                   in-bounds, finite row whose score is masked, so P = 0);
//   MMA warp        S_j = Q_half . KV_j^T   (M=128 heads, N=64, K=288; A and B
//                   K-major in smem) issued one block ahead of
//                   O += P_j . V_j          (M=128, N=256, K=64; A = P from
//                   TMEM, B = the same KV stage read MN-major);
//   softmax warps   thread = head: partial S from TMEM, swap with the peer by
//                   st.async (completion counted in bytes on the peer's
//                   mbarrier), mask, max, exp2, running sum; P (bf16) back into
//                   TMEM.  The running max is only moved when a block exceeds it
//                   by more than 2^8 (then O is rescaled in TMEM), so P <= 256.
// The kernel is persistent: each cluster walks tokens t = c, c + C, ... with
// one barrier/TMEM setup, prefetches the next token's Q into L2, and the
// softmax warps store a token's output (O / l in bf16, LSE from CTA 0) while
// the tensor cores already run the next token's first score tiles.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kBN = 64;        // keys per block
constexpr int kAtoms = 5;      // 64-column atoms gathered per CTA
constexpr int kQAtom = 128 * 128;       // bytes of one Q atom (128 rows)
constexpr int kKVAtom = kBN * 128;      // bytes of one KV atom (64 rows)
constexpr int kStage = kAtoms * kKVAtom; // 40 KB
constexpr int kXStride = 68;           // floats per row of the swap buffer (pad: no bank conflicts)
constexpr int kThreads = 192;          // producer, MMA, 4 softmax warps
constexpr float kRescaleLog2 = 8.f;    // move the running max only when exceeded by this

constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + kAtoms * kQAtom;          // 80 KB
constexpr int OFF_X = OFF_KV + 2 * kStage;               // 160 KB
constexpr int OFF_BAR = OFF_X + 128 * kXStride * 4;      // + 34 KB
constexpr int NBAR = 20;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int kSmem = OFF_MISC + 64 + 1024;

// barrier slots
constexpr int B_KVF = 0, B_KVE = 2, B_SF = 4, B_SE = 6, B_PF = 8, B_PE = 10, B_XF = 12, B_XE = 13, B_QF = 14,
              B_QE = 15, B_OF = 16, B_OE = 17, B_DONE = 18, B_QA = 19;

// TMEM columns
constexpr uint32_t TM_O = 0;
constexpr uint32_t TM_S = 256;  // two buffers of 64
constexpr uint32_t TM_P = 384;  // two buffers of 32 (bf16 pairs)
constexpr uint32_t kTmemCols = 512;

struct Params {
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

// Latent row of a selected entry: >= 0 valid, -1 skipped, -2 bad page (skipped, flagged).
template <bool PAGED>
__device__ __forceinline__ int latent_row(const Params &p, int t, int32_t s, int ctx)
{
    if (!PAGED)
        return (s >= 0 && s < p.S) ? s : -1;
    if (s < 0 || s >= ctx)
        return -1;
    const int lp = s / p.page_size;
    if (lp >= p.max_pages)
        return -1;
    const int page = p.block_table[(int64_t)t * p.max_pages + lp];
    if (page < 0 || page >= p.num_pages)
        return -2;
    return page * p.page_size + s % p.page_size;
}

// Could the entry be valid at all (range check only, used to count blocks)?
template <bool PAGED>
__device__ __forceinline__ bool in_range(const Params &p, int32_t s, int ctx)
{
    return PAGED ? (s >= 0 && s < ctx) : (s >= 0 && s < p.S);
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
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv, Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * i; };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    volatile int *nb_s = reinterpret_cast<volatile int *>(smem + OFF_MISC + 8); // [2]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int cid = blockIdx.x >> 1;
    const int ncl = gridDim.x >> 1;

    // ---- one-time setup
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_KVF + i), 1);
            mbar_init(bar(B_KVE + i), 1);
            mbar_init(bar(B_SF + i), 1);
            mbar_init(bar(B_SE + i), 4);
            mbar_init(bar(B_PF + i), 4);
            mbar_init(bar(B_PE + i), 1);
        }
        mbar_init(bar(B_XF), 1);
        mbar_init(bar(B_XE), 4);
        mbar_init(bar(B_QF), 1);
        mbar_init(bar(B_QE), 1);
        mbar_init(bar(B_OF), 1);
        mbar_init(bar(B_OE), 4);
        mbar_init(bar(B_DONE), 1);
        mbar_init(bar(B_QA), 4);
        *abort_flag = 0;
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
    if (warp == 1)
        tmem_alloc(sbase + OFF_MISC, kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all(); // both CTAs' barriers exist before any remote operation
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------- producer
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_kv);
        uint32_t J = 0;
        int u = 0;
        bool ok = true;
        for (int t = cid; ok && t < p.T; t += ncl, ++u) {
            const int32_t *idx_row = p.idx + (int64_t)t * p.k;
            const int ctx = PAGED ? p.ctx_len[t] : 0;
            // blocks up to the last in-range entry; the first one gives a fallback row
            int last = -1, first = 0x7fffffff;
#pragma unroll 8
            for (int i = lane; i < p.k; i += 32)
                if (in_range<PAGED>(p, idx_row[i], ctx)) {
                    last = i;
                    first = first < i ? first : i;
                }
            for (int o = 16; o > 0; o >>= 1) {
                const int y = __shfl_xor_sync(0xffffffffu, last, o);
                const int z = __shfl_xor_sync(0xffffffffu, first, o);
                last = y > last ? y : last;
                first = z < first ? z : first;
            }
            const int nb = last < 0 ? 0 : last / kBN + 1;
            int fb_row = nb > 0 ? latent_row<PAGED>(p, t, idx_row[first], ctx) : 0;
            if (fb_row < 0)
                fb_row = 0;
            // the Q buffer and the nb slot are reused: the MMA warp must be done
            // reading Q and the softmax warps must have taken the previous token
            if (u >= 1 && (!mbar_wait_warp(bar(B_QE), (u - 1) & 1, abort_flag, p.status) ||
                           !mbar_wait_warp(bar(B_QA), (u - 1) & 1, abort_flag, p.status))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                nb_s[u & 1] = nb;
                if (nb > 0) {
                    mbar_arrive_expect_tx(bar(B_QF), kAtoms * p.H * 128);
                    for (int a = 0; a < kAtoms; ++a)
                        tma_load_2d(sbase + OFF_Q + a * kQAtom, &tm_q, bar(B_QF), (int)(256 * rank) + 64 * a,
                                    t * p.H);
                } else {
                    mbar_arrive(bar(B_QF));
                }
                if (t + ncl < p.T)
                    for (int a = 0; a < kAtoms; ++a)
                        tma_prefetch_l2_2d(&tm_q, (int)(256 * rank) + 64 * a, (t + ncl) * p.H);
            }
            __syncwarp();
            // rows of block 0; each later block's rows are resolved while the
            // stage it will use is still busy
            auto resolve = [&](int j, int &rl, int &rh) {
                const int i0 = j * kBN + lane, i1 = i0 + 32;
                rl = i0 < p.k ? latent_row<PAGED>(p, t, idx_row[i0], ctx) : -1;
                rh = i1 < p.k ? latent_row<PAGED>(p, t, idx_row[i1], ctx) : -1;
                if (PAGED && (rl == -2 || rh == -2))
                    atomicOr(p.status, DSA_DEV_BAD_PAGE);
                if (rl < 0) rl = fb_row; // masked in the softmax
                if (rh < 0) rh = fb_row;
            };
            int r_lo = 0, r_hi = 0;
            if (nb > 0)
                resolve(0, r_lo, r_hi);
            for (int j = 0; j < nb; ++j, ++J) {
                const int st = J & 1;
                int rows[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int src = (4 * lane + e) & 31;
                    const int vlo = __shfl_sync(0xffffffffu, r_lo, src);
                    const int vhi = __shfl_sync(0xffffffffu, r_hi, src);
                    rows[e] = lane < 8 ? vlo : vhi;
                }
                if (j + 1 < nb)
                    resolve(j + 1, r_lo, r_hi);
                if (J >= 2 && !mbar_wait_warp(bar(B_KVE + st), ((J >> 1) - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t stage = sbase + OFF_KV + st * kStage;
                if (lane == 0)
                    mbar_arrive_expect_tx(bar(B_KVF + st), kStage);
                __syncwarp();
                if (lane < 16) {
#pragma unroll
                    for (int a = 0; a < kAtoms; ++a)
                        tma_gather4(stage + a * kKVAtom + lane * 4 * 128, &tm_kv, bar(B_KVF + st),
                                    (int)(256 * rank) + 64 * a, rows[0], rows[1], rows[2], rows[3]);
                }
                __syncwarp();
            }
        }
        // drain: every copy this warp issued has landed before the CTA exits
        if (lane == 0) {
            for (uint32_t i = J >= 2 ? J - 2 : 0; i < J; ++i)
                mbar_drain(bar(B_KVF + (i & 1)), (i >> 1) & 1);
            if (u >= 1)
                mbar_drain(bar(B_QF), (u - 1) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc_qk = idesc_f32acc(128, kBN, 1u, false, false);
        constexpr uint32_t idesc_pv = idesc_f32acc(128, 256, 1u, false, true);
        const int ks0 = 2 * (int)rank; // first 16-column k-step of this CTA's score half
        uint32_t J = 0;
        int u = 0, v = 0;
        bool ok = true;
        auto issue_qk = [&](uint32_t Jq) -> bool {
            const int st = Jq & 1, b = Jq & 1;
            if (!mbar_wait_warp(bar(B_KVF + st), (Jq >> 1) & 1, abort_flag, p.status))
                return false;
            if (Jq >= 2 && !mbar_wait_warp(bar(B_SE + b), ((Jq >> 1) - 1) & 1, abort_flag, p.status))
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
                umma_commit(bar(B_SF + b));
            }
            __syncwarp();
            return true;
        };
        for (int t = cid; ok && t < p.T; t += ncl, ++u) {
            if (!mbar_wait_warp(bar(B_QF), u & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            const int nb = nb_s[u & 1];
            if (nb == 0) {
                if (lane == 0)
                    umma_commit(bar(B_QE));
                __syncwarp();
                continue;
            }
            tc_fence_after();
            if (!issue_qk(J)) {
                ok = false;
                break;
            }
            for (int j = 0; j < nb; ++j, ++J) {
                if (j + 1 < nb) {
                    if (!issue_qk(J + 1)) {
                        ok = false;
                        break;
                    }
                } else if (lane == 0) {
                    umma_commit(bar(B_QE)); // Q no longer read once these MMAs complete
                }
                const int b = J & 1;
                if (!mbar_wait_warp(bar(B_PF + b), (J >> 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                if (j == 0 && v >= 1 && !mbar_wait_warp(bar(B_OE), (v - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t stage = sbase + OFF_KV + b * kStage;
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint64_t bd = sdesc(stage + kk * 16 * 128, kKVAtom, 1024, 2);
                        umma_f16_ts(tmem + TM_O, tmem + TM_P + 32 * b + 8 * kk, bd, idesc_pv,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(bar(B_PE + b));
                    umma_commit(bar(B_KVE + b));
                    if (j + 1 == nb)
                        umma_commit(bar(B_OF));
                }
                __syncwarp();
            }
            ++v;
        }
        if (lane == 0) {
            umma_commit(bar(B_DONE));
            mbar_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax + epilogue
        const int quad = warp & 3;
        const int h = quad * 32 + lane;                  // head = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        float *xrow = reinterpret_cast<float *>(smem + OFF_X) + h * kXStride;
        const uint32_t x_remote = mapa_shared(smem_u32(xrow), peer);
        const uint32_t xf_remote = mapa_shared(bar(B_XF), peer);
        const uint32_t xe_remote = mapa_shared(bar(B_XE), peer);
        uint32_t J = 0;
        int u = 0, v = 0;
        bool ok = true;
        for (int t = cid; ok && t < p.T; t += ncl, ++u) {
            const int32_t *idx_row = p.idx + (int64_t)t * p.k;
            const int ctx = PAGED ? p.ctx_len[t] : 0;
            if (!mbar_wait_warp(bar(B_QF), u & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            const int nb = nb_s[u & 1];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_QA)); // this token's nb slot has been read
            float m_run = -INFINITY; // running max, log2 domain
            float l_run = 0.f;
            int32_t raw0 = lane < p.k ? idx_row[lane] : -1;
            int32_t raw1 = lane + 32 < p.k ? idx_row[lane + 32] : -1;
            for (int j = 0; j < nb; ++j, ++J) {
                const int b = J & 1;
                // validity of this block's 64 entries; prefetch the next block's indices
                const uint32_t vm_lo = __ballot_sync(0xffffffffu, latent_row<PAGED>(p, t, raw0, ctx) >= 0);
                const uint32_t vm_hi = __ballot_sync(0xffffffffu, latent_row<PAGED>(p, t, raw1, ctx) >= 0);
                {
                    const int n0 = (j + 1) * kBN + lane;
                    raw0 = n0 < p.k ? idx_row[n0] : -1;
                    raw1 = n0 + 32 < p.k ? idx_row[n0 + 32] : -1;
                }
                // 1. partial scores of this CTA
                if (!mbar_wait_warp(bar(B_SF + b), (J >> 1) & 1, abort_flag, p.status)) {
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
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_SE + b));
                // 2. swap partial scores with the peer CTA
                if (J >= 1 && !mbar_wait_warp<true>(bar(B_XE), (J - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < kBN; c += 4)
                    st_async_v4(x_remote + c * 4, sc[c], sc[c + 1], sc[c + 2], sc[c + 3], xf_remote);
                if (threadIdx.x == 64)
                    mbar_arrive_expect_tx(bar(B_XF), 128 * kBN * 4);
                if (!mbar_wait_warp<true>(bar(B_XF), J & 1, abort_flag, p.status)) {
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
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_remote(xe_remote);
                // 3. mask, block max (log2 domain)
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    const bool vld = ((c < 32 ? vm_lo : vm_hi) >> (c & 31)) & 1u;
                    sc[c] = vld ? sc[c] * p.scale_log2 : -INFINITY;
                    mx[c & 3] = fmaxf(mx[c & 3], sc[c]);
                }
                const float bmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
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
                    // O holds this token's blocks < j (j >= 1 here): wait for PV_{J-1}, scale rows
                    if (!mbar_wait_warp(bar(B_PE + ((J - 1) & 1)), ((J - 1) >> 1) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
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
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < kBN; c += 2) {
                    const float p0 = fast_exp2(sc[c] - m_use);
                    const float p1 = fast_exp2(sc[c + 1] - m_use);
                    ls[(c >> 1) & 3] += p0 + p1;
                    pk[c >> 1] = pack_bf16x2(p0, p1);
                }
                l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                if (J >= 2 && !mbar_wait_warp(bar(B_PE + b), ((J >> 1) - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st32(tmem + lane_off + TM_P + 32 * b, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_PF + b));
            }
            if (!ok)
                break;
            // ---- epilogue: O / l -> bf16, LSE
            const bool store = h < p.H;
            __nv_bfloat16 *orow = p.out + ((int64_t)t * p.H + h) * kDv + 256 * rank;
            if (nb > 0) {
                if (!mbar_wait_warp(bar(B_OF), v & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                ++v;
                tc_fence_after();
                const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
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
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_OE));
            } else if (store) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow);
                for (int c = 0; c < 256 / 8; ++c)
                    dst[c] = make_uint4(0, 0, 0, 0);
            }
            if (store && rank == 0)
                p.lse[(int64_t)t * p.H + h] =
                    l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        }
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
    CUtensorMap tq, tkv;
    if (!encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kD, (uint64_t)a.T * a.H, kD * 2, 64, a.H,
                        CU_TENSOR_MAP_SWIZZLE_128B, err, errlen))
        return DSA_ERR_CUDA;
    // one row high: the box of a gather4 load
    if (!encode_tmap_2d(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.kv, kD, (uint64_t)(a.S > 0 ? a.S : 1), kD * 2, 64,
                        1, CU_TENSOR_MAP_SWIZZLE_128B, err, errlen))
        return DSA_ERR_CUDA;
    Params p;
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
    // persistent: one cluster per pair of SMs, each walking tokens c, c + C, ...
    int clusters = num_sms() / 2;
    if (clusters > a.T)
        clusters = a.T;
    if (clusters < 1)
        clusters = 1;
    sparse_mla_kernel<PAGED><<<dim3(2 * clusters), kThreads, kSmem, stream>>>(tq, tkv, p);
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
