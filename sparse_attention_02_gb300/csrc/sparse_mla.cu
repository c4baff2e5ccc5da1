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
//   CTA r keeps O[:, 256r : 256r+256) in TMEM, gathers its V quarter (latent
//   columns [256r, 256r+256), four 64-column swizzle atoms) and its half of the
//   RoPE columns ([512+32r, 512+32r+32), one 32-column atom) of every selected
//   row, and computes the PARTIAL scores over exactly those 288 columns (a
//   K-split of QK^T, no duplicated MMA work); the two CTAs swap their
//   partial-score tiles through distributed shared memory.  Both CTAs then
//   add the same two halves in the same way, so they hold bit-identical
//   scores, run the same softmax (identical P, m and l) and each applies P to
//   its own V quarter.  Stages are 36 KB (three or four in flight); the last
//   160 of this CTA's Q columns live in TMEM (the score MMA reads them as a TMEM
//   A operand), the first 128 in shared memory.

// The swap carries the raw fp32 partial scores (32 KB per 64-key block).  The
// sender warps stage them in shared memory and the copy engine moves them
// (cp.async.bulk into the peer's shared memory, 2 KB per warp and 16-key
// quarter, two staging slots per warp so staging overlaps the copies, one
// arrival barrier per quarter so the add starts with the first): remote stores
// issued by the warps themselves moved a third of that rate, the issue of 2048
// 16-byte stores per block competing with the gathers.
// The softmax warps add the peer's partials to their own in fp32 and apply the
// log2 softmax scale, (own + peer) * scale: the add commutes, so both CTAs hold
// bit-identical scores whose error is that of the fp32 accumulation alone, a
// few fp32 ulps of |S| at any score magnitude (a sharp, one-key softmax with
// scores of tens of nats included).  With the add in the sender warps the
// senders carried the whole swap and set the block rate.
// Partials rounded to fp16 would halve the swap, but put an error of
// ~|S| * 2^-11 on every score and hence on LSE.
//
// Per 64-key block j (double-buffered S buffers, one P buffer; prefill: two
// swap buffers and three KV stages, decode: one and four):
//   producer warps  four warps cp.async the 64 selected rows x 576 B into the
//                   SW128 / SW64 K-major layouts (one 128-byte line per 8
//                   lanes), zero-fill invalid entries, and arrive on the
//                   stage's mbarrier as their copies land
//                   (cp.async.mbarrier.arrive.noinc); at each token they also
//                   write the TMEM part of Q (lane = head);
//   MMA warps       S_j = Q_half . KV_j^T   (M=128 heads, N=64, K=288; A from
//                   smem or TMEM, B K-major in smem), even and odd blocks from
//                   two warps, and
//                   O += P_j . V_j          (M=128, N=256, K=64; A = P from
//                   TMEM, B = the same KV stage read MN-major) from a third.
//                   One thread serialises its tcgen05.mma issue at ~100 cycles
//                   per instruction whatever N is, so the N=64 score MMAs need
//                   two issuing warps to keep the tensor pipe fed;
//   sender warps    thread = head, one warp per TMEM lane quadrant: the
//                   block's 64 partial scores from TMEM in two loads (the S
//                   buffer is then free for them), into shared memory one
//                   16-key quarter at a time, and a bulk copy per quarter to
//                   the peer (completion counted in bytes on the peer's
//                   per-quarter mbarrier) as soon as the peer's softmax warps
//                   have read the previous block's;
//   softmax warps   thread = head, two warps per TMEM lane quadrant, each with
//                   32 of the block's keys: own partial from the S buffer
//                   (then free for the next score MMAs once the senders have
//                   read it too), peer partial from the swap buffer as its two
//                   quarters land (then free for the peer's next block), sum,
//                   scale, mask, max (agreed with the sibling warp through a
//                   spare TMEM column), exp2, running sum; P (bf16) into the
//                   block's P buffer once its previous PV is done.  The
//                   running max only moves when a block exceeds it by more
//                   than 2^8 (then O is rescaled in TMEM), so P <= 256.
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
constexpr int kBN = 64;                  // keys per block
constexpr int kVAtoms = 4;               // 64-column atoms of this CTA's V quarter per stage
constexpr int kQAtom = 128 * 128;        // bytes of one full Q atom (128 rows x 128 B, SW128)
constexpr int kQSmemAtoms = 2;           // Q atoms in shared memory; atoms 2, 3 and the RoPE half sit in TMEM
constexpr int kKVAtom = kBN * 128;       // bytes of one KV atom (64 rows x 128 B, SW128)
constexpr int kKVHalf = kBN * 64;        // bytes of the RoPE half atom (64 rows x 64 B, SW64)
constexpr int kStage = kVAtoms * kKVAtom + kKVHalf; // 36 KB
constexpr int kPf = 3;                   // paged: blocks ahead whose latent rows the producers resolve
constexpr int kXBuf = 128 * kBN * 4;     // one swap buffer: 128 heads x 64 fp32 partial scores
constexpr int kProdWarps = 4;
constexpr int kPvWarp = kProdWarps;      // all PV MMAs (fixed accumulation order) + TMEM owner
constexpr int kQkWarp0 = kProdWarps + 1; // score MMAs of even blocks; kQkWarp0 + 1: odd blocks
constexpr int kSendWarp0 = kProdWarps + 3;
constexpr int kSendWarps = 4;            // one per TMEM lane quadrant: partial scores out to the peer
constexpr int kSoftWarp0 = kSendWarp0 + kSendWarps;
constexpr int kSoftWarps = 8;            // two per TMEM lane quadrant, 32 keys of each block apiece
constexpr int kThreads = 32 * (kSoftWarp0 + kSoftWarps);
constexpr float kRescaleLog2 = 8.f;      // move the running max only when exceeded by this

constexpr int NBAR = 48;

// Shared-memory layout.  Prefill: three KV stages and two swap buffers (the
// peer's next block may land while this one's is read: 23.0 ms against 23.5 ms
// with four stages and one buffer at L = 32768).  Decode: four stages and one
// swap buffer (its rows come from HBM, so the deeper gather ring matters more:
// 78 us against 85 us at B = 64).
template <bool PAGED> struct Layout {
    static constexpr int kNStage = PAGED ? 4 : 3;
    static constexpr int kNX = PAGED ? 1 : 2;                // swap buffers, 32 KB each
    static constexpr int OFF_Q = 0;                          // two full Q atoms
    static constexpr int OFF_KV = OFF_Q + kQSmemAtoms * kQAtom;
    static constexpr int OFF_X = OFF_KV + kNStage * kStage;
    static constexpr int OFF_STG = OFF_X + kNX * kXBuf;      // two 16-key quarters of this CTA's partials, staged
    static constexpr int OFF_BAR = OFF_STG + kXBuf / 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int kSmem = OFF_MISC + 64 + 1024;
    static_assert(kSmem <= 232448, "dynamic shared memory above the 227 KB a CTA may hold");
};

// barrier slots
// [J & 1] for S buffers, [J % kNX] for swap buffers, [J % kNP] for P buffers
constexpr int kNP = 1; // P buffers in TMEM (one: its TMEM columns hold a Q atom instead)
constexpr int B_KVF = 0, B_KVE = 4, B_SF = 8, B_SE = 10, B_XE = 14, B_PF = 16, B_PE = 18,
              B_QF = 22, B_QE = 23, B_QA = 24, B_OF = 25, B_OE = 26, B_DONE = 27,
              B_RB = 28,  // [quad][parity]: sibling softmax warps swapped their block max
              B_RL = 36,  // [quad]: sibling softmax warps swapped their row sums
              B_XQ = 40;  // [xb][q]: the peer's partials of keys [16 q, 16 q + 16) landed in swap buffer xb

// TMEM columns
constexpr uint32_t TM_O = 0;
constexpr uint32_t TM_S = 256;  // two buffers of 64 fp32 partial scores
constexpr uint32_t TM_P = 384;  // kNP buffers of 32 (bf16 pairs)
constexpr uint32_t TM_QT = 416; // Q: atoms 2 and 3 (32 columns of bf16 pairs each) and the RoPE half (16)
constexpr uint32_t TM_RED = 496; // per-head values swapped between the two softmax warps of a quadrant
constexpr uint32_t kTmemCols = 512;

struct Params {
    const __nv_bfloat16 *q;    // [T, H, 576]
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
    // work split (decode with fewer rows than clusters): see Units
    int split, nbk, ncl;       // split flag, 64-key blocks per row (ceil(k / 64)), clusters in the grid
    float *ws_o;               // [2 * ncl, H, 512] fp32 partial outputs (normalised by their own sum)
    float *ws_lse;             // [2 * ncl, H] fp32 partial LSEs
};

// Work units of cluster c.  Unsplit: whole rows t = c, c + ncl, ...  Split:
// the cluster's share [start(c), start(c + 1)) of the flattened (row, 64-key
// block) space, start(c) = floor(c * T * nbk / ncl), cut at row boundaries.
// With T < ncl a share is shorter than a row, so it touches at most two rows;
// a piece that is not a whole row goes to workspace slot 2c + (its row - the
// share's first row), and combine_kernel merges the pieces of each row.
struct Unit {
    int t, jb, je; // row, blocks [jb, je)
    int slot;      // -1: the whole row, written to out/lse directly
};

__device__ __forceinline__ int64_t share_start(const Params &p, int c)
{
    return (int64_t)c * p.T * p.nbk / p.ncl;
}

struct Units {
    int64_t g, g1;
    int t_first, cid;
    __device__ Units(const Params &p, int c) : cid(c)
    {
        if (p.split) {
            g = share_start(p, c);
            g1 = share_start(p, c + 1);
            t_first = static_cast<int>(g / p.nbk);
        } else {
            g = c;
            g1 = p.T;
            t_first = 0;
        }
    }
    __device__ bool next(const Params &p, Unit &u)
    {
        if (g >= g1)
            return false;
        if (!p.split) {
            u.t = static_cast<int>(g);
            u.jb = 0;
            u.je = p.nbk;
            u.slot = -1;
            g += p.ncl;
            return true;
        }
        u.t = static_cast<int>(g / p.nbk);
        u.jb = static_cast<int>(g - (int64_t)u.t * p.nbk);
        const int64_t row_end = (int64_t)(u.t + 1) * p.nbk;
        const int64_t end = row_end < g1 ? row_end : g1;
        u.je = static_cast<int>(end - (int64_t)u.t * p.nbk);
        u.slot = (u.jb == 0 && u.je == p.nbk) ? -1 : 2 * cid + (u.t - t_first);
        g = end;
        return true;
    }
    // row of the unit after the current one, or -1
    __device__ int peek_row(const Params &p) const
    {
        if (g >= g1)
            return -1;
        return p.split ? static_cast<int>(g / p.nbk) : static_cast<int>(g);
    }
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

// Copy engine: `bytes` of this CTA's shared memory into a peer's (both 16-byte
// aligned, a multiple of 16 bytes), completion counted on the peer's mbarrier.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes, uint32_t bar_cluster)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_cluster),
                 "r"(src_cta), "r"(bytes), "r"(bar_cluster)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

template <bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q, Params p)
{
    using Lay = Layout<PAGED>;
    constexpr int kNStage = Lay::kNStage, kNX = Lay::kNX;
    constexpr int OFF_Q = Lay::OFF_Q, OFF_KV = Lay::OFF_KV, OFF_X = Lay::OFF_X, OFF_STG = Lay::OFF_STG,
                  OFF_BAR = Lay::OFF_BAR, OFF_MISC = Lay::OFF_MISC;
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

    // ---- one-time setup
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNStage; ++i) {
            mbar_init(bar(B_KVF + i), 32 * kProdWarps);
            mbar_init(bar(B_KVE + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SF + i), 1);
            mbar_init(bar(B_SE + i), kSoftWarps + kSendWarps);
        }
        for (int i = 0; i < kNX; ++i) {
            mbar_init(bar(B_XE + i), kSoftWarps); // the peer's softmax warps have read its contents
        }
        for (int i = 0; i < kNP; ++i) {
            mbar_init(bar(B_PF + i), kSoftWarps);
            mbar_init(bar(B_PE + i), 1);
        }
        for (int i = 0; i < 4 * kNX; ++i) {
            mbar_init(bar(B_XQ + i), 1);
            mbar_arrive_expect_tx(bar(B_XQ + i), kXBuf / 4); // armed for blocks 0 .. kNX - 1
        }
        mbar_init(bar(B_QF), 1 + kProdWarps); // the Q TMA (expect_tx) + each producer's TMEM part
        mbar_init(bar(B_QE), 2);
        mbar_init(bar(B_QA), kSoftWarps + kSendWarps + 1); // softmax, sender and PV warps read each token's nb slot
        mbar_init(bar(B_OF), 1);
        mbar_init(bar(B_OE), kSoftWarps);
        mbar_init(bar(B_DONE), 3);
        for (int i = 0; i < 8; ++i)
            mbar_init(bar(B_RB + i), 2);
        for (int i = 0; i < 4; ++i)
            mbar_init(bar(B_RL + i), 2);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // Q rows >= H stay zero (their scores are computed but never stored).
    if (p.H < 128) {
        const int nz = 128 - p.H;
        for (int i = threadIdx.x; i < kQSmemAtoms * nz * 8; i += kThreads) {
            const int a = i / (nz * 8), rem = i % (nz * 8);
            *reinterpret_cast<uint4 *>(smem + OFF_Q + a * kQAtom + (p.H + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == kPvWarp)
        tmem_alloc(sbase + OFF_MISC, kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all(); // both CTAs' barriers exist before any remote operation
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    grid_dep_wait(); // no global memory before this: the previous kernel may still be running
    grid_dep_launch();

    if (warp < kProdWarps) {
        // ------------------------------------------------------ producers
        // Warp pw fills rows [16 pw, 16 pw + 16) of each stage.  Lanes 0..15
        // hold those rows' latent-row indices; one cp.async instruction moves
        // four rows x 128 B (lane = 8 x row-in-4 + 16-byte chunk).  At each
        // token, warp pw also writes TMEM lane quadrant pw's part of Q.
        const int pw = warp;
        const int q_row0 = 16 * pw;
        const __nv_bfloat16 *kv_cols = p.kv + 256 * rank;          // this CTA's V quarter
        const __nv_bfloat16 *rope_cols = p.kv + 512 + 32 * rank;   // this CTA's half of the RoPE columns
        uint32_t J = 0;
        int u = 0;
        bool ok = true;
        Units it(p, cid);
        Unit un;
        for (; ok && it.next(p, un); ++u) {
            const int t = un.t;
            const int32_t *idx_row = p.idx + (int64_t)t * p.k;
            const int ctx = PAGED ? p.ctx_len[t] : 0;
            // the unit's blocks up to its last in-range entry.  Paged (decode: the
            // scan sits before the unit's first gather, nothing hides it):
            // backwards, 128 entries (one 16-byte load per lane) at a time, so a
            // row whose last block holds an in-range entry (every row whose
            // context reaches k) takes one round (all 2048 entries read forwards
            // cost ~7 us); prefill overlaps the scan with the previous token's blocks
            int last = -1;
            const int i_beg = un.jb * kBN;
            const int i_end = un.je * kBN < p.k ? un.je * kBN : p.k;
            if (PAGED && (p.k & 3) == 0 && (reinterpret_cast<uintptr_t>(p.idx) & 15u) == 0) {
                const int4 *q4 = reinterpret_cast<const int4 *>(idx_row);
                for (int c1 = i_end; c1 > i_beg && last < 0; c1 -= 128) {
                    // i_beg, i_end and i are multiples of 4: a load is wholly inside or
                    // wholly before [i_beg, c1)
                    const int i = c1 - 128 + 4 * lane;
                    if (i >= i_beg) {
                        const int4 v = __ldg(q4 + (i >> 2));
                        const int vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (in_range<PAGED>(p, vv[e], ctx))
                                last = i + e;
                    }
                    for (int o = 16; o > 0; o >>= 1) {
                        const int y = __shfl_xor_sync(0xffffffffu, last, o);
                        last = y > last ? y : last;
                    }
                }
            } else {
#pragma unroll 8
                for (int i = i_beg + lane; i < i_end; i += 32)
                    if (in_range<PAGED>(p, idx_row[i], ctx))
                        last = i;
            }
            for (int o = 16; o > 0; o >>= 1) {
                const int y = __shfl_xor_sync(0xffffffffu, last, o);
                last = y > last ? y : last;
            }
            const int nb = last < 0 ? 0 : last / kBN + 1 - un.jb;
            // Q (shared memory and TMEM parts) is reused: the score MMAs must be
            // done reading the previous token's Q; warp 0 also reuses the nb slot,
            // which the softmax, sender and PV warps must have taken
            if (u >= 1 && !mbar_wait_warp(bar(B_QE), (u - 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            if (pw == 0) {
                if (u >= 1 && !mbar_wait_warp(bar(B_QA), (u - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    nb_s[u & 1] = nb;
                    const int x0 = 256 * rank; // this CTA's Q columns: its V quarter ...
                    if (nb > 0) {
                        mbar_arrive_expect_tx(bar(B_QF), kQSmemAtoms * p.H * 128);
                        for (int a = 0; a < kQSmemAtoms; ++a)
                            tma_load_2d(sbase + OFF_Q + a * kQAtom, &tm_q, bar(B_QF), x0 + 64 * a, t * p.H);
                    } else {
                        mbar_arrive(bar(B_QF));
                    }
                    const int tn = it.peek_row(p);
                    if (tn >= 0 && tn != t) {
                        for (int a = 0; a < 4; ++a)
                            tma_prefetch_l2_2d(&tm_q, x0 + 64 * a, tn * p.H);
                        tma_prefetch_l2_2d(&tm_q, 512, tn * p.H); // ... and its RoPE half
                    }
                }
                __syncwarp();
            }
            if (nb > 0) {
                // TMEM part of Q for heads 32 pw .. 32 pw + 31 (lane = head): atoms 2 and 3
                // of the V quarter (128 columns) and the RoPE half (32 columns), as bf16
                // pairs, the A-operand layout of a TMEM-sourced MMA
                const int h = 32 * pw + lane;
                const uint32_t tq = tmem + (static_cast<uint32_t>(32 * pw) << 16) + TM_QT;
                const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + ((int64_t)t * p.H + (h < p.H ? h : 0)) * kD);
#pragma unroll 1
                for (int a = 0; a < 2; ++a) {
                    uint32_t qa[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v = h < p.H ? __ldg(qrow + (256 * rank + 128 + 64 * a) / 8 + c) : make_uint4(0, 0, 0, 0);
                        qa[4 * c] = v.x;
                        qa[4 * c + 1] = v.y;
                        qa[4 * c + 2] = v.z;
                        qa[4 * c + 3] = v.w;
                    }
                    tmem_st32(tq + 32 * a, qa);
                    tmem_st_wait();
                }
                {
                    uint32_t qr[16];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v = h < p.H ? __ldg(qrow + (512 + 32 * rank) / 8 + c) : make_uint4(0, 0, 0, 0);
                        qr[4 * c] = v.x;
                        qr[4 * c + 1] = v.y;
                        qr[4 * c + 2] = v.z;
                        qr[4 * c + 3] = v.w;
                    }
                    tmem_st16(tq + 64, qr);
                }
                tmem_st_wait();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_QF));
            auto resolve = [&](int j) -> int {
                const int i = j * kBN + q_row0 + (lane & 15);
                const int r = i < p.k ? latent_row<PAGED>(p, t, idx_row[i], ctx) : -1;
                if (PAGED && r == -2 && lane < 16)
                    atomicOr(p.status, DSA_DEV_BAD_PAGE);
                return r;
            };
            // Paged (decode): the two dependent loads that locate a latent row
            // (selected position, then block-table entry) run as a software
            // pipeline one block apart, kPf blocks ahead of the gather, so no
            // load result is waited for in the iteration that issued it.  (An L2
            // prefetch of the rows kPf blocks ahead measured 2 us slower per
            // launch at 64 rows and is not issued.)
            auto pf_raw_of = [&](int jj) -> int { // selected position of block jb + jj for this lane's row
                const int i = (un.jb + jj) * kBN + q_row0 + (lane & 15);
                return (jj < nb && i < p.k) ? __ldg(idx_row + i) : -1;
            };
            auto pf_page_of = [&](int sp) -> int { // its pool page, or -1 (no load when out of range)
                if (sp < 0 || sp >= ctx || sp / p.page_size >= p.max_pages)
                    return -1;
                return __ldg(p.block_table + (int64_t)t * p.max_pages + sp / p.page_size);
            };
            auto pf_row_of = [&](int sp, int page) -> int { // latent row, -1 skipped, -2 bad page
                if (sp < 0 || sp >= ctx || sp / p.page_size >= p.max_pages)
                    return -1;
                if (page < 0 || page >= p.num_pages) {
                    if (lane < 16)
                        atomicOr(p.status, DSA_DEV_BAD_PAGE);
                    return -2;
                }
                return page * p.page_size + sp % p.page_size;
            };
            // Paged: rw[q] is this lane's latent row of block j + q; the rows of
            // block j + kPf come out of a pipeline whose loads are a block apart
            // (position of block j + kPf + 2, page of block j + kPf + 1 issued
            // now) and join the ring.
            int rw[kPf];
            int pf_s = -1, pf_page = -1, pf_raw = -1;
            int my_row = -1;
            if (PAGED) {
                int sp[kPf + 2], pg[kPf + 1];
#pragma unroll
                for (int jj = 0; jj < kPf + 2; ++jj)
                    sp[jj] = pf_raw_of(jj);
#pragma unroll
                for (int jj = 0; jj < kPf + 1; ++jj)
                    pg[jj] = pf_page_of(sp[jj]);
#pragma unroll
                for (int jj = 0; jj < kPf; ++jj)
                    rw[jj] = pf_row_of(sp[jj], pg[jj]);
                pf_s = sp[kPf];
                pf_page = pg[kPf];
                pf_raw = sp[kPf + 1];
            } else {
                my_row = nb > 0 ? resolve(un.jb) : -1;
            }
            for (int j = 0; j < nb; ++j, ++J) {
                const int st = J % kNStage;
                int cur;
                if (PAGED) {
                    cur = rw[0];
#pragma unroll
                    for (int q = 0; q + 1 < kPf; ++q)
                        rw[q] = rw[q + 1];
                    rw[kPf - 1] = pf_row_of(pf_s, pf_page); // block j + kPf
                    pf_s = pf_raw;                          // block j + kPf + 1: its page
                    pf_page = pf_page_of(pf_raw);
                    pf_raw = pf_raw_of(j + kPf + 2);        // block j + kPf + 2: its position
                } else {
                    cur = my_row;
                    if (j + 1 < nb)
                        my_row = resolve(un.jb + j + 1); // next block's rows, ahead of the stage wait
                }
                if (J >= kNStage &&
                    !mbar_wait_warp(bar(B_KVE + st), ((J / kNStage) - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t stage = sbase + OFF_KV + st * kStage;
                const int cc = lane & 7;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int il = 4 * m + (lane >> 3);
                    const int row = __shfl_sync(0xffffffffu, cur, il);
                    const int rl = q_row0 + il;
                    const int64_t roff = (int64_t)(row >= 0 ? row : 0) * kD;
                    const uint32_t dst = stage + rl * 128 + ((cc ^ (rl & 7)) << 4); // SW128 atoms
                    const uint32_t bytes = row >= 0 ? 16u : 0u;
#pragma unroll
                    for (int a = 0; a < kVAtoms; ++a)
                        cp_async_16_zfill(dst + a * kKVAtom, kv_cols + roff + a * 64 + cc * 8, bytes);
                    if (cc < 4) // RoPE half: 64-byte rows, SW64 (16-byte chunk ^ (row / 2) % 4)
                        cp_async_16_zfill(stage + kVAtoms * kKVAtom + rl * 64 + ((cc ^ ((rl >> 1) & 3)) << 4),
                                          rope_cols + roff + cc * 8, bytes);
                }
                cp_async_arrive_noinc(bar(B_KVF + st));
            }
        }
        cp_async_wait_all(); // every copy this warp issued has landed before the CTA exits
        if (pw == 0 && lane == 0 && u >= 1)
            mbar_drain(bar(B_QF), (u - 1) & 1);
        __syncwarp();
    } else if (warp == kPvWarp) {
        // -------------------------------------------------- PV MMA issuer
        constexpr uint32_t idesc_pv = idesc_f32acc(128, 256, 1u, false, true);
        // B of PV k-step kk: 16 keys further down the stage (kk * 16 rows * 128 B = kk * 128 units)
        const uint64_t pv_desc0 = sdesc(sbase + OFF_KV, kKVAtom, 1024, 2);
        uint32_t J = 0;
        int u = 0, v = 0;
        bool ok = true;
        Units it(p, cid);
        Unit un;
        for (; ok && it.next(p, un); ++u) {
            if (!mbar_wait_warp(bar(B_QF), u & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            const int nb = nb_s[u & 1];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_QA));
            for (int j = 0; j < nb; ++j, ++J) {
                const int pb = J % kNP, st = J % kNStage;
                // the stage (landed long before P) first, so its proxy fence is off the P -> PV hop
                if (!mbar_wait_warp(bar(B_KVF + st), (J / kNStage) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                fence_proxy_async_smem(); // the stage was written by cp.async (generic proxy)
                if ((j == 0 && v >= 1 && !mbar_wait_warp(bar(B_OE), (v - 1) & 1, abort_flag, p.status)) ||
                    !mbar_wait_warp(bar(B_PF + pb), (J / kNP) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t vd = pv_desc0 + static_cast<uint64_t>((st * kStage) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        umma_f16_ts(tmem + TM_O, tmem + TM_P + 32 * pb + 8 * kk, vd + static_cast<uint64_t>(kk * 128),
                                    idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(bar(B_PE + pb));
                    umma_commit(bar(B_KVE + st));
                    if (j + 1 == nb)
                        umma_commit(bar(B_OF));
                }
                __syncwarp();
            }
            if (nb > 0)
                ++v;
        }
        if (lane == 0) {
            umma_commit(bar(B_DONE));
            mbar_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else if (warp < kSendWarp0) {
        // -------------------------------- score MMA issuers (block parity)
        const uint32_t par = static_cast<uint32_t>(warp - kQkWarp0);
        constexpr uint32_t idesc_qk = idesc_f32acc(128, kBN, 1u, false, false);
        uint32_t J = 0;
        int u = 0;
        bool ok = true;
        // This CTA's 288 score columns: its V quarter [256 r, 256 r + 256) (16
        // k-steps of 16 columns) and its half of the RoPE columns [512 + 32 r,
        // +32) (2 k-steps).  A operand: k-steps 0..7 from the two Q atoms in
        // shared memory, k-steps 8..17 from TMEM (atoms 2 and 3, then the RoPE
        // half).  B operand: the stage's four SW128 atoms, then its SW64 RoPE
        // half atom.  Descriptors are precomputed: the issue loop is one add and
        // one tcgen05.mma per k-step.
        uint64_t qd[4 * kQSmemAtoms];
        uint32_t bofs[16]; // B offset of k-step s < 16 within a KV stage, 16-byte units
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            if (s < 4 * kQSmemAtoms)
                qd[s] = sdesc(sbase + OFF_Q + (s >> 2) * kQAtom + (s & 3) * 32, 16, 1024, 2);
            bofs[s] = static_cast<uint32_t>(((s >> 2) * kKVAtom + (s & 3) * 32) >> 4);
        }
        const uint64_t kv_desc0 = sdesc(sbase + OFF_KV, 16, 1024, 2);
        const uint64_t kvh_desc0 = sdesc(sbase + OFF_KV + kVAtoms * kKVAtom, 16, 512, 4);
        Units it(p, cid);
        Unit un;
        for (; ok && it.next(p, un); ++u) {
            if (!mbar_wait_warp(bar(B_QF), u & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            const int nb = nb_s[u & 1];
            tc_fence_after();
            for (int j = 0; j < nb; ++j, ++J) {
                if ((J & 1u) != par)
                    continue;
                const int st = J % kNStage, b = J & 1;
                if (!mbar_wait_warp(bar(B_KVF + st), (J / kNStage) & 1, abort_flag, p.status) ||
                    (J >= 2 && !mbar_wait_warp(bar(B_SE + b), ((J >> 1) - 1) & 1, abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                fence_proxy_async_smem(); // the stage was written by cp.async (generic proxy)
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t soff = static_cast<uint64_t>((st * kStage) >> 4);
                    const uint64_t sd = kv_desc0 + soff, sdh = kvh_desc0 + soff;
                    const uint32_t d_tmem = tmem + TM_S + 64 * b;
                    umma_f16_ss(d_tmem, qd[0], sd + bofs[0], idesc_qk, 0u);
#pragma unroll
                    for (int s = 1; s < 4 * kQSmemAtoms; ++s)
                        umma_f16_ss(d_tmem, qd[s], sd + bofs[s], idesc_qk, 1u);
#pragma unroll
                    for (int s = 4 * kQSmemAtoms; s < 16; ++s)
                        umma_f16_ts(d_tmem, tmem + TM_QT + 8 * (s - 4 * kQSmemAtoms), sd + bofs[s], idesc_qk, 1u);
#pragma unroll
                    for (int s = 16; s < 18; ++s)
                        umma_f16_ts(d_tmem, tmem + TM_QT + 8 * (s - 4 * kQSmemAtoms),
                                    sdh + static_cast<uint64_t>(2 * (s - 16)), idesc_qk, 1u);
                    umma_commit(bar(B_SF + b));
                }
                __syncwarp();
            }
            // Q is free for the next token once this warp's score MMAs complete
            if (lane == 0)
                umma_commit(bar(B_QE));
            __syncwarp();
        }
        if (lane == 0) {
            umma_commit(bar(B_DONE));
            mbar_drain(bar(B_DONE), 0);
        }
        __syncwarp();
    } else if (warp < kSoftWarp0) {
        // -------------------------------- score senders
        // Thread = head (TMEM lane), all 64 keys of each block.  The block's 64
        // partial-score columns are read first (two TMEM loads, one wait), which
        // frees the S buffer, then go to the peer one 16-key quarter at a time:
        // staged in shared memory (two slots per warp), then a bulk copy of the
        // warp's 32 head rows (completion counted in bytes on the peer's
        // per-quarter mbarrier, which the peer's softmax warps wait on and
        // re-arm).  The next block's copies wait until the peer's softmax warps
        // have read this one's.  Per-warp handshakes per quarter measured slower (the waits
        // inside the copy loop cost more than the coupling they remove).
        const int quad = warp & 3;
        const int h = quad * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t xe_remote0 = mapa_shared(bar(B_XE), peer);
        // swap buffer: four quarters of 16 keys
        // ([q][head][16 fp32], 64-byte rows, chunk c of head h's row at c ^ ((h >> 1) & 3): eight
        // consecutive heads storing or reading the same chunk hit eight different banks; staging: two
        // 2 KB slots per warp, one quarter of its 32 head rows each)
        const uint32_t qsw = static_cast<uint32_t>((h >> 1) & 3);
        uint8_t *stg_row = smem + OFF_STG + quad * 4096 + lane * 64;
        const uint32_t stg_q = sbase + OFF_STG + quad * 4096;
        const uint32_t x_remote_q = mapa_shared(sbase + OFF_X + quad * 32 * 64, peer);
        const uint32_t xq_remote0 = mapa_shared(bar(B_XQ), peer);
        uint32_t J = 0;
        int u = 0;
        bool ok = true;
        Units it(p, cid);
        Unit un;
        for (; ok && it.next(p, un); ++u) {
            if (!mbar_wait_warp(bar(B_QF), u & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            const int nb = nb_s[u & 1];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_QA)); // this token's nb slot has been read
            for (int j = 0; j < nb; ++j, ++J) {
                const int b = J & 1;
                const int xb = J % kNX;
                const uint32_t s_cols = tmem + lane_off + TM_S + 64 * b;
                // the peer's swap buffer xb must be free (its softmax warps have read block J - kNX)
                if (!mbar_wait_warp(bar(B_SF + b), (J >> 1) & 1, abort_flag, p.status) ||
                    (J >= kNX &&
                     !mbar_wait_warp<true>(bar(B_XE + xb), ((J / kNX) - 1) & 1, abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t ra[32], rb[32];
                tmem_ld32(s_cols, ra);
                tmem_ld32(s_cols + 32, rb);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_SE + b)); // this warp has read the block's partials
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    // slot qq & 1 is free once the copy issued two quarters ago has read it
                    if (lane == 0)
                        bulk_wait_read1();
                    __syncwarp();
                    uint8_t *srow = stg_row + (qq & 1) * 2048;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int e = 16 * (qq & 1) + 4 * cc;
                        const uint32_t *r = qq < 2 ? ra : rb;
                        *reinterpret_cast<uint4 *>(srow + ((static_cast<uint32_t>(cc) ^ qsw) << 4)) =
                            make_uint4(r[e], r[e + 1], r[e + 2], r[e + 3]);
                    }
                    fence_proxy_async_smem(); // the copy engine reads what the generic stores wrote
                    __syncwarp();
                    if (lane == 0) {
                        // this warp's 32 head rows of the quarter (2 KB, contiguous in both buffers)
                        bulk_s2cluster(x_remote_q + xb * kXBuf + qq * (kXBuf / 4), stg_q + (qq & 1) * 2048, 32 * 64,
                                       xq_remote0 + 8u * (4 * xb + qq));
                        bulk_commit();
                    }
                }
            }
        }
        if (lane == 0)
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); // this warp's copies are complete
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax + epilogue
        // Warp half hf of a lane quadrant owns keys [32 hf, 32 hf + 32) of every
        // block, O columns [128 hf, 128 hf + 128) in the epilogue and a partial
        // row sum; the two warps agree on each block's max before exponentiating.
        const int sw = warp - kSoftWarp0;
        const int quad = warp & 3;
        const int hf = sw >> 2;
        const int h = quad * 32 + lane;                  // head = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t red = tmem + lane_off + TM_RED;
        const uint8_t *xq_row = smem + OFF_X + h * 64;
        const uint32_t xqsw = static_cast<uint32_t>((h >> 1) & 3);
        const uint32_t xe_remote_sm = mapa_shared(bar(B_XE), peer);
        uint32_t J = 0;
        int u = 0, v = 0;
        bool ok = true;
        Units it(p, cid);
        Unit un;
        for (; ok && it.next(p, un); ++u) {
            const int t = un.t;
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
            float m_run = -INFINITY; // running max, log2 domain (same in both sibling warps)
            float l_run = 0.f;       // this warp's partial row sum
            const int i0 = un.jb * kBN + 32 * hf + lane;
            int32_t raw = i0 < p.k ? idx_row[i0] : -1;
            // Paged: an entry is valid when its position is in the context and its
            // block-table entry names a pool page.  The block-table entry of block
            // j + 1 and the position of block j + 2 are loaded during block j, so
            // the mask never waits for a load.
            auto page_of = [&](int32_t sp) -> int {
                if (sp < 0 || sp >= ctx || sp / p.page_size >= p.max_pages)
                    return -1;
                return __ldg(p.block_table + (int64_t)t * p.max_pages + sp / p.page_size);
            };
            int pg = 0, raw_n = -1;
            if (PAGED) {
                pg = page_of(raw);
                const int n1 = i0 + kBN;
                raw_n = n1 < p.k ? idx_row[n1] : -1;
            }
            for (int j = 0; j < nb; ++j, ++J) {
                const int b = J & 1;
                // validity of this warp's 32 entries; the next block's index ahead
                uint32_t vmask;
                if (PAGED) {
                    vmask = __ballot_sync(0xffffffffu, raw >= 0 && raw < ctx && pg >= 0 && pg < p.num_pages);
                    raw = raw_n;
                    pg = page_of(raw);
                    const int n2 = i0 + (j + 2) * kBN;
                    raw_n = n2 < p.k ? idx_row[n2] : -1;
                } else {
                    vmask = __ballot_sync(0xffffffffu, latent_row<PAGED>(p, t, raw, ctx) >= 0);
                    const int n0 = (un.jb + j + 1) * kBN + 32 * hf + lane;
                    raw = n0 < p.k ? idx_row[n0] : -1;
                }
                // 1. this CTA's partial scores of the warp's 32 keys from the S buffer (free for
                //    block J + 2 once the senders have read it too)
                const int pb = J % kNP;
                if (!mbar_wait_warp(bar(B_SF + b), (J >> 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float sc[32];
                {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_off + TM_S + 64 * b + 32 * hf, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        sc[c] = __uint_as_float(r[c]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_SE + b));
                // the peer's partials of this warp's two quarters, each added as it lands:
                // (own + peer) * scale in fp32 (the add commutes: both CTAs hold the same bits)
                const int xb = J % kNX;
                bool got = true;
#pragma unroll
                for (int qh = 0; qh < 2; ++qh) {
                    if (!mbar_wait_warp<true>(bar(B_XQ + 4 * xb + 2 * hf + qh), (J / kNX) & 1, abort_flag, p.status)) {
                        got = false;
                        break;
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float4 pv = *reinterpret_cast<const float4 *>(
                            xq_row + xb * kXBuf + (2 * hf + qh) * (kXBuf / 4) + ((static_cast<uint32_t>(c) ^ xqsw) << 4));
                        const int e0 = 16 * qh + 4 * c;
                        sc[e0] = (sc[e0] + pv.x) * p.scale_log2;
                        sc[e0 + 1] = (sc[e0 + 1] + pv.y) * p.scale_log2;
                        sc[e0 + 2] = (sc[e0 + 2] + pv.z) * p.scale_log2;
                        sc[e0 + 3] = (sc[e0 + 3] + pv.w) * p.scale_log2;
                    }
                }
                if (!got) {
                    ok = false;
                    break;
                }
                __syncwarp(); // every lane has read its rows of the two quarters
                if (lane == 0) {
                    if (quad == 0) // both quarters' phases of block J are complete: arm them for block J + kNX
                        for (int q = 2 * hf; q < 2 * hf + 2; ++q)
                            mbar_arrive_expect_tx(bar(B_XQ + 4 * xb + q), kXBuf / 4);
                    mbar_arrive_remote_relaxed(xe_remote_sm + 8u * xb); // the peer may send into buffer xb again
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    sc[c] = ((vmask >> c) & 1u) ? sc[c] : -INFINITY;
                    mx[c & 3] = fmaxf(mx[c & 3], sc[c]);
                }
                const float hmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                // 4. block max over both halves: swap through a spare TMEM column
                tmem_st1(red + 2 * b + hf, __float_as_uint(hmax));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_RB + 2 * quad + b));
                if (!mbar_wait_warp(bar(B_RB + 2 * quad + b), (J >> 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t omax_bits = tmem_ld1(red + 2 * b + (hf ^ 1));
                tmem_ld_wait();
                const float bmax = fmaxf(hmax, __uint_as_float(omax_bits));
                // 5. move the running max only when it is exceeded by more than 2^8
                //    (same decision in both sibling warps; each rescales its O half)
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
                    if (!mbar_wait_warp(bar(B_PE + (J - 1) % kNP), ((J - 1) / kNP) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 128 * hf; c0 < 128 * hf + 128; c0 += 32) {
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
                // 6. P = exp2(S - m), partial sum, bf16 pairs into this warp's half of P
                uint32_t pk[16];
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float p0 = fast_exp2(sc[c] - m_use);
                    const float p1 = fast_exp2(sc[c + 1] - m_use);
                    ls[(c >> 1) & 3] += p0 + p1;
                    pk[c >> 1] = pack_bf16x2(p0, p1);
                }
                l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                // P buffer pb is free once the PV MMAs of block J - kNP are done
                if (J >= kNP && !mbar_wait_warp(bar(B_PE + pb), ((J / kNP) - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st16(tmem + lane_off + TM_P + 32 * pb + 16 * hf, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(B_PF + pb));
            }
            if (!ok)
                break;
            // ---- epilogue: row sum of both halves (fixed order), O / l -> bf16, LSE
            tmem_st1(red + 4 + 2 * (u & 1) + hf, __float_as_uint(l_run));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(B_RL + quad));
            if (!mbar_wait_warp(bar(B_RL + quad), u & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float l_other = __uint_as_float(tmem_ld1(red + 4 + 2 * (u & 1) + (hf ^ 1)));
            tmem_ld_wait();
            const float l_tot = hf == 0 ? l_run + l_other : l_other + l_run;
            const bool store = h < p.H;
            const bool part = un.slot >= 0; // a piece of a split row: fp32 O / l and LSE into the workspace
            __nv_bfloat16 *orow = p.out + ((int64_t)t * p.H + h) * kDv + 256 * rank + 128 * hf;
            float *prow = part ? p.ws_o + ((int64_t)un.slot * p.H + h) * kDv + 256 * rank + 128 * hf : nullptr;
            if (nb > 0) {
                if (!mbar_wait_warp(bar(B_OF), v & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                ++v;
                tc_fence_after();
                const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_off + TM_O + 128 * hf + c0, r);
                    tmem_ld_wait();
                    if (part) {
                        if (store) {
                            float4 *dst = reinterpret_cast<float4 *>(prow + c0);
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                dst[c] = make_float4(__uint_as_float(r[4 * c]) * inv_l, __uint_as_float(r[4 * c + 1]) * inv_l,
                                                     __uint_as_float(r[4 * c + 2]) * inv_l,
                                                     __uint_as_float(r[4 * c + 3]) * inv_l);
                        }
                        continue;
                    }
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
            } else if (store && part) {
                float4 *dst = reinterpret_cast<float4 *>(prow);
                for (int c = 0; c < 128 / 4; ++c)
                    dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (store) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow);
                for (int c = 0; c < 128 / 8; ++c)
                    dst[c] = make_uint4(0, 0, 0, 0);
            }
            if (store && rank == 0 && hf == 0) {
                const float lv = l_tot > 0.f ? (m_run + __log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
                if (part)
                    p.ws_lse[(int64_t)un.slot * p.H + h] = lv;
                else
                    p.lse[(int64_t)t * p.H + h] = lv;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all(); // no CTA leaves while its peer may still touch its smem
    if (warp == kPvWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merges the pieces of each split row: for a row covered by clusters
// c_lo < ... < c_hi with piece LSEs L_c and outputs O_c (each normalised by
// its own sum), LSE = ln sum_c exp(L_c) and O = sum_c exp(L_c - LSE) O_c,
// rounded to bf16 (the split-and-merge identity of a softmax).  Rows that one
// cluster held whole were written directly and are skipped.  Block (t, y):
// heads [8y, 8y + 8), one warp per head, 16 columns per lane.
__global__ void __launch_bounds__(256) combine_kernel(Params p)
{
    grid_dep_wait();
    grid_dep_launch();
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const int64_t total = (int64_t)p.T * p.nbk;
    auto cluster_of = [&](int64_t g) { return static_cast<int>(((g + 1) * p.ncl + total - 1) / total - 1); };
    const int c_lo = cluster_of((int64_t)t * p.nbk), c_hi = cluster_of((int64_t)(t + 1) * p.nbk - 1);
    const int h = 8 * blockIdx.y + (threadIdx.x >> 5);
    if (c_lo == c_hi || h >= p.H)
        return;
    const int np = c_hi - c_lo + 1;
    const int col = lane * 16;
    auto slot_of = [&](int c) { return 2 * c + (t - static_cast<int>(share_start(p, c) / p.nbk)); };
    // lane q holds the LSE of piece q0 + q of each group of 32
    float lmax = -INFINITY;
    for (int q0 = 0; q0 < np; q0 += 32) {
        const int q = q0 + lane;
        if (q < np)
            lmax = fmaxf(lmax, p.ws_lse[(int64_t)slot_of(c_lo + q) * p.H + h]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        acc[e] = 0.f;
    float wsum = 0.f;
    if (lmax != -INFINITY) {
        for (int q0 = 0; q0 < np; q0 += 32) {
            const int q = q0 + lane;
            const float wl = q < np ? expf(p.ws_lse[(int64_t)slot_of(c_lo + q) * p.H + h] - lmax) : 0.f;
            const int nq = np - q0 < 32 ? np - q0 : 32;
#pragma unroll 4
            for (int e = 0; e < nq; ++e) {
                const float wgt = __shfl_sync(0xffffffffu, wl, e);
                wsum += wgt;
                const float4 *src =
                    reinterpret_cast<const float4 *>(p.ws_o + ((int64_t)slot_of(c_lo + q0 + e) * p.H + h) * kDv + col);
                const float4 x0 = src[0], x1 = src[1], x2 = src[2], x3 = src[3];
                const float xs[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                      x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    acc[c] += wgt * xs[c];
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        o[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((int64_t)t * p.H + h) * kDv + col);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    if (lane == 0)
        p.lse[(int64_t)t * p.H + h] = lmax == -INFINITY ? -INFINITY : lmax + logf(wsum);
}

// Clusters and split decision of a launch.  Decode cuts rows into pieces only
// when at most two thirds of the clusters would otherwise have a row: a piece
// costs its own Q load, pipeline fill and fp32 partial store plus the merge,
// which measured a loss at 64 rows on 76 clusters, break-even at 48 and a gain
// below (1.3x at 32 rows, 1.7x at 8).  Prefill never splits.
struct Plan {
    int clusters, split, nbk;
};

Plan plan(bool paged, int T, int k)
{
    Plan pl;
    pl.nbk = (k + kBN - 1) / kBN;
    int clusters = num_sms() / 2;
    if (clusters < 1)
        clusters = 1;
    pl.split = 0;
    if (paged) {
        const int64_t tot = (int64_t)T * pl.nbk;
        const int ncl = tot < clusters ? static_cast<int>(tot) : clusters;
        if (3 * (int64_t)T <= 2 * (int64_t)ncl) {
            pl.split = 1;
            pl.clusters = ncl;
            return pl;
        }
    }
    pl.clusters = T < clusters ? (T > 0 ? T : 1) : clusters;
    return pl;
}

template <bool PAGED>
int launch(const MlaArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    static std::atomic<bool> attr_set[64];
    constexpr int kSmem = Layout<PAGED>::kSmem;
    if (cudaError_t e_attr = raise_smem_limit_once(sparse_mla_kernel<PAGED>, kSmem, attr_set);
        e_attr != cudaSuccess) {
        snprintf(err, errlen, "cudaFuncSetAttribute(sparse_mla): %s", cudaGetErrorString(e_attr));
        return DSA_ERR_CUDA;
    }
    // Q as [T*H rows, 576 cols]: 64-column boxes (SW128)
    CUtensorMap tq;
    if (!encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kD, (uint64_t)a.T * a.H, kD * 2, 64, a.H,
                        CU_TENSOR_MAP_SWIZZLE_128B, err, errlen))
        return DSA_ERR_CUDA;
    Params p;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
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
    // persistent: one cluster per pair of SMs, each walking its work units
    const Plan pl = plan(PAGED, a.T, a.k);
    p.split = pl.split;
    p.nbk = pl.nbk;
    p.ncl = pl.clusters;
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    if (pl.split) {
        const size_t o_bytes = (size_t)2 * pl.clusters * a.H * kDv * sizeof(float);
        if (!a.workspace || a.workspace_bytes < o_bytes + (size_t)2 * pl.clusters * a.H * sizeof(float)) {
            snprintf(err, errlen, "workspace too small for the split decode");
            return DSA_ERR_WORKSPACE;
        }
        p.ws_o = static_cast<float *>(a.workspace);
        p.ws_lse = reinterpret_cast<float *>(static_cast<char *>(a.workspace) + o_bytes);
    }
    cudaError_t e = launch_pdl(sparse_mla_kernel<PAGED>, dim3(2 * pl.clusters), dim3(kThreads), kSmem, stream, 1, tq, p);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "sparse_mla launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    if (pl.split) {
        e = launch_pdl(combine_kernel, dim3(a.T, (a.H + 7) / 8), dim3(256), 0, stream, 1, p);
        if (e != cudaSuccess) {
            snprintf(err, errlen, "sparse_mla combine launch: %s", cudaGetErrorString(e));
            return DSA_ERR_CUDA;
        }
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

// Split decode: [2 * clusters, H, 512] fp32 partial outputs, then [2 * clusters, H] fp32 LSEs.
size_t mla_decode_workspace_bytes(int B, int H, int k)
{
    const Plan pl = plan(true, B, k);
    return pl.split ? (size_t)2 * pl.clusters * H * (kDv + 1) * sizeof(float) : 0;
}

} // namespace dsa
