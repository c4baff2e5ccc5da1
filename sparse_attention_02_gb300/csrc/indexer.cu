// Lightning indexer on sm_103a: FP8 tcgen05 GEMM with a fused ReLU / head-weight
// / causal-mask epilogue.
//
// Defines (release summary "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency
// with DeepSeek Sparse Attention", section "Method"):
//     I[t,s] = sum_j w[t,j] * ReLU(q[t,j] . k[s]),   s <= t,
// with q and k stored as FP8 E4M3 codes and one positive scale per token.
// Because the scales are positive they factor out of the ReLU:
//     I[t,s] = q_scale[t] * k_scale[s] * sum_j w[t,j] * ReLU(q8[t,j] . k8[s]),
// so the MMA runs on the raw codes, q_scale is folded into w once per CTA and
// k_scale is applied once per key.
//
// Tiling.  One MMA (M = 128 keys, N = tokens x heads, K = d_I) per group of
// tokens that share a key tile:
//     A = 128 key rows of k8   (K-major, TMA tile, swizzle = d_I bytes)
//     B = N query rows of q8   (row = token * H_I + head, K-major)
//     D = TMEM [128 lanes = keys] x [N columns = (token, head)] fp32
// With keys on the lanes, the sum over heads runs along a thread's own TMEM
// columns.
//
// Roles (one CTA, warp-specialised):
//   warp 0      TMA producer: the CTA's query tiles once, then key tiles
//               through an NSTAGE ring (paged: one TMA per page of the tile).
//   warp 1      TMEM allocator and MMA issuer (one elected lane).
//   warps 2..   epilogue, up to four warps per TMEM lane quadrant.  Two TMEM
//               accumulators alternate so the MMA of one item overlaps the
//               epilogue of the other.  Contiguous keys with H_I a multiple of
//               8 (prefill): the epilogue reads 16-lane x 256-bit fragments,
//               each thread holds two keys and a fixed quarter of every
//               8-column block, so its head weights stay in registers; the
//               head sum ends in a four-lane shuffle reduce.  Otherwise (paged
//               decode, H_I = 4) each thread owns one key lane and reads the
//               weights from shared memory.
#include "common.cuh"
#include "launch.h"

#include <limits.h>
#include <stdio.h>

namespace dsa {
namespace {

constexpr int kTileKeys = 128;
constexpr int kCandRegions = 128; // candidate-mode regions per row: one per lane writing the row

template <int HI, int DI, bool PAGED>
struct IdxCfg {
    // Fragment epilogue (16x256b TMEM loads, head weights held in registers)
    // whenever each token's head block is a whole number of 8-column repeats.
    static constexpr bool FRAG = HI % 8 == 0 && !PAGED;
    static constexpr int G = PAGED ? 1 : 256 / HI;        // tokens per accumulator
    static constexpr int NGROUP = (PAGED || FRAG) ? 1 : 2; // token groups sharing a key tile
    static constexpr int R = G * NGROUP;                  // query rows per CTA
    static constexpr int N = G * HI;                      // MMA N
    static constexpr int EPI_SPLIT = N >= 256 ? 4 : (N >= 128 ? 2 : 1); // warps per TMEM lane quadrant
    static constexpr int NEPI = 4 * EPI_SPLIT;            // epilogue warps
    static constexpr int THREADS = 64 + 32 * NEPI;
    static constexpr int NSTAGE = PAGED ? 6 : (NGROUP == 1 ? 8 : 4); // key tiles in flight
    // 32x32b epilogue: TMEM columns and tokens per thread
    static constexpr int NC = N / EPI_SPLIT;
    static constexpr int TPT = NC / HI;
    // fragment epilogue: lane halves per warp, columns per warp, 8-column
    // repeats per warp, tokens per warp, repeats per token, repeats per 64-column chunk
    static constexpr int NLH = EPI_SPLIT >= 2 ? 1 : 2;
    static constexpr int NCW = N / (EPI_SPLIT >= 2 ? EPI_SPLIT / 2 : 1);
    static constexpr int REPS = NCW / 8;
    static constexpr int TPW = NCW / HI;
    static constexpr int RPT = HI / 8;
    static constexpr int CHUNK_REPS = REPS >= 8 ? 8 : REPS;
    static constexpr int QTILE = N * DI;                  // bytes
    static constexpr int KSTAGE = kTileKeys * DI;         // bytes
    static constexpr int ACC_COLS = N < 32 ? 32 : N;
    static constexpr int TMEM_COLS = 2 * ACC_COLS <= 64 ? 64 : (2 * ACC_COLS <= 128 ? 128 : (2 * ACC_COLS <= 256 ? 256 : 512));
    static constexpr uint32_t SWZ = DI == 128 ? 2u : (DI == 64 ? 4u : 6u);
    static constexpr uint32_t SBO = 8 * DI;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = ((OFF_Q + NGROUP * QTILE + 1023) / 1024) * 1024;
    static constexpr int OFF_WQ = OFF_K + NSTAGE * KSTAGE;
    static constexpr int OFF_POS = OFF_WQ + R * HI * 4;
    static constexpr int OFF_BAR = ((OFF_POS + R * 4 + 7) / 8) * 8;
    static constexpr int NBAR = 2 * NSTAGE + 4 + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024; // + slack for 1024-B alignment of the base
    static_assert(N >= 16 && N <= 256 && N % 16 == 0, "MMA N");
    static_assert(FRAG || (NC % 32 == 0 && NC % HI == 0), "epilogue split");
    static_assert(!FRAG || ((CHUNK_REPS == 8 || CHUNK_REPS == 4) && REPS % CHUNK_REPS == 0 && TPW >= 1 &&
                            (TPW == 1 || TPW % 2 == 0) && CHUNK_REPS % RPT == 0), "fragment epilogue split");
    static_assert(DI == 32 || DI == 64 || DI == 128, "d_I");
};

// In the fragment epilogue every kAbsEvery-th column repeat forms ReLU(x) * w
// as (x + |x|) * (w / 2), which is the same rounded product and FMA, on the FMA
// pipe instead of the ALU pipe that carries the max of the other repeats
// (L = 32768: every 3rd or 4th 5.21 ms, 5th 5.13, 6th 5.04-5.06, 8th 5.12).
constexpr int kAbsEvery = 6;

struct Params {
    const float *q_scale;
    const float *w;
    const float *k_scale;
    const int32_t *q_pos;
    const int32_t *block_table;
    float *logits;
    int64_t ld;
    int T, S, max_pages, num_pages, page_size, splits;
    unsigned *status;
    // candidate mode and row filter (see IndexerArgs)
    const float *thr;
    uint2 *cand;
    int32_t *cand_cnt;
    int cap;
    const int32_t *row_flag;
};

// FUSED: candidate mode.  Instead of writing logits, the epilogue appends
// every key whose score is >= the row's threshold to the row's candidate list.
// A row is scored by 8 epilogue warps (TMEM lane quadrant x lane half) and, in
// each, by the 16 lanes of one parity; its list is kCandRegions = 128 fixed
// regions of p.cap entries, one per such lane, which counts its candidates in
// a register: no atomics, no cross-lane step.  Each lane writes its count to
// cand_cnt[row][region] when done.  Same arithmetic as the logits mode, so the
// same fp32 scores.
template <int HI, int DI, bool PAGED, bool FUSED = false>
__global__ void __launch_bounds__(IdxCfg<HI, DI, PAGED>::THREADS, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, Params p)
{
    using C = IdxCfg<HI, DI, PAGED>;
    static_assert(!FUSED || (C::FRAG && C::R <= 8 && C::TPW >= 2 && C::NLH == 1 && 8 * C::NEPI == kCandRegions),
                  "candidate mode: fragment epilogue (every lane stores), one lane half per warp, 8 rows or fewer");
    __shared__ float thr_s[FUSED ? C::R : 1];
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    float *wq_s = reinterpret_cast<float *>(smem + C::OFF_WQ);
    int *pos_s = reinterpret_cast<int *>(smem + C::OFF_POS);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::NSTAGE + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * C::NSTAGE + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * C::NSTAGE + 2 + a); };
    const uint32_t q_bar = bar0 + 8u * (2 * C::NSTAGE + 4);
    const uint32_t done_bar = bar0 + 8u * (2 * C::NSTAGE + 5);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    int *tiles_s = reinterpret_cast<int *>(smem + C::OFF_MISC + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cg = PAGED ? blockIdx.x : (gridDim.x - 1 - blockIdx.x); // heavy groups first
    const int r0 = cg * C::R;

    grid_dep_wait();
    grid_dep_launch();
    if (p.row_flag) {
        // row filter: a CTA none of whose rows is flagged has nothing to do
        int any = 0;
        for (int i = 0; i < C::R; ++i)
            any |= (r0 + i < p.T) ? p.row_flag[r0 + i] : 0;
        if (!any)
            return; // uniform
    }
    // ---- setup: row positions, folded weights, tile range
    const int64_t key_limit = PAGED ? (int64_t)p.max_pages * p.page_size : (int64_t)p.S;
    const int64_t lim = (key_limit < p.ld ? key_limit : p.ld) - 1;
    if (threadIdx.x < C::R) {
        const int r = r0 + threadIdx.x;
        int pos = -1;
        if (r < p.T) {
            int64_t qp = p.q_pos[r];
            if (qp > lim) {
                atomicOr(p.status, DSA_DEV_BAD_POSITION);
                qp = lim;
            }
            pos = qp < 0 ? -1 : (int)qp;
        }
        pos_s[threadIdx.x] = pos;
        if constexpr (FUSED) {
            thr_s[threadIdx.x] = r < p.T ? p.thr[r] : INFINITY;
        }
    }
    for (int i = threadIdx.x; i < C::R * HI; i += C::THREADS) {
        const int r = r0 + i / HI;
        wq_s[i] = r < p.T ? p.w[(int64_t)r * HI + (i % HI)] * p.q_scale[r] : 0.f;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), C::NEPI); // one arrival per epilogue warp
        }
        mbar_init(q_bar, 1);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int mx = -1;
        for (int i = 0; i < C::R; ++i)
            mx = pos_s[i] > mx ? pos_s[i] : mx;
        const int n_tiles = mx < 0 ? 0 : mx / kTileKeys + 1;
        const int per = (n_tiles + p.splits - 1) / p.splits;
        const int t0 = blockIdx.y * per;
        const int t1 = t0 + per < n_tiles ? t0 + per : n_tiles;
        tiles_s[0] = t0;
        tiles_s[1] = t1 > t0 ? t1 : t0;
    }
    __syncthreads();
    const int kt0 = tiles_s[0], kt1 = tiles_s[1];
    if (kt1 <= kt0) {
        if constexpr (FUSED) {
            if (threadIdx.x < C::R * kCandRegions && r0 + threadIdx.x / kCandRegions < p.T)
                p.cand_cnt[(int64_t)r0 * kCandRegions + threadIdx.x] = 0;
        }
        return; // uniform: nothing to score in this split
    }

    if (warp == 1) {
        tmem_alloc(sbase + C::OFF_MISC, C::TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int ntiles = kt1 - kt0;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            mbar_arrive_expect_tx(q_bar, C::NGROUP * C::QTILE);
            for (int g = 0; g < C::NGROUP; ++g)
                tma_load_2d(sbase + C::OFF_Q + g * C::QTILE, &tm_q, q_bar, 0, (r0 + g * C::G) * HI);
        }
        int issued = 0;
        // paged: lane j holds the pool page of logical page bt_base + j; the warp
        // refills all 32 with one load each when a tile runs past them
        int bt_base = INT_MIN / 2, bt_page = -1;
        for (int it = 0; it < ntiles; ++it) {
            const int s = it % C::NSTAGE;
            const int kt = kt0 + it;
            if (PAGED) {
                const int lp0 = (kt * kTileKeys) / p.page_size;
                if (lp0 < bt_base || lp0 + kTileKeys / p.page_size > bt_base + 32) {
                    bt_base = lp0;
                    const int lp = lp0 + lane;
                    bt_page = lp < p.max_pages ? __ldg(p.block_table + (int64_t)r0 * p.max_pages + lp) : -1;
                }
            }
            if (it >= C::NSTAGE &&
                !mbar_wait_warp(empty_bar(s), ((it / C::NSTAGE) - 1) & 1, abort_flag, p.status))
                break;
            const uint32_t dst = sbase + C::OFF_K + s * C::KSTAGE;
            if (!PAGED) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(s), C::KSTAGE);
                    tma_load_2d(dst, &tm_k, full_bar(s), 0, kt * kTileKeys);
                }
            } else {
                if (lane == 0)
                    mbar_arrive_expect_tx(full_bar(s), C::KSTAGE);
                const int per_tile = kTileKeys / p.page_size;
                const int lp0 = (kt * kTileKeys) / p.page_size;
                for (int j = 0; j < per_tile; ++j) {
                    const int page = __shfl_sync(0xffffffffu, bt_page, lp0 + j - bt_base);
                    // An invalid page loads out-of-range rows: TMA fills zeros and
                    // the epilogue skips those keys.
                    const int row = (page >= 0 && page < p.num_pages) ? page * p.page_size
                                                                      : p.num_pages * p.page_size;
                    if (lane == 0)
                        tma_load_2d(dst + j * p.page_size * DI, &tm_k, full_bar(s), 0, row);
                }
            }
            ++issued;
            __syncwarp();
        }
        // drain: every load issued to the ring has landed before the CTA exits
        if (lane == 0) {
            mbar_drain(q_bar, 0);
            for (int it = issued - C::NSTAGE > 0 ? issued - C::NSTAGE : 0; it < issued; ++it)
                mbar_drain(full_bar(it % C::NSTAGE), (it / C::NSTAGE) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_f32acc(128, C::N, 0u, false, false);
        bool ok = mbar_wait_warp(q_bar, 0, abort_flag, p.status);
        for (int it = 0; ok && it < ntiles; ++it) {
            const int s = it % C::NSTAGE;
            if (!mbar_wait_warp(full_bar(s), (it / C::NSTAGE) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            for (int g = 0; g < C::NGROUP; ++g) {
                const int item = it * C::NGROUP + g;
                const int a = item & 1, use = item >> 1;
                if (use >= 1 && !mbar_wait_warp(acce_bar(a), (use - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t abase = sbase + C::OFF_K + s * C::KSTAGE;
                    const uint32_t bbase = sbase + C::OFF_Q + g * C::QTILE;
#pragma unroll
                    for (int kk = 0; kk < DI / 32; ++kk) {
                        const uint64_t ad = sdesc(abase + kk * 32, 16, C::SBO, C::SWZ);
                        const uint64_t bd = sdesc(bbase + kk * 32, 16, C::SBO, C::SWZ);
                        umma_f8f6f4(tmem + a * C::ACC_COLS, ad, bd, idesc, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(accf_bar(a));
                }
                __syncwarp();
            }
            if (!ok)
                break;
            if (lane == 0)
                umma_commit(empty_bar(s));
            __syncwarp();
        }
        // all issued MMAs complete before TMEM is released
        if (lane == 0) {
            umma_commit(done_bar);
            mbar_drain(done_bar, 0);
        }
        __syncwarp();
    } else if constexpr (C::FRAG) {
        // ------------------------------------------- epilogue (fragment form)
        // Warp (quad, j) reads TMEM lanes quad*32 + 16*lh .. +16 and the column
        // block [cb, cb + NCW).  Thread (g, tq) = (lane / 4, lane % 4) holds keys
        // g and g + 8 of that lane half and, of every 8-column repeat, the two
        // columns 2*tq and 2*tq + 1, so its head weights are fixed for the whole
        // CTA and live in registers; the two keys share them.  The sum over the
        // heads finishes with a reduce-scatter over the four lanes of a group:
        // afterwards lane (g, tq) owns key g + 8*(tq >> 1).
        //
        // TMEM is read in 32-column chunks through two register buffers: the
        // load of chunk k+1 is in flight while chunk k is summed, and the first
        // chunk of the next item is loaded before this item's reduce and store.
        constexpr int CPL = C::REPS / 4;      // chunks per lane half
        constexpr int NCH = C::NLH * CPL;     // chunks per item
        static_assert(NCH % 2 == 0, "chunk double buffer");
        const int quad = warp & 3;
        const int j = (warp - 2) >> 2;
        const int lh0 = C::NLH == 1 ? (j & 1) : 0;
        const int cb = (C::NLH == 1 ? (j >> 1) : 0) * C::NCW;
        const int tb = cb / HI; // CTA-local row of the warp's first token
        // candidate mode: this lane's region of each of its rows (the rows of its
        // parity), its counters there and the rows' thresholds
        constexpr int FH = C::TPW >= 2 ? C::TPW / 2 : 1;
        const int region = (quad * 2 + lh0) * 16 + (lane >> 1);
        int wcnt[FH];
        float thr_r[FH];
        uint2 *cbase[FH]; // this lane's region of each of its rows (null past T)
#pragma unroll
        for (int i = 0; i < FH; ++i) {
            wcnt[i] = 0;
            const int lr = tb + (C::TPW >= 2 ? (lane & 1) * FH : 0) + i;
            thr_r[i] = FUSED ? thr_s[lr] : 0.f;
            cbase[i] = (FUSED && r0 + lr < p.T) ? p.cand + ((int64_t)(r0 + lr) * kCandRegions + region) * p.cap
                                                : nullptr;
        }
        const int g = lane >> 2, tq = lane & 3;
        const int b1 = tq >> 1, b0 = tq & 1;
        uint64_t w2[C::REPS];
#pragma unroll
        for (int m = 0; m < C::REPS; ++m) {
            const int c = cb + 8 * m + 2 * tq;
            const float sc = (m % kAbsEvery == kAbsEvery - 1) ? 0.5f : 1.f;
            w2[m] = f32x2_pack(wq_s[c] * sc, wq_s[c + 1] * sc);
        }
        auto chunk_addr = [&](int acc_slot, int k) -> uint32_t {
            const int lh = C::NLH == 1 ? lh0 : k / CPL;
            return tmem + (static_cast<uint32_t>(quad * 32 + 16 * lh) << 16) + acc_slot * C::ACC_COLS + cb +
                   32 * (k % CPL);
        };
        // the key this thread stores for each lane half of tile kt and its scale;
        // a key without storage (past S, or on a missing page) gets INT_MAX, which
        // fails every causal test below
        auto key_info = [&](int kt, int (&sk)[C::NLH], float (&ksc)[C::NLH]) {
#pragma unroll
            for (int l = 0; l < C::NLH; ++l) {
                const int lh = C::NLH == 1 ? lh0 : l;
                const int s = kt * kTileKeys + quad * 32 + 16 * lh + g + 8 * b1;
                bool kok;
                if (!PAGED) {
                    kok = s < p.S;
                    ksc[l] = kok ? p.k_scale[s] : 0.f;
                } else {
                    const int lp = s / p.page_size;
                    const int page = lp < p.max_pages ? p.block_table[(int64_t)r0 * p.max_pages + lp] : -1;
                    kok = page >= 0 && page < p.num_pages;
                    if (!kok && s <= pos_s[0])
                        atomicOr(p.status, DSA_DEV_BAD_PAGE);
                    ksc[l] = kok ? p.k_scale[(int64_t)page * p.page_size + s % p.page_size] : 0.f;
                }
                sk[l] = kok ? s : INT_MAX;
            }
        };
        uint32_t buf0[16], buf1[16];
        // key index and scale of the current item and the next two (loads in flight)
        int skey[C::NLH], skey1[C::NLH];
        float ks[C::NLH], ks1[C::NLH];
        key_info(kt0, skey, ks);
        if (ntiles > 1)
            key_info(kt0 + 1, skey1, ks1);
        bool ok = mbar_wait_warp(accf_bar(0), 0, abort_flag, p.status);
        if (ok) {
            tc_fence_after();
            tmem_ld16x256b_x4(chunk_addr(0, 0), buf0);
        }
        for (int it = 0; ok && it < ntiles; ++it) {
            const int a = it & 1;
            int skey2[C::NLH];
            float ks2[C::NLH];
            if (it + 2 < ntiles)
                key_info(kt0 + it + 2, skey2, ks2);
            uint64_t acc[C::NLH][2][C::TPW];
#pragma unroll
            for (int l = 0; l < C::NLH; ++l)
#pragma unroll
                for (int row = 0; row < 2; ++row)
#pragma unroll
                    for (int t = 0; t < C::TPW; ++t)
                        acc[l][row][t] = 0ull;
#pragma unroll
            for (int k = 0; k < NCH; ++k) {
                uint32_t(&cur)[16] = (k & 1) ? buf1 : buf0;
                uint32_t(&nxt)[16] = (k & 1) ? buf0 : buf1;
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    asm volatile("" : "+r"(cur[i])); // consumers stay behind the wait
                if (k == NCH - 1) {
                    // every chunk of this item is in the warp's registers
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(acce_bar(a));
                }
                if (k + 1 < NCH) {
                    tmem_ld16x256b_x4(chunk_addr(a, k + 1), nxt);
                } else if (it + 1 < ntiles) {
                    if (mbar_wait_warp(accf_bar(a ^ 1), ((it + 1) >> 1) & 1, abort_flag, p.status)) {
                        tc_fence_after();
                        tmem_ld16x256b_x4(chunk_addr(a ^ 1, 0), nxt);
                    } else {
                        ok = false;
                    }
                }
                const int l = k / CPL;
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {
                    const int m = (k % CPL) * 4 + mm;
                    const int tc = m / C::RPT;
#pragma unroll
                    for (int row = 0; row < 2; ++row) {
                        float x0 = __uint_as_float(cur[4 * mm + 2 * row]);
                        float x1 = __uint_as_float(cur[4 * mm + 2 * row + 1]);
                        if (m % kAbsEvery == kAbsEvery - 1) {
                            x0 = x0 + fabsf(x0);
                            x1 = x1 + fabsf(x1);
                        } else {
                            x0 = fmaxf(x0, 0.f);
                            x1 = fmaxf(x1, 0.f);
                        }
                        f32x2_fma(acc[l][row][tc], f32x2_pack(x0, x1), w2[m]);
                    }
                }
            }
#pragma unroll
            for (int l = 0; l < C::NLH; ++l) {
                // reduce-scatter over lanes tq = 0..3: bit 1 picks the key row,
                // bit 0 the half of the token list
                float u[C::TPW];
#pragma unroll
                for (int i = 0; i < C::TPW; ++i) {
                    const float2 e0 = f32x2_unpack(acc[l][0][i]);
                    const float2 e1 = f32x2_unpack(acc[l][1][i]);
                    const float v0 = e0.x + e0.y, v1 = e1.x + e1.y;
                    const float keep = b1 ? v1 : v0;
                    const float send = b1 ? v0 : v1;
                    u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                }
                constexpr int H = C::TPW >= 2 ? C::TPW / 2 : 1;
                float y[H];
                if constexpr (C::TPW >= 2) {
#pragma unroll
                    for (int i = 0; i < H; ++i) {
                        const float keep = b0 ? u[H + i] : u[i];
                        const float send = b0 ? u[i] : u[H + i];
                        y[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                    }
                } else {
                    y[0] = u[0] + __shfl_xor_sync(0xffffffffu, u[0], 1);
                }
                const int s = skey[l];
                if (C::TPW >= 2 || b0 == 0) {
#pragma unroll
                    for (int i = 0; i < H; ++i) {
                        const int lr = tb + (C::TPW >= 2 ? b0 * H : 0) + i;
                        const int rg = r0 + lr;
                        if constexpr (!FUSED) {
                            if (rg < p.T && s <= pos_s[lr])
                                p.logits[(int64_t)rg * p.ld + s] = y[i] * ks[l];
                        } else {
                            const float v = y[i] * ks[l];
                            if (s <= pos_s[lr] && v >= thr_r[i] && cbase[i]) {
                                if (wcnt[i] < p.cap)
                                    cbase[i][wcnt[i]] = make_uint2(__float_as_uint(v), static_cast<uint32_t>(s));
                                ++wcnt[i];
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int l = 0; l < C::NLH; ++l) {
                skey[l] = skey1[l];
                ks[l] = ks1[l];
                skey1[l] = skey2[l];
                ks1[l] = ks2[l];
            }
        }
        tmem_ld_wait(); // no load of this warp outlives the loop
        if constexpr (FUSED) {
#pragma unroll
            for (int i = 0; i < FH; ++i) {
                const int rg = r0 + tb + (lane & 1) * FH + i;
                if (rg < p.T)
                    p.cand_cnt[(int64_t)rg * kCandRegions + region] = wcnt[i];
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int key_in_tile = quad * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        // paged: this thread's key's pool page and scale run two and one tiles
        // ahead (page of tile it + 2 and scale of tile it + 1 loaded during tile
        // it), so no tile waits on the block table
        auto page_of = [&](int it) -> int {
            const int64_t sk = (int64_t)(kt0 + it) * kTileKeys + key_in_tile;
            const int lp = (int)(sk / p.page_size);
            return (it < ntiles && lp < p.max_pages) ? __ldg(p.block_table + (int64_t)r0 * p.max_pages + lp) : -1;
        };
        auto scale_of = [&](int it, int page) -> float {
            const int64_t sk = (int64_t)(kt0 + it) * kTileKeys + key_in_tile;
            return (page >= 0 && page < p.num_pages) ? __ldg(p.k_scale + (int64_t)page * p.page_size + sk % p.page_size)
                                                     : 0.f;
        };
        int pg0 = 0, pg1 = 0;
        float ks0 = 0.f;
        if (PAGED) {
            pg0 = page_of(0);
            pg1 = page_of(1);
            ks0 = scale_of(0, pg0);
        }
        for (int it = 0; it < ntiles; ++it) {
            const int kt = kt0 + it;
            const int64_t s = (int64_t)kt * kTileKeys + key_in_tile;
            float ks = 0.f;
            bool key_ok = true;
            if (!PAGED) {
                key_ok = s < p.S;
                ks = key_ok ? p.k_scale[s] : 0.f;
            } else {
                key_ok = pg0 >= 0 && pg0 < p.num_pages;
                if (!key_ok && s <= pos_s[0] && lane == 0)
                    atomicOr(p.status, DSA_DEV_BAD_PAGE);
                ks = ks0;
                ks0 = scale_of(it + 1, pg1);
                pg0 = pg1;
                pg1 = page_of(it + 2);
            }
            bool ok = true;
            for (int g = 0; g < C::NGROUP; ++g) {
                const int item = it * C::NGROUP + g;
                const int a = item & 1, use = item >> 1;
                if (!mbar_wait_warp(accf_bar(a), use & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int row_base = g * C::G + half * C::TPT; // CTA-local row of token 0
                const uint32_t cbase = lane_base + a * C::ACC_COLS + half * C::NC;
                // all of this thread's columns in flight at once, one wait; the
                // accumulator is released as soon as the values are in registers
                uint32_t r[C::NC];
#pragma unroll
                for (int c0 = 0; c0 < C::NC; c0 += 32)
                    tmem_ld32(cbase + c0, *reinterpret_cast<uint32_t(*)[32]>(r + c0));
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acce_bar(a));
                float acc[C::TPT];
#pragma unroll
                for (int t = 0; t < C::TPT; ++t) {
                    const float4 *w4 = reinterpret_cast<const float4 *>(wq_s + (row_base + t) * HI);
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int h4 = 0; h4 < HI / 4; ++h4) {
                        const float4 wv = w4[h4];
                        const int col = t * HI + 4 * h4;
                        a0 = fmaf(fmaxf(__uint_as_float(r[col]), 0.f), wv.x, a0);
                        a1 = fmaf(fmaxf(__uint_as_float(r[col + 1]), 0.f), wv.y, a1);
                        a0 = fmaf(fmaxf(__uint_as_float(r[col + 2]), 0.f), wv.z, a0);
                        a1 = fmaf(fmaxf(__uint_as_float(r[col + 3]), 0.f), wv.w, a1);
                    }
                    acc[t] = a0 + a1;
                }
                if (key_ok) {
#pragma unroll
                    for (int t = 0; t < C::TPT; ++t) {
                        const int lr = row_base + t;
                        const int r = r0 + lr;
                        if (r < p.T && s <= pos_s[lr])
                            p.logits[(int64_t)r * p.ld + s] = acc[t] * ks;
                    }
                }
            }
            if (!ok)
                break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Paged form for batches of at most kFlatRows rows (decode): a persistent grid
// of two CTAs per SM.  Row r needs key tiles [0, q_pos[r] / 128 + 1); the rows'
// tiles laid end to end form one list, and CTA c takes the contiguous share
// [c * total / C, (c + 1) * total / C), so every CTA scores the same number of
// tiles whatever the context lengths and pays its setup once.  A share crosses
// row boundaries: the query tile (TMA) and the folded head weights of each row
// it touches go through two buffers, so the next row's query loads while the
// current row is scored.  Roles as above: warp 0 loads, warp 1 issues the
// MMAs, warps 2..5 (one per TMEM lane quadrant, one key per thread) reduce
// over the heads.
constexpr int kFlatRows = 1024;

template <int HI, int DI>
struct FlatCfg {
    static constexpr int N = HI;
    static constexpr int NEPI = 4;
    static constexpr int THREADS = 64 + 32 * NEPI;
    static constexpr int NSTAGE = 5;
    static constexpr int QTILE = N * DI;
    static constexpr int KSTAGE = kTileKeys * DI;
    static constexpr int TMEM_COLS = 2 * N <= 64 ? 64 : (2 * N <= 128 ? 128 : 256);
    static constexpr uint32_t SWZ = 2u; // d_I = 128: 128-byte rows, 128-byte swizzle
    static constexpr uint32_t SBO = 8 * DI;
    static constexpr int OFF_Q = 0;                                 // two query tiles
    static constexpr int OFF_K = ((2 * QTILE + 1023) / 1024) * 1024; // key ring
    static constexpr int OFF_W = OFF_K + NSTAGE * KSTAGE;           // [2][HI] folded weights
    static constexpr int OFF_PRE = OFF_W + 2 * HI * 4;              // [kFlatRows + 1] tile prefix
    static constexpr int OFF_SC = ((OFF_PRE + (kFlatRows + 1) * 4 + 127) / 128) * 128; // [NSTAGE][128] key scales
    static constexpr int OFF_SA = OFF_SC + NSTAGE * kTileKeys * 4;  // [2][128] scales of each accumulator's tile
    static constexpr int OFF_BAR = OFF_SA + 2 * kTileKeys * 4;
    static constexpr int NBAR = 2 * NSTAGE + 2 + 2 + 2 + 2 + 2 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024;
    static_assert(DI == 128 && N % 32 == 0 && N >= 32 && N <= 128, "flat indexer shape");
};

// Units of a share: (row r, its tiles [a, b)) in order.
struct FlatUnits {
    int g, g1;
    __device__ FlatUnits(int g0_, int g1_) : g(g0_), g1(g1_) {}
    __device__ bool next(const int *pre, int T, int &r, int &a, int &b)
    {
        if (g >= g1)
            return false;
        int lo = 0, hi = T - 1; // last row with pre[row] <= g: the non-empty row holding tile g
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= g)
                lo = mid;
            else
                hi = mid - 1;
        }
        r = lo;
        const int e = pre[r + 1] < g1 ? pre[r + 1] : g1;
        a = g - pre[r];
        b = e - pre[r];
        g = e;
        return true;
    }
};

template <int HI, int DI>
__global__ void __launch_bounds__(FlatCfg<HI, DI>::THREADS, 2)
    indexer_paged_flat_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_ks, Params p)
{
    using C = FlatCfg<HI, DI>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    float *wq_s = reinterpret_cast<float *>(smem + C::OFF_W);
    int *pre_s = reinterpret_cast<int *>(smem + C::OFF_PRE);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::NSTAGE + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * C::NSTAGE + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * C::NSTAGE + 2 + a); };
    auto qfull_bar = [&](int b) { return bar0 + 8u * (2 * C::NSTAGE + 4 + b); };
    auto qempty_bar = [&](int b) { return bar0 + 8u * (2 * C::NSTAGE + 6 + b); };
    auto sready_bar = [&](int a) { return bar0 + 8u * (2 * C::NSTAGE + 8 + a); };
    const uint32_t done_bar = bar0 + 8u * (2 * C::NSTAGE + 10);
    // key scales: each stage's, copied by the TMA beside the keys, then each
    // accumulator's, copied there by the MMA warp for the epilogue
    float *sc_stage = reinterpret_cast<float *>(smem + C::OFF_SC);
    float *sc_acc = reinterpret_cast<float *>(smem + C::OFF_SA);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    int *pos_s = reinterpret_cast<int *>(smem + C::OFF_MISC + 8); // [2]: position of the row in each buffer

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t key_limit = (int64_t)p.max_pages * p.page_size;
    const int64_t lim = (key_limit < p.ld ? key_limit : p.ld) - 1;
    auto clamp_pos = [&](int r) -> int {
        int64_t qp = p.q_pos[r];
        if (qp > lim)
            qp = lim;
        return qp < 0 ? -1 : static_cast<int>(qp);
    };

    grid_dep_wait();
    grid_dep_launch();
    // ---- tile prefix over the rows (warp 0; lane l sums rows [l * per, l * per + per))
    if (warp == 0) {
        const int per = (p.T + 31) / 32;
        int cnt = 0;
        for (int i = 0; i < per; ++i) {
            const int r = lane * per + i;
            if (r < p.T) {
                if (blockIdx.x == 0 && p.q_pos[r] > lim)
                    atomicOr(p.status, DSA_DEV_BAD_POSITION);
                const int pos = clamp_pos(r);
                cnt += pos < 0 ? 0 : pos / kTileKeys + 1;
            }
        }
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        int run = x - cnt;
        for (int i = 0; i < per; ++i) {
            const int r = lane * per + i;
            if (r < p.T) {
                pre_s[r] = run;
                const int pos = clamp_pos(r);
                run += pos < 0 ? 0 : pos / kTileKeys + 1;
            }
        }
        if (lane == 31)
            pre_s[p.T] = x;
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), C::NEPI);
            mbar_init(qfull_bar(a), 1);
            mbar_init(qempty_bar(a), 1 + C::NEPI); // the MMAs of the row, then each epilogue warp
            mbar_init(sready_bar(a), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int total = pre_s[p.T];
    const int g0 = static_cast<int>((int64_t)blockIdx.x * total / gridDim.x);
    const int g1 = static_cast<int>((int64_t)(blockIdx.x + 1) * total / gridDim.x);
    if (g1 <= g0)
        return; // uniform: an empty share

    if (warp == 1)
        tmem_alloc(sbase + C::OFF_MISC, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    FlatUnits units(g0, g1);
    int r = 0, ta = 0, tb = 0;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
        }
        int it = 0, u = 0;
        bool ok = true;
        while (ok && units.next(pre_s, p.T, r, ta, tb)) {
            const int qb = u & 1;
            if (u >= 2 && !mbar_wait_warp(qempty_bar(qb), ((u >> 1) - 1) & 1, abort_flag, p.status))
                break;
            const float qs = p.q_scale[r];
            for (int h = lane; h < HI; h += 32)
                wq_s[qb * HI + h] = p.w[(int64_t)r * HI + h] * qs;
            if (lane == 0)
                pos_s[qb] = clamp_pos(r);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(qfull_bar(qb), C::QTILE);
                tma_load_2d(sbase + C::OFF_Q + qb * C::QTILE, &tm_q, qfull_bar(qb), 0, r * HI);
            }
            ++u;
            // lane j holds the pool page of logical page bt_base + j
            int bt_base = INT_MIN / 2, bt_page = -1;
            const int per_tile = kTileKeys / p.page_size;
            for (int kt = ta; kt < tb; ++kt, ++it) {
                const int s = it % C::NSTAGE;
                const int lp0 = (kt * kTileKeys) / p.page_size;
                if (lp0 < bt_base || lp0 + per_tile > bt_base + 32) {
                    bt_base = lp0;
                    const int lp = lp0 + lane;
                    bt_page = lp < p.max_pages ? __ldg(p.block_table + (int64_t)r * p.max_pages + lp) : -1;
                }
                if (it >= C::NSTAGE &&
                    !mbar_wait_warp(empty_bar(s), ((it / C::NSTAGE) - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = sbase + C::OFF_K + s * C::KSTAGE;
                const uint32_t sdst = smem_u32(sc_stage + s * kTileKeys);
                if (lane == 0)
                    mbar_arrive_expect_tx(full_bar(s), C::KSTAGE + kTileKeys * 4);
                for (int j = 0; j < per_tile; ++j) {
                    const int page = __shfl_sync(0xffffffffu, bt_page, lp0 + j - bt_base);
                    // an invalid page loads rows past the pool: TMA fills the codes and the
                    // scales with zeros, and a zero scale makes the epilogue skip the key
                    const bool pok = page >= 0 && page < p.num_pages;
                    const int row = pok ? page * p.page_size : p.num_pages * p.page_size;
                    if (lane == 0) {
                        tma_load_2d(dst + j * p.page_size * DI, &tm_k, full_bar(s), 0, row);
                        tma_load_2d(sdst + j * p.page_size * 4, &tm_ks, full_bar(s), 0, pok ? page : p.num_pages);
                    }
                }
                __syncwarp();
            }
        }
        // drain: every load issued has landed before the CTA exits
        if (lane == 0) {
            for (int v = u - 2 > 0 ? u - 2 : 0; v < u; ++v)
                mbar_drain(qfull_bar(v & 1), (v >> 1) & 1);
            for (int i = it - C::NSTAGE > 0 ? it - C::NSTAGE : 0; i < it; ++i)
                mbar_drain(full_bar(i % C::NSTAGE), (i / C::NSTAGE) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_f32acc(128, C::N, 0u, false, false);
        int it = 0, u = 0;
        bool ok = true;
        while (ok && units.next(pre_s, p.T, r, ta, tb)) {
            const int qb = u & 1;
            if (!mbar_wait_warp(qfull_bar(qb), (u >> 1) & 1, abort_flag, p.status))
                break;
            for (int kt = ta; kt < tb; ++kt, ++it) {
                const int s = it % C::NSTAGE;
                const int acc = it & 1, use = it >> 1;
                if (!mbar_wait_warp(full_bar(s), (it / C::NSTAGE) & 1, abort_flag, p.status) ||
                    (use >= 1 && !mbar_wait_warp(acce_bar(acc), (use - 1) & 1, abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the tile's key scales go with its accumulator (the epilogue released
                // this slot's previous scales together with the accumulator)
                reinterpret_cast<float4 *>(sc_acc + acc * kTileKeys)[lane] =
                    reinterpret_cast<const float4 *>(sc_stage + s * kTileKeys)[lane];
                __syncwarp();
                if (lane == 0) {
                    const uint32_t abase = sbase + C::OFF_K + s * C::KSTAGE;
                    const uint32_t bbase = sbase + C::OFF_Q + qb * C::QTILE;
#pragma unroll
                    for (int kk = 0; kk < DI / 32; ++kk) {
                        const uint64_t ad = sdesc(abase + kk * 32, 16, C::SBO, C::SWZ);
                        const uint64_t bd = sdesc(bbase + kk * 32, 16, C::SBO, C::SWZ);
                        umma_f8f6f4(tmem + acc * C::N, ad, bd, idesc, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(accf_bar(acc));
                    mbar_arrive(sready_bar(acc));
                    umma_commit(empty_bar(s));
                }
                __syncwarp();
            }
            if (lane == 0)
                umma_commit(qempty_bar(qb)); // the query tile is free once these MMAs complete
            __syncwarp();
            ++u;
        }
        if (lane == 0) {
            umma_commit(done_bar);
            mbar_drain(done_bar, 0);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int key_in_tile = quad * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        int it = 0, u = 0;
        bool ok = true;
        while (ok && units.next(pre_s, p.T, r, ta, tb)) {
            const int qb = u & 1;
            if (!mbar_wait_warp(qfull_bar(qb), (u >> 1) & 1, abort_flag, p.status))
                break;
            const int pos = pos_s[qb];
            const float4 *w4 = reinterpret_cast<const float4 *>(wq_s + qb * HI);
            for (int kt = ta; kt < tb; ++kt, ++it) {
                const int64_t s = (int64_t)kt * kTileKeys + key_in_tile;
                const int acc = it & 1, use = it >> 1;
                if (!mbar_wait_warp(accf_bar(acc), use & 1, abort_flag, p.status) ||
                    !mbar_wait_warp(sready_bar(acc), use & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                // the key's scale (zero for a key on a page outside the pool)
                const float ks = sc_acc[acc * kTileKeys + key_in_tile];
                const bool key_ok = ks > 0.f;
                if (!key_ok && s <= pos && lane == 0)
                    atomicOr(p.status, DSA_DEV_BAD_PAGE);
                tc_fence_after();
                uint32_t v[HI];
#pragma unroll
                for (int c0 = 0; c0 < HI; c0 += 32)
                    tmem_ld32(lane_base + acc * C::N + c0, *reinterpret_cast<uint32_t(*)[32]>(v + c0));
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acce_bar(acc));
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int h4 = 0; h4 < HI / 4; ++h4) {
                    const float4 wv = w4[h4];
                    a0 = fmaf(fmaxf(__uint_as_float(v[4 * h4]), 0.f), wv.x, a0);
                    a1 = fmaf(fmaxf(__uint_as_float(v[4 * h4 + 1]), 0.f), wv.y, a1);
                    a0 = fmaf(fmaxf(__uint_as_float(v[4 * h4 + 2]), 0.f), wv.z, a0);
                    a1 = fmaf(fmaxf(__uint_as_float(v[4 * h4 + 3]), 0.f), wv.w, a1);
                }
                if (key_ok && s <= pos)
                    p.logits[(int64_t)r * p.ld + s] = (a0 + a1) * ks;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(qempty_bar(qb)); // done with this buffer's weights and position
            ++u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int HI, int DI, bool PAGED>
int launch_cfg(const IndexerArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    using C = IdxCfg<HI, DI, PAGED>;
    static std::atomic<bool> attr_set[64];
    if (cudaError_t e_attr = raise_smem_limit_once(indexer_kernel<HI, DI, PAGED>, C::SMEM, attr_set);
        e_attr != cudaSuccess) {
        snprintf(err, errlen, "cudaFuncSetAttribute(indexer): %s", cudaGetErrorString(e_attr));
        return DSA_ERR_CUDA;
    }
    const CUtensorMapSwizzle swz = DI == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                             : (DI == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    CUtensorMap tq, tk;
    if (!encode_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q8, DI, (uint64_t)a.T * HI, DI, DI, C::N, swz, err,
                        errlen))
        return DSA_ERR_CUDA;
    if (!PAGED) {
        if (!encode_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k8, DI, (uint64_t)a.S, DI, DI, kTileKeys, swz, err,
                            errlen))
            return DSA_ERR_CUDA;
    } else {
        if (!encode_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k8, DI, (uint64_t)a.num_pages * a.page_size, DI,
                            DI, a.page_size, swz, err, errlen))
            return DSA_ERR_CUDA;
    }
    Params p;
    p.q_scale = a.q_scale;
    p.w = a.w;
    p.k_scale = a.k_scale;
    p.q_pos = a.q_pos;
    p.block_table = a.block_table;
    p.logits = a.logits;
    p.ld = a.ld;
    p.T = a.T;
    p.S = a.S;
    p.max_pages = a.max_pages;
    p.num_pages = a.num_pages;
    p.page_size = a.page_size;
    p.thr = a.thr;
    p.cand = a.cand;
    p.cand_cnt = a.cand_cnt;
    p.cap = a.cap;
    p.row_flag = a.row_flag;
    p.status = device_status_ptr();
    if (!p.status) {
        snprintf(err, errlen, "device status word unavailable");
        return DSA_ERR_CUDA;
    }
    if constexpr (PAGED && DI == 128 && (HI == 64 || HI == 32)) {
        // decode-sized batches: the persistent flat schedule (tile counts fit int)
        const int64_t keys = (int64_t)a.max_pages * a.page_size < a.ld ? (int64_t)a.max_pages * a.page_size : a.ld;
        // (the key scales travel by TMA, which wants a 16-byte aligned base)
        if (a.T <= kFlatRows && (int64_t)a.T * ((keys + kTileKeys - 1) / kTileKeys) < INT_MAX &&
            (reinterpret_cast<uintptr_t>(a.k_scale) & 15u) == 0) {
            using F = FlatCfg<HI, DI>;
            CUtensorMap tks; // k_scale as [num_pages, page_size] fp32, one page per box
            if (!encode_tmap_2d(&tks, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.k_scale, a.page_size, a.num_pages,
                                (uint64_t)a.page_size * 4, a.page_size, 1, CU_TENSOR_MAP_SWIZZLE_NONE, err, errlen))
                return DSA_ERR_CUDA;
            static std::atomic<bool> flat_attr[64];
            if (cudaError_t e_attr = raise_smem_limit_once(indexer_paged_flat_kernel<HI, DI>, F::SMEM, flat_attr);
                e_attr != cudaSuccess) {
                snprintf(err, errlen, "cudaFuncSetAttribute(indexer flat): %s", cudaGetErrorString(e_attr));
                return DSA_ERR_CUDA;
            }
            p.splits = 1;
            cudaError_t e = launch_pdl(indexer_paged_flat_kernel<HI, DI>, dim3(2 * num_sms()), dim3(F::THREADS),
                                       F::SMEM, stream, 1, tq, tk, tks, p);
            if (e != cudaSuccess) {
                snprintf(err, errlen, "indexer launch: %s", cudaGetErrorString(e));
                return DSA_ERR_CUDA;
            }
            return DSA_OK;
        }
    }
    const int groups = (a.T + C::R - 1) / C::R;
    int splits = 1;
    if (PAGED) {
        // enough CTAs for ~4 per SM over the batch; tiles per split follow each row's length
        const int target = 4 * num_sms();
        splits = (target + groups - 1) / groups;
        if (splits < 1) splits = 1;
        if (splits > 64) splits = 64;
    }
    p.splits = splits;
    dim3 grid(groups, splits);
    cudaError_t e;
    if constexpr (C::FRAG && C::R <= 8) {
        if (a.cand) {
            static std::atomic<bool> fused_attr[64];
            if (cudaError_t e_attr = raise_smem_limit_once(indexer_kernel<HI, DI, PAGED, true>, C::SMEM, fused_attr);
                e_attr != cudaSuccess) {
                snprintf(err, errlen, "cudaFuncSetAttribute(indexer candidates): %s", cudaGetErrorString(e_attr));
                return DSA_ERR_CUDA;
            }
            e = launch_pdl(indexer_kernel<HI, DI, PAGED, true>, grid, dim3(C::THREADS), C::SMEM, stream, 1, tq, tk, p);
            if (e != cudaSuccess) {
                snprintf(err, errlen, "indexer launch: %s", cudaGetErrorString(e));
                return DSA_ERR_CUDA;
            }
            return DSA_OK;
        }
    }
    if (a.cand) {
        snprintf(err, errlen, "indexer: candidate mode needs contiguous keys and H_I in {32, 64}");
        return DSA_ERR_UNSUPPORTED;
    }
    e = launch_pdl(indexer_kernel<HI, DI, PAGED>, grid, dim3(C::THREADS), C::SMEM, stream, 1, tq, tk, p);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "indexer launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

} // namespace

int launch_indexer(const IndexerArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    const bool paged = a.block_table != nullptr;
    if (a.HI == 64 && a.dI == 128)
        return paged ? launch_cfg<64, 128, true>(a, stream, err, errlen) : launch_cfg<64, 128, false>(a, stream, err, errlen);
    if (a.HI == 32 && a.dI == 128)
        return paged ? launch_cfg<32, 128, true>(a, stream, err, errlen) : launch_cfg<32, 128, false>(a, stream, err, errlen);
    if (a.HI == 4 && a.dI == 32 && !paged)
        return launch_cfg<4, 32, false>(a, stream, err, errlen);
    snprintf(err, errlen, "indexer: unsupported (H_I=%d, d_I=%d, %s)", a.HI, a.dI, paged ? "paged" : "contiguous");
    return DSA_ERR_UNSUPPORTED;
}

} // namespace dsa
