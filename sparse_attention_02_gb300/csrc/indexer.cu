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
// With keys on the lanes, the sum over heads is a loop over the columns a
// thread reads from its own TMEM lane, and the 32 threads of a warp store 32
// consecutive keys of a logits row (128 coalesced bytes).
//
// Roles (one CTA, warp-specialised):
//   warp 0      TMA producer: the CTA's query tiles once, then key tiles
//               through an NSTAGE ring (paged: one TMA per page of the tile).
//   warp 1      TMEM allocator and MMA issuer (one elected lane).
//   warps 2..   epilogue, up to four warps per TMEM lane quadrant: TMEM ->
//               registers (all columns in flight, one wait), ReLU, weighted
//               head sum (w read as float4 broadcasts), key scale, masked
//               store.  Two TMEM accumulators alternate so the MMA of one item
//               overlaps the epilogue of the other.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

constexpr int kTileKeys = 128;

template <int HI, int DI, bool PAGED>
struct IdxCfg {
    static constexpr int G = PAGED ? 1 : 256 / HI;        // tokens per accumulator
    static constexpr int NGROUP = PAGED ? 1 : 2;          // token groups sharing a key tile
    static constexpr int R = G * NGROUP;                  // query rows per CTA
    static constexpr int N = G * HI;                      // MMA N
    static constexpr int EPI_SPLIT = N >= 256 ? 4 : (N >= 128 ? 2 : 1); // warps per TMEM lane quadrant
    static constexpr int NEPI = 4 * EPI_SPLIT;            // epilogue warps
    static constexpr int THREADS = 64 + 32 * NEPI;
    static constexpr int NSTAGE = PAGED ? 6 : 4;
    static constexpr int NC = N / EPI_SPLIT;              // TMEM columns per epilogue thread
    static constexpr int TPT = NC / HI;                   // tokens per epilogue thread
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
    static_assert(NC % 32 == 0 && NC % HI == 0, "epilogue split");
    static_assert(DI == 32 || DI == 64 || DI == 128, "d_I");
};

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
};

template <int HI, int DI, bool PAGED>
__global__ void __launch_bounds__(IdxCfg<HI, DI, PAGED>::THREADS, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, Params p)
{
    using C = IdxCfg<HI, DI, PAGED>;
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
            mbar_init(acce_bar(a), C::NEPI * 32);
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
    if (kt1 <= kt0)
        return; // uniform: nothing to score in this split

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
        for (int it = 0; it < ntiles; ++it) {
            const int s = it % C::NSTAGE;
            if (it >= C::NSTAGE &&
                !mbar_wait_warp(empty_bar(s), ((it / C::NSTAGE) - 1) & 1, abort_flag, p.status))
                break;
            if (lane == 0) {
                const int kt = kt0 + it;
                const uint32_t dst = sbase + C::OFF_K + s * C::KSTAGE;
                mbar_arrive_expect_tx(full_bar(s), C::KSTAGE);
                if (!PAGED) {
                    tma_load_2d(dst, &tm_k, full_bar(s), 0, kt * kTileKeys);
                } else {
                    const int per_tile = kTileKeys / p.page_size;
                    for (int j = 0; j < per_tile; ++j) {
                        const int lp = (kt * kTileKeys) / p.page_size + j;
                        int page = lp < p.max_pages ? p.block_table[(int64_t)r0 * p.max_pages + lp] : -1;
                        // An invalid page loads out-of-range rows: TMA fills zeros and
                        // the epilogue skips those keys.
                        const int row = (page >= 0 && page < p.num_pages) ? page * p.page_size
                                                                          : p.num_pages * p.page_size;
                        tma_load_2d(dst + j * p.page_size * DI, &tm_k, full_bar(s), 0, row);
                    }
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
    } else {
        // --------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int key_in_tile = quad * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        for (int it = 0; it < ntiles; ++it) {
            const int kt = kt0 + it;
            const int64_t s = (int64_t)kt * kTileKeys + key_in_tile;
            float ks = 0.f;
            bool key_ok = true;
            if (!PAGED) {
                key_ok = s < p.S;
                ks = key_ok ? p.k_scale[s] : 0.f;
            } else {
                const int lp = (int)(s / p.page_size);
                const int page = lp < p.max_pages ? p.block_table[(int64_t)r0 * p.max_pages + lp] : -1;
                key_ok = page >= 0 && page < p.num_pages;
                if (!key_ok && s <= pos_s[0] && lane == 0)
                    atomicOr(p.status, DSA_DEV_BAD_PAGE);
                ks = key_ok ? p.k_scale[(int64_t)page * p.page_size + s % p.page_size] : 0.f;
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

template <int HI, int DI, bool PAGED>
int launch_cfg(const IndexerArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    using C = IdxCfg<HI, DI, PAGED>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(indexer_kernel<HI, DI, PAGED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) {
            snprintf(err, errlen, "cudaFuncSetAttribute(indexer): %s", cudaGetErrorString(e));
            return DSA_ERR_CUDA;
        }
        attr_set[dev] = true;
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
    p.status = device_status_ptr();
    if (!p.status) {
        snprintf(err, errlen, "device status word unavailable");
        return DSA_ERR_CUDA;
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
    indexer_kernel<HI, DI, PAGED><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, p);
    cudaError_t e = cudaGetLastError();
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
