// Fused lightning indexer -> top-k on sm_103a: the top-k of every query row's
// index scores without the scores ever reaching memory.
//
// Defines the same result as dsa_indexer_logits followed by dsa_topk (release
// summary "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency with DeepSeek
// Sparse Attention", section "Method": index scores against all prior tokens,
// then the top-k of them; "AMD Instinct MI355X GPUs Power DeepSeek-V3.2-Exp",
// section "Computational Efficiency": attention cost goes from O(L^2) to
// O(Lk), which at long context leaves the indexer's L^2 scores as the quadratic
// part).  Written out, a row of L keys costs 4 L bytes of scores to write and
// read back; the fused path keeps ~1.25k + 256 of them.
//
// Steps, all on the caller's stream:
//   1. gather      the keys at a fixed stride over [0, S): nsamp sample keys
//                  (sample_count) p_j = floor(j S / nsamp), and for every row
//                  the last sample at or before its position;
//   2. indexer     the rows' scores against the samples (the same kernel and
//                  arithmetic as dsa_indexer_logits, samples as keys);
//   3. threshold   per row, a score about 1.25k + 256 of the row's keys reach
//                  (topk_threshold_kernel); -inf for rows of at most cap keys;
//   4. indexer     candidate mode: every key scoring at or above its row's
//                  threshold is appended to the row's list (score, position);
//                  no scores are written;
//   5. select      exact top-k of each list, ascending positions
//                  (topk_candidates_kernel); a row whose count missed [k, cap]
//                  is flagged;
//   6. indexer     full scores for the flagged rows only (CTAs without one exit);
//   7. top-k       the row kernel of dsa_topk on those rows only.
// Steps 6 and 7 find nothing to do unless a row's samples misled its
// threshold; either way every row's result is that of the two-call path.
#include "common.cuh"
#include "launch.h"

#include <stdio.h>

namespace dsa {
namespace {

// Sampled keys: 2048, or S / 32 for prefixes past 65536 keys (a row of n keys
// then sees about 2048 n / S of them, and the rank its threshold sits at,
// r ~ (1.25 k + 256) * samples / S, stays near 90 or more: the candidate count
// misses [k, cap] for a row like its samples with a probability of the order
// of 1e-2 at the smallest r and far less above; sampling costs ~3 % of the
// indexer's work).
int sample_count(int S) { return S <= 2048 ? S : (S / 32 > 2048 ? S / 32 : 2048); }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A row's candidate list holds at most cap_for(k) entries for the select; the
// indexer writes it as 128 per-lane regions of cap_for(k) / 64 entries (about
// three times what a lane finds at the threshold).
int cap_for(int k) { return 2 * k > 4096 ? 2 * k : 4096; }
constexpr int kLaneRegions = 128;

struct Layout {
    size_t k8s, kss, qpos_s, vlen, samp, thr, cand, cand_cnt, flag, fb_logits, total;
};

Layout layout(int T, int S, int dI, int k)
{
    const int nsamp = sample_count(S);
    const size_t cap = static_cast<size_t>(cap_for(k));
    Layout l;
    size_t o = 0;
    l.k8s = o;
    o += align256(static_cast<size_t>(nsamp) * dI);
    l.kss = o;
    o += align256(static_cast<size_t>(nsamp) * 4);
    l.qpos_s = o;
    o += align256(static_cast<size_t>(T) * 4);
    l.vlen = o;
    o += align256(static_cast<size_t>(T) * 4);
    l.samp = o;
    o += align256(static_cast<size_t>(T) * nsamp * 4);
    l.thr = o;
    o += align256(static_cast<size_t>(T) * 4);
    l.cand = o;
    o += align256(static_cast<size_t>(T) * kLaneRegions * (cap / 64) * 8);
    l.cand_cnt = o;
    o += align256(static_cast<size_t>(T) * kLaneRegions * 4); // per row, one count per list region
    l.flag = o;
    o += align256(static_cast<size_t>(T) * 4);
    l.fb_logits = o;
    o += align256(static_cast<size_t>(T) * S * 4);
    l.total = o;
    return l;
}

// Sample keys (codes and scales) at p_j = floor(j S / nsamp), and per row the
// index of its last sample at or before min(q_pos, S - 1) (-1 for none):
// p_j <= q  <=>  j <= floor((nsamp (q + 1) - 1) / S); and the row's key count
// min(q_pos + 1, S) for the top-k of the flagged rows.
__global__ void __launch_bounds__(256)
    sample_keys_kernel(const uint8_t *__restrict__ k8, const float *__restrict__ k_scale, int S, int dI, int nsamp,
                       const int32_t *__restrict__ q_pos, int T, uint8_t *__restrict__ k8s, float *__restrict__ kss,
                       int32_t *__restrict__ qpos_s, int32_t *__restrict__ vlen)
{
    grid_dep_wait();
    grid_dep_launch();
    const int chunks = dI / 16; // 16-byte pieces of a key row
    const int64_t nkey = static_cast<int64_t>(nsamp) * chunks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nkey + nsamp + T;
         i += stride) {
        if (i < nkey) {
            const int j = static_cast<int>(i / chunks), c = static_cast<int>(i % chunks);
            const int64_t pj = static_cast<int64_t>(j) * S / nsamp;
            reinterpret_cast<uint4 *>(k8s + static_cast<int64_t>(j) * dI)[c] =
                __ldg(reinterpret_cast<const uint4 *>(k8 + pj * dI) + c);
        } else if (i < nkey + nsamp) {
            const int j = static_cast<int>(i - nkey);
            kss[j] = __ldg(k_scale + static_cast<int64_t>(j) * S / nsamp);
        } else {
            const int t = static_cast<int>(i - nkey - nsamp);
            int64_t q = q_pos[t];
            q = q > S - 1 ? S - 1 : q;
            int64_t js = q < 0 ? -1 : (static_cast<int64_t>(nsamp) * (q + 1) - 1) / S;
            js = js > nsamp - 1 ? nsamp - 1 : js;
            qpos_s[t] = static_cast<int32_t>(js);
            vlen[t] = static_cast<int32_t>(q < 0 ? 0 : q + 1);
        }
    }
}

} // namespace

size_t indexer_topk_workspace_bytes(int T, int S, int dI, int k) { return layout(T, S, dI, k).total; }

int launch_indexer_topk(const IndexerTopkArgs &a, cudaStream_t stream, char *err, size_t errlen)
{
    const Layout l = layout(a.T, a.S, a.dI, a.k);
    if (!a.workspace || a.workspace_bytes < l.total) {
        snprintf(err, errlen, "workspace too small for the fused indexer -> top-k (%zu bytes needed)", l.total);
        return DSA_ERR_WORKSPACE;
    }
    const int cap = cap_for(a.k);
    if (topk_candidates_smem(a.S, cap) > 232448 - 2048) {
        snprintf(err, errlen, "fused indexer -> top-k: S = %d is beyond its shared-memory bitmaps", a.S);
        return DSA_ERR_UNSUPPORTED;
    }
    char *ws = static_cast<char *>(a.workspace);
    uint8_t *k8s = reinterpret_cast<uint8_t *>(ws + l.k8s);
    float *kss = reinterpret_cast<float *>(ws + l.kss);
    int32_t *qpos_s = reinterpret_cast<int32_t *>(ws + l.qpos_s);
    int32_t *vlen = reinterpret_cast<int32_t *>(ws + l.vlen);
    float *samp = reinterpret_cast<float *>(ws + l.samp);
    float *thr = reinterpret_cast<float *>(ws + l.thr);
    uint2 *cand = reinterpret_cast<uint2 *>(ws + l.cand);
    int32_t *cand_cnt = reinterpret_cast<int32_t *>(ws + l.cand_cnt);
    int32_t *flag = reinterpret_cast<int32_t *>(ws + l.flag);
    float *fb_logits = reinterpret_cast<float *>(ws + l.fb_logits);
    const int nsamp = sample_count(a.S);

    // 1. sample keys and per-row sample positions
    const int64_t items = static_cast<int64_t>(nsamp) * (a.dI / 16) + nsamp + a.T;
    int blocks = static_cast<int>((items + 255) / 256);
    blocks = blocks > 4 * num_sms() ? 4 * num_sms() : blocks;
    cudaError_t e = launch_pdl(sample_keys_kernel, dim3(blocks), dim3(256), 0, stream, 1,
                               static_cast<const uint8_t *>(a.k8), a.k_scale, a.S, a.dI, nsamp, a.q_pos, a.T, k8s, kss,
                               qpos_s, vlen);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "sample keys launch: %s", cudaGetErrorString(e));
        return DSA_ERR_CUDA;
    }
    // 2. scores against the samples
    IndexerArgs is{a.q8, a.q_scale, a.w, a.T, a.HI, a.dI, k8s, kss, nsamp, nullptr, 0, 0, 0, qpos_s, samp, nsamp};
    int rc = launch_indexer(is, stream, err, errlen);
    if (rc != DSA_OK)
        return rc;
    // 3. per-row thresholds
    rc = launch_topk_threshold(samp, nsamp, a.T, a.q_pos, qpos_s, a.S, a.k, cap, thr, stream, err, errlen);
    if (rc != DSA_OK)
        return rc;
    // 4. candidates
    IndexerArgs ic{a.q8, a.q_scale, a.w, a.T, a.HI, a.dI, a.k8, a.k_scale, a.S, nullptr, 0, 0, 0, a.q_pos,
                   fb_logits, a.S};
    ic.thr = thr;
    ic.cand = cand;
    ic.cand_cnt = cand_cnt;
    ic.cap = cap / 64; // entries per lane region
    rc = launch_indexer(ic, stream, err, errlen);
    if (rc != DSA_OK)
        return rc;
    // 5. exact top-k of the candidates; rows whose count missed [k, cap] flagged
    rc = launch_topk_candidates(cand, cand_cnt, cap, a.T, a.q_pos, a.S, a.k, a.idx, flag, stream, err, errlen);
    if (rc != DSA_OK)
        return rc;
    // 6-7. the flagged rows from full scores
    IndexerArgs ifb{a.q8, a.q_scale, a.w, a.T, a.HI, a.dI, a.k8, a.k_scale, a.S, nullptr, 0, 0, 0, a.q_pos,
                    fb_logits, a.S};
    ifb.row_flag = flag;
    rc = launch_indexer(ifb, stream, err, errlen);
    if (rc != DSA_OK)
        return rc;
    TopkArgs tk{fb_logits, a.S, a.T, vlen, a.k, a.idx};
    tk.row_flag = flag;
    return launch_topk(tk, stream, err, errlen);
}

} // namespace dsa
