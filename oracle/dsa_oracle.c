/*
 * DSA oracle: TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of DeepSeek Sparse Attention (DSA) as the
 * pages define it:
 *   - "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency with DeepSeek Sparse
 *     Attention" (release summary), section "Method": the index score
 *     I[t,s] = sum_j w[t,j] * ReLU(q[t,j] . k[s]) against all prior tokens, a
 *     top-k (k = 2048) selection per query, and MLA attention in MQA mode that
 *     reads only the selected latent-KV rows (one latent row shared by every
 *     query head of the token).
 *   - "AMD Instinct MI355X GPUs Power DeepSeek-V3.2-Exp", section "DeepSeek
 *     Sparse Attention (DSA)": lightning indexer in FP8 over a few heads, then
 *     fine-grained top-2048 token selection feeding the main attention.
 *   - the same release summary, "Key claims": the high-performance kernels come
 *     as indexer-logit kernels "incl. paged versions" and sparse-attention
 *     kernels, which is why paged variants exist here.
 *
 * Nothing here is tiled, fused or reordered beyond the definition: every
 * quantity is computed from its formula in fp64 after decoding the stored FP8
 * and BF16 bits with this file's own decoders.  Rows (and heads) are
 * independent, so any subset of query rows can be computed exactly; OpenMP
 * only splits independent loops (the keys of an index row, rows and heads of
 * attention).
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Readings of points the pages leave open (each one is listed in the design
 * notes):
 *   causal bound      a query at absolute position t scores keys s in [0, t]
 *                     (the token itself included);
 *   FP8 scales        one positive fp32 scale per token for q (over all heads)
 *                     and one per key token for k; dequantised value =
 *                     code * scale;
 *   top-k order       larger score first, then smaller index; -0 equals +0;
 *                     the selected indices are returned in ascending order,
 *                     padded with -1 when fewer than k candidates exist;
 *   attention         softmax over the valid selected rows of
 *                     sm_scale * <Q[t,h,:D], KV[s,:D]>, output uses the first
 *                     Dv columns of the same latent row as V; LSE is the
 *                     natural log of the softmax denominator;
 *   invalid entries   prefill: an index outside [0, S) is skipped; paged: a
 *                     logical position outside [0, ctx_len) or a page id
 *                     outside [0, num_pages) is skipped.  A row with nothing
 *                     valid gives O = 0 and LSE = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- decoders */

/* FP8 E4M3 ("fn" variant, the FP8 format the indexer runs in): 1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits, subnormals when the exponent
 * field is 0, no infinities, and S.1111.111 is NaN.  Largest finite value is
 * 1.75 * 2^8 = 448. */
double dsa_oracle_e4m3(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int ex = (code >> 3) & 15;
    int man = code & 7;
    double mag;
    if (ex == 15 && man == 7)
        return NAN;
    if (ex == 0)
        mag = ldexp((double)man / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return sign ? -mag : mag;
}

/* BF16: the upper 16 bits of an IEEE-754 binary32. */
double dsa_oracle_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int dsa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------- per-token FP8 quantiser
 * The indexer runs in FP8 ("AMD Instinct MI355X GPUs Power DeepSeek-V3.2-Exp",
 * "DeepSeek Sparse Attention (DSA)", item 1; release summary, "Method"), with
 * one scale per token; the gist page's indexer test script casts along chosen
 * dimensions to E4M3 with an option for power-of-two ("UE8M0") scales.  The
 * formulas are not printed; the readings taken here:
 *   mode 0   scale = fp32(amax / 448), or 1 when the row is all zero;
 *   mode 1   scale = the smallest power of two not below fp32(amax / 448),
 *            or 1 when the row is all zero;
 *   code     E4M3 nearest to fp32(x / scale), ties to the even code,
 *            magnitudes above 448 saturate to 448.
 * The divisions are single-precision on purpose: the code is an integer that a
 * rounding decides, so both sides take that decision in the kernel's precision.
 */

/* E4M3 code of a finite value: binary search of |v| among the 127 ordered
 * non-negative finite codes (the decoder above gives their values), nearest
 * wins, a tie goes to the code with an even mantissa (even code). */
uint8_t dsa_oracle_e4m3_encode(float v)
{
    if (isnan(v))
        return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 126; /* dsa_oracle_e4m3(lo) <= a < dsa_oracle_e4m3(hi) */
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (dsa_oracle_e4m3((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    const double dlo = a - dsa_oracle_e4m3((uint8_t)lo);
    const double dhi = dsa_oracle_e4m3((uint8_t)hi) - a;
    int code;
    if (dlo < dhi)
        code = lo;
    else if (dhi < dlo)
        code = hi;
    else
        code = (lo % 2 == 0) ? lo : hi;
    return (uint8_t)(sign | code);
}

/* Rows of cols fp32 values -> E4M3 codes [rows, cols] and one fp32 scale per row. */
void dsa_oracle_quantize_fp8(const float *x, int64_t rows, int64_t cols, int mode, uint8_t *codes, float *scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        float amax = 0.f;
        for (int64_t c = 0; c < cols; ++c) {
            const float m = fabsf(xr[c]);
            if (m > amax)
                amax = m;
        }
        float s = 1.f;
        if (amax > 0.f) {
            const float ratio = amax / 448.f;
            if (mode == 0) {
                s = ratio;
            } else {
                int e;
                const double f = frexp((double)ratio, &e); /* ratio = f * 2^e, f in [0.5, 1) */
                s = (float)(f == 0.5 ? (double)ratio : ldexp(1.0, e));
            }
        }
        scale[r] = s;
        for (int64_t c = 0; c < cols; ++c) {
            const float q = xr[c] / s;
            codes[r * cols + c] = dsa_oracle_e4m3_encode(q);
        }
    }
}

/* ----------------------------------------------------------- lightning index
 * I[t,s] = sum_j w[t,j] * ReLU( sum_d qdeq[t,j,d] * kdeq[s,d] )
 * with qdeq = e4m3(q8) * q_scale[t] and kdeq = e4m3(k8) * k_scale[s].
 */
static double index_score(const uint8_t *q8t, double qs, const float *wt, int HI, int dI,
                          const uint8_t *k8s, double ks)
{
    double score = 0.0;
    for (int j = 0; j < HI; ++j) {
        double dot = 0.0;
        for (int d = 0; d < dI; ++d)
            dot += (dsa_oracle_e4m3(q8t[(int64_t)j * dI + d]) * qs) *
                   (dsa_oracle_e4m3(k8s[d]) * ks);
        score += (double)wt[j] * (dot > 0.0 ? dot : 0.0);
    }
    return score;
}

/* Contiguous keys.  Query row r (r < n) has FP8 codes q8[r,HI,dI], scale
 * q_scale[r], head weights w[r,HI] and absolute position q_pos[r]; it is scored
 * against keys s = 0 .. min(q_pos[r], S-1).  out[r*ld + s] receives I[r,s];
 * other entries are left untouched. */
void dsa_oracle_indexer(const uint8_t *q8, const float *q_scale, const float *w,
                        const int32_t *q_pos, int n, int HI, int dI,
                        const uint8_t *k8, const float *k_scale, int S,
                        double *out, int64_t ld)
{
    for (int r = 0; r < n; ++r) {
        const uint8_t *q8t = q8 + (int64_t)r * HI * dI;
        const float *wt = w + (int64_t)r * HI;
        int last = q_pos[r];
        if (last > S - 1)
            last = S - 1;
#pragma omp parallel for schedule(dynamic, 64)
        for (int s = 0; s <= last; ++s)
            out[(int64_t)r * ld + s] =
                index_score(q8t, q_scale[r], wt, HI, dI, k8 + (int64_t)s * dI, k_scale[s]);
    }
}

/* Paged keys.  Row r belongs to a sequence of length ctx_len[r]; its query sits
 * at position ctx_len[r]-1 and is scored against the sequence's positions
 * 0 .. ctx_len[r]-1.  Logical position s lives in pool page
 * block_table[r*max_pages + s/page_size], slot s % page_size; the pool holds
 * k8_pool[num_pages, page_size, dI] codes and k_scale_pool[num_pages, page_size]
 * scales.  A position whose page id is outside [0, num_pages) is left
 * untouched in out. */
void dsa_oracle_indexer_paged(const uint8_t *q8, const float *q_scale, const float *w,
                              const int32_t *ctx_len, int n, int HI, int dI,
                              const uint8_t *k8_pool, const float *k_scale_pool,
                              int num_pages, int page_size,
                              const int32_t *block_table, int max_pages,
                              double *out, int64_t ld)
{
    for (int r = 0; r < n; ++r) {
        const uint8_t *q8t = q8 + (int64_t)r * HI * dI;
        const float *wt = w + (int64_t)r * HI;
        int len = ctx_len[r];
        if (len > max_pages * page_size)
            len = max_pages * page_size;
#pragma omp parallel for schedule(dynamic, 64)
        for (int s = 0; s < len; ++s) {
            int page = block_table[(int64_t)r * max_pages + s / page_size];
            if (page < 0 || page >= num_pages)
                continue;
            int64_t slot = (int64_t)page * page_size + s % page_size;
            out[(int64_t)r * ld + s] =
                index_score(q8t, q_scale[r], wt, HI, dI, k8_pool + slot * dI, k_scale_pool[slot]);
        }
    }
}

/* ------------------------------------------------------------------ top-k
 * For each row: the min(k, n) candidates s in [0, n) with the largest value,
 * ranked by (value descending, index ascending) through a full stable sort,
 * then written in ascending index order and padded with -1.
 */
typedef struct {
    double v;
    int32_t s;
} cand_t;

static int cmp_rank(const void *a, const void *b)
{
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->s > y->s) - (x->s < y->s);
}

static int cmp_int32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

void dsa_oracle_topk(const double *vals, int64_t ld, int rows, const int32_t *valid_len,
                     int k, int32_t *idx)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < rows; ++r) {
        int n = valid_len[r];
        if (n < 0) n = 0;
        if (n > ld) n = (int)ld;
        cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(n > 0 ? n : 1));
        for (int s = 0; s < n; ++s) {
            c[s].v = vals[(int64_t)r * ld + s];
            c[s].s = s;
        }
        qsort(c, (size_t)n, sizeof(cand_t), cmp_rank);
        int m = n < k ? n : k;
        int32_t *o = idx + (int64_t)r * k;
        for (int i = 0; i < m; ++i)
            o[i] = c[i].s;
        qsort(o, (size_t)m, sizeof(int32_t), cmp_int32);
        for (int i = m; i < k; ++i)
            o[i] = -1;
        free(c);
    }
}

/* ------------------------------------------------------- sparse MLA (MQA)
 * For query row r and head h over its valid selected rows s_i:
 *   S_i = sm_scale * sum_{d<D} Q[r,h,d] * KV[s_i,d]
 *   O[r,h,v] = sum_i softmax(S)_i * KV[s_i,v]        (v < Dv)
 *   LSE[r,h] = ln sum_i exp(S_i)
 * The softmax is evaluated as exp(S_i - max) / sum exp(S_j - max), which is the
 * same quantity.  `row_of` maps a selected entry to a latent row (or -1 when
 * the entry is invalid).
 */
static void attend(const uint16_t *q_rh, const uint16_t *kv, const int64_t *rows_sel, int nsel,
                   int D, int Dv, double sm_scale, double *score, double *o, double *lse)
{
    double m = -INFINITY;
    int any = 0;
    for (int i = 0; i < nsel; ++i) {
        if (rows_sel[i] < 0)
            continue;
        const uint16_t *c = kv + rows_sel[i] * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += dsa_oracle_bf16(q_rh[d]) * dsa_oracle_bf16(c[d]);
        score[i] = sm_scale * dot;
        if (score[i] > m) m = score[i];
        any = 1;
    }
    for (int v = 0; v < Dv; ++v)
        o[v] = 0.0;
    if (!any) {
        *lse = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int i = 0; i < nsel; ++i) {
        if (rows_sel[i] < 0)
            continue;
        double p = exp(score[i] - m);
        const uint16_t *c = kv + rows_sel[i] * D;
        z += p;
        for (int v = 0; v < Dv; ++v)
            o[v] += p * dsa_oracle_bf16(c[v]);
    }
    for (int v = 0; v < Dv; ++v)
        o[v] /= z;
    *lse = m + log(z);
}

/* Prefill: q[n,H,D], kv[S,D] (BF16 bits), idx[n,k]; an entry outside [0,S) is
 * skipped.  out[n,H,Dv], lse[n,H]. */
void dsa_oracle_sparse_mla(const uint16_t *q, const uint16_t *kv, int S,
                           const int32_t *idx, int n, int H, int D, int Dv, int k,
                           double sm_scale, double *out, double *lse)
{
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int r = 0; r < n; ++r) {
        for (int h = 0; h < H; ++h) {
            int64_t *rows_sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)k);
            double *score = (double *)malloc(sizeof(double) * (size_t)k);
            for (int i = 0; i < k; ++i) {
                int32_t s = idx[(int64_t)r * k + i];
                rows_sel[i] = (s >= 0 && s < S) ? (int64_t)s : -1;
            }
            attend(q + ((int64_t)r * H + h) * D, kv, rows_sel, k, D, Dv, sm_scale, score,
                   out + ((int64_t)r * H + h) * Dv, lse + (int64_t)r * H + h);
            free(score);
            free(rows_sel);
        }
    }
}

/* Paged decode: row r is the newest token of a sequence of length ctx_len[r]
 * (its position is ctx_len[r]-1); idx[r,k] holds logical positions, translated
 * through block_table[r, max_pages] into kv_pool[num_pages, page_size, D].  A
 * position outside [0, ctx_len[r]) or on a page id outside [0, num_pages) is
 * skipped. */
void dsa_oracle_sparse_mla_paged(const uint16_t *q, const uint16_t *kv_pool,
                                 int num_pages, int page_size,
                                 const int32_t *block_table, int max_pages,
                                 const int32_t *ctx_len, const int32_t *idx,
                                 int n, int H, int D, int Dv, int k,
                                 double sm_scale, double *out, double *lse)
{
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int r = 0; r < n; ++r) {
        for (int h = 0; h < H; ++h) {
            int64_t *rows_sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)k);
            double *score = (double *)malloc(sizeof(double) * (size_t)k);
            for (int i = 0; i < k; ++i) {
                int32_t s = idx[(int64_t)r * k + i];
                rows_sel[i] = -1;
                if (s < 0 || s >= ctx_len[r] || s / page_size >= max_pages)
                    continue;
                int page = block_table[(int64_t)r * max_pages + s / page_size];
                if (page < 0 || page >= num_pages)
                    continue;
                rows_sel[i] = (int64_t)page * page_size + s % page_size;
            }
            attend(q + ((int64_t)r * H + h) * D, kv_pool, rows_sel, k, D, Dv, sm_scale, score,
                   out + ((int64_t)r * H + h) * Dv, lse + (int64_t)r * H + h);
            free(score);
            free(rows_sel);
        }
    }
}

/* ------------------------------------------- indexer warm-up (training path)
 * Release summary "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency with
 * DeepSeek Sparse Attention", section "Method": before sparse training, a
 * dense warm-up trains only the lightning indexer, against a
 * KL-divergence-to-main-attention target.  Readings (the pages give no
 * formula): the target of query token t is the main attention's dense causal
 * distribution over its keys s <= t, averaged over the H query heads (the
 * indexer has one distribution per token, shared by all heads in MQA mode);
 * the indexer's distribution is softmax over s <= t of I[t,s]; the loss of
 * row t is KL(target || indexer) = sum_s p (ln p - ln softmax(I)_s), 0 ln 0 = 0;
 * gradients are those of the sum of the rows' losses with respect to w and to
 * the dequantised indexer inputs q = code * q_scale, k = code * k_scale (the
 * quantiser passes gradients straight through); ReLU'(0) = 0.
 */

/* p[r*ld + s] for s <= min(q_pos[r], S-1): the mean over heads h of
 * softmax_s(sm_scale * <Q[r,h,:D], KV[s,:D]>) over s in [0, q_pos[r]]; entries
 * past the row are left untouched. */
void dsa_oracle_attn_target(const uint16_t *q, const uint16_t *kv, int S, const int32_t *q_pos, int n, int H, int D,
                            double sm_scale, double *p, int64_t ld)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
        int last = q_pos[r];
        if (last > S - 1)
            last = S - 1;
        if (last < 0)
            continue;
        const int cnt = last + 1;
        double *sc = (double *)malloc(sizeof(double) * (size_t)cnt);
        double *acc = p + (int64_t)r * ld;
        for (int s = 0; s < cnt; ++s)
            acc[s] = 0.0;
        for (int h = 0; h < H; ++h) {
            const uint16_t *qh = q + ((int64_t)r * H + h) * D;
            double m = -INFINITY;
            for (int s = 0; s < cnt; ++s) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += dsa_oracle_bf16(qh[d]) * dsa_oracle_bf16(kv[(int64_t)s * D + d]);
                sc[s] = sm_scale * dot;
                if (sc[s] > m)
                    m = sc[s];
            }
            double z = 0.0;
            for (int s = 0; s < cnt; ++s)
                z += exp(sc[s] - m);
            for (int s = 0; s < cnt; ++s)
                acc[s] += exp(sc[s] - m) / z / H;
        }
        free(sc);
    }
}

/* The warm-up loss and its gradients for query rows r < n over keys s <= q_pos[r]
 * (clamped to S-1), from dequantised fp64 inputs q[n,HI,dI], k[S,dI] and head
 * weights w[n,HI], given the target p[r*ldp + s]:
 *   a[r,j,s] = <q[r,j,:], k[s,:]>,  I[r,s] = sum_j w[r,j] max(a, 0)
 *   L[r]     = sum_s p (ln p - (I - lse_r)),  lse_r = ln sum_s exp I[r,s]
 *   g[r,s]   = softmax(I)_s - p[r,s]                       (dL/dI, rows of p sum to 1)
 *   dw[r,j]  = sum_s g max(a, 0)
 *   dq[r,j,:] = sum_s g w[r,j] [a > 0] k[s,:]
 *   dk[s,:]  = sum_r sum_j g w[r,j] [a > 0] q[r,j,:]
 * loss[n], dw[n,HI], dq[n,HI,dI] are written; dk[S,dI] is zeroed and then
 * accumulated over the rows.
 * ReLU'(0) = 0, and the decision [a > 0] is taken on the exact a: see relu_on. */

/* [a > 0] for a = <qv, kv> of dI terms, given the fp64 sum a and sabs = sum |q_d k_d|.
 * The fp64 sum is off by at most 2 dI 2^-53 sabs (products and additions each
 * rounded once), so its sign stands beyond dI 2^-50 sabs.  Below that the sum is
 * formed again in binary128, where for FP8-dequantised inputs it is exact: every
 * product of (code x scale) values has at most 2 x 28 significant bits, all of
 * them share the factor of the two scales, and their exponents span the codes'
 * 36 bits, so dI = 128 terms fit in 56 + 36 + 7 < 113 bits.  (A sum that cancels
 * to exactly 0 can come out of fp64 as a tiny nonzero value.) */
static int relu_on(const double *qv, const double *kv, int dI, double a, double sabs)
{
    if (fabs(a) > (double)dI * 0x1p-50 * sabs)
        return a > 0.0;
    _Float128 acc = 0;
    for (int d = 0; d < dI; ++d)
        acc += (_Float128)qv[d] * (_Float128)kv[d];
    return acc > 0;
}

void dsa_oracle_indexer_kl(const double *q, const double *w, const int32_t *q_pos, int n, int HI, int dI,
                           const double *k, int S, const double *p, int64_t ldp, double *loss, double *dw, double *dq,
                           double *dk)
{
    for (int64_t i = 0; i < (int64_t)S * dI; ++i)
        dk[i] = 0.0;
    /* per row: I, softmax, loss, g; then dw, dq (rows in parallel) */
    double *g_all = (double *)malloc(sizeof(double) * (size_t)n * (size_t)(S > 0 ? S : 1));
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
        int last = q_pos[r];
        if (last > S - 1)
            last = S - 1;
        double *g = g_all + (int64_t)r * S;
        const double *qr = q + (int64_t)r * HI * dI;
        const double *wr = w + (int64_t)r * HI;
        for (int j = 0; j < HI; ++j)
            dw[(int64_t)r * HI + j] = 0.0;
        for (int64_t i = 0; i < (int64_t)HI * dI; ++i)
            dq[(int64_t)r * HI * dI + i] = 0.0;
        if (last < 0) {
            loss[r] = 0.0;
            continue;
        }
        const int cnt = last + 1;
        double m = -INFINITY;
        for (int s = 0; s < cnt; ++s) {
            double I = 0.0;
            for (int j = 0; j < HI; ++j) {
                double a = 0.0;
                for (int d = 0; d < dI; ++d)
                    a += qr[(int64_t)j * dI + d] * k[(int64_t)s * dI + d];
                I += wr[j] * (a > 0.0 ? a : 0.0);
            }
            g[s] = I; /* holds I for now */
            if (I > m)
                m = I;
        }
        double z = 0.0;
        for (int s = 0; s < cnt; ++s)
            z += exp(g[s] - m);
        const double lse = m + log(z);
        double L = 0.0;
        for (int s = 0; s < cnt; ++s) {
            const double ps = p[(int64_t)r * ldp + s];
            if (ps > 0.0)
                L += ps * (log(ps) - (g[s] - lse));
            g[s] = exp(g[s] - lse) - ps;
        }
        loss[r] = L;
        for (int s = 0; s < cnt; ++s) {
            for (int j = 0; j < HI; ++j) {
                double a = 0.0, sabs = 0.0;
                for (int d = 0; d < dI; ++d) {
                    const double t = qr[(int64_t)j * dI + d] * k[(int64_t)s * dI + d];
                    a += t;
                    sabs += fabs(t);
                }
                if (relu_on(qr + (int64_t)j * dI, k + (int64_t)s * dI, dI, a, sabs)) {
                    dw[(int64_t)r * HI + j] += g[s] * a;
                    for (int d = 0; d < dI; ++d)
                        dq[((int64_t)r * HI + j) * dI + d] += g[s] * wr[j] * k[(int64_t)s * dI + d];
                }
            }
        }
    }
    /* dk: keys in parallel, each summing over the rows that see it */
#pragma omp parallel for schedule(dynamic, 16)
    for (int s = 0; s < S; ++s) {
        for (int r = 0; r < n; ++r) {
            int last = q_pos[r];
            if (last > S - 1)
                last = S - 1;
            if (s > last)
                continue;
            const double gs = g_all[(int64_t)r * S + s];
            const double *qr = q + (int64_t)r * HI * dI;
            for (int j = 0; j < HI; ++j) {
                double a = 0.0, sabs = 0.0;
                for (int d = 0; d < dI; ++d) {
                    const double t = qr[(int64_t)j * dI + d] * k[(int64_t)s * dI + d];
                    a += t;
                    sabs += fabs(t);
                }
                if (relu_on(qr + (int64_t)j * dI, k + (int64_t)s * dI, dI, a, sabs))
                    for (int d = 0; d < dI; ++d)
                        dk[(int64_t)s * dI + d] += gs * w[(int64_t)r * HI + j] * qr[(int64_t)j * dI + d];
            }
        }
    }
    free(g_all);
}
