/*
 * dsa.h: C ABI of libdsa.so, the GB300 (sm_103a) hot path of DeepSeek Sparse
 * Attention (DSA).
 *
 * The method (release summary "DeepSeek-V3.2-Exp: Boosting Long-Context
 * Efficiency with DeepSeek Sparse Attention", section "Method"; AMD article
 * "AMD Instinct MI355X GPUs Power DeepSeek-V3.2-Exp", section "DeepSeek Sparse
 * Attention (DSA)") has three stages, one entry point each, plus the paged
 * decode form of the attention stage:
 *   1. lightning indexer   I[t,s] = sum_j w[t,j] * ReLU(q[t,j] . k[s]), in FP8
 *   2. top-k selection     the k (= 2048) highest-scoring prior tokens per query
 *   3. sparse MLA          MQA-mode attention over only the selected latent rows
 *
 * Conventions shared by every entry point
 *   - Every pointer named as a tensor is a DEVICE pointer; shapes are row-major
 *     and contiguous unless a leading dimension is given.  The caller owns every
 *     buffer; the library allocates nothing, frees nothing and keeps no pointer
 *     after a call returns.
 *   - Work is enqueued asynchronously on `stream` (0 = legacy default stream).
 *     Nothing synchronises inside the library and nothing falls back to the
 *     host.
 *   - Arguments are checked on the host before any launch.  On error the call
 *     returns a non-zero dsa_status, launches nothing, leaves outputs untouched
 *     and records a message for dsa_last_error().
 *   - Data-dependent problems that only the device can see (a bad page id, a
 *     position past the buffer, a pipeline wait that ran out of time) never
 *     cause an out-of-bounds access: the kernel skips the offending element and
 *     sets a bit in a per-device status word, read with dsa_get_device_status().
 *   - "FP8" is E4M3 (OCP "fn" variant, max 448), passed as raw bytes.  "bf16" is
 *     IEEE binary32 truncated to its upper 16 bits, passed as raw uint16.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dsa_stream_t; /* same type as cudaStream_t */

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent shapes   */
    DSA_ERR_UNSUPPORTED = 2, /* a size the library has no kernel for (see below)   */
    DSA_ERR_ALIGNMENT = 3,   /* a pointer or stride breaks a 16-byte TMA rule       */
    DSA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than the query says    */
    DSA_ERR_CUDA = 5,        /* a CUDA runtime/driver call or a launch failed       */
    DSA_ERR_DEVICE = 6       /* dsa_get_device_status() found a device-side error   */
} dsa_status;

/* Bits of the device status word (dsa_get_device_status). */
#define DSA_DEV_TIMEOUT      0x1u /* a bounded pipeline wait gave up; outputs of that CTA are invalid */
#define DSA_DEV_BAD_POSITION 0x2u /* a query position / valid length exceeded the key range or ld     */
#define DSA_DEV_BAD_PAGE     0x4u /* a block-table entry outside [0, num_pages); those keys skipped    */

/* Message for the last failing call on this host thread ("" if none). */
const char *dsa_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int dsa_version(void);

/*
 * dsa_get_device_status: copy the device status word of the current device to
 * *status_out (DSA_DEV_* bits, 0 = clean) and clear it.  Enqueued on `stream`
 * and then waits for that stream, so it sees every earlier kernel on it.
 * Returns DSA_ERR_CUDA if the copy fails.
 */
int dsa_get_device_status(dsa_stream_t stream, uint32_t *status_out);

/*
 * dsa_selftest_wait_timeout: exercises the failure detection that every
 * kernel's pipeline waits share (the pages have no counterpart).  Launches
 * one CTA that waits, through the same bounded mbarrier wait, on a barrier
 * nothing arrives on; after limit_us microseconds (1 .. 1000000) the wait
 * gives up, sets DSA_DEV_TIMEOUT in the device status word and the kernel
 * returns, leaving the context usable.  Read the bit with
 * dsa_get_device_status().  Nothing faults, traps or hangs.
 */
int dsa_selftest_wait_timeout(uint32_t limit_us, dsa_stream_t stream);

/*
 * dsa_indexer_logits: lightning-indexer scores (stage 1).
 *
 * Defines, for each query row r at absolute position p = q_pos[r] and each key
 * position s in [0, p]:
 *     logits[r*ld_logits + s] = sum_{j<H_I} w[r,j] * ReLU( sum_{d<d_I}
 *                               (q8[r,j,d]*q_scale[r]) * (k8[s,d]*k_scale[s]) )
 * ("DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency with DeepSeek Sparse
 * Attention", section "Method": index score against all prior tokens, ReLU,
 * FP8, few heads).  The query's own position is included (causal s <= p).
 * Entries with s > p are unspecified (the kernel may write -inf there, but
 * never at or past ld_logits).
 *
 *   q8        [T, H_I, d_I]  FP8 codes of the indexer queries
 *   q_scale   [T]            fp32, > 0: one dequantisation scale per query token
 *   w         [T, H_I]       fp32 head weights (any sign)
 *   q_pos     [T]            int32 absolute position of each query row
 *   logits    [T, ld_logits] fp32 output, ld_logits >= 1 + max position used
 *
 * Keys, contiguous form (block_table == NULL):
 *   k8        [S, d_I]       FP8 codes;   k_scale [S] fp32 > 0
 *   A position q_pos[r] >= S is clamped to S-1 and flagged DSA_DEV_BAD_POSITION.
 * Keys, paged form (block_table != NULL; used by decode, "indexer-logit kernels
 * (incl. paged versions)", same page, "Key claims"):
 *   k8        [num_pages, page_size, d_I] pool of FP8 codes
 *   k_scale   [num_pages, page_size]      fp32 scales
 *   block_table [T, max_pages] int32: row r's logical page i lives in pool page
 *             block_table[r*max_pages + i]; a key at logical position s lives at
 *             slot s % page_size of page block_table[r*max_pages + s/page_size].
 *   S is ignored.  Each row is its own sequence.  An out-of-range page id is
 *   skipped (its logits are left unwritten) and flagged DSA_DEV_BAD_PAGE.
 *
 * Supported sizes: (H_I, d_I) = (64,128) or (32,128), contiguous or paged;
 * (4,32) contiguous only; any other pair returns DSA_ERR_UNSUPPORTED.
 * page_size in {32, 64, 128}; T >= 0 (T = 0 is a no-op).
 * Alignment: q8 and k8 16-byte aligned; ld_logits >= 1.
 */
int dsa_indexer_logits(const void *q8, const float *q_scale, const float *w,
                       int T, int H_I, int d_I,
                       const void *k8, const float *k_scale, int S,
                       const int32_t *block_table, int max_pages, int num_pages, int page_size,
                       const int32_t *q_pos,
                       float *logits, int64_t ld_logits, dsa_stream_t stream);

/*
 * dsa_quantize_fp8: per-token FP8 (E4M3) quantisation of the indexer inputs.
 *
 * The indexer runs in FP8 with one positive scale per token ("AMD Instinct
 * MI355X GPUs Power DeepSeek-V3.2-Exp", section "DeepSeek Sparse Attention
 * (DSA)", item 1; release summary "DeepSeek-V3.2-Exp: Boosting Long-Context
 * Efficiency with DeepSeek Sparse Attention", section "Method"); the gist
 * page's indexer test script casts to E4M3 with an option for power-of-two
 * (UE8M0) scales.  For each row r of cols values x[r*cols + c]:
 *   DSA_SCALE_AMAX  scale[r] = amax / 448 in fp32 (1 for an all-zero row)
 *   DSA_SCALE_POW2  scale[r] = the smallest power of two >= that ratio
 *                   (1 for an all-zero row)
 *   codes[r*cols + c] = E4M3 nearest to x / scale[r] (fp32 division), ties to
 *                   the even code, magnitudes above 448 saturated to 448.
 * The indexer's q rows are tokens over all H_I * d_I entries, its k rows
 * tokens over d_I; dequantised value = code * scale.
 *
 *   x      [rows, cols] fp32, contiguous;  codes [rows, cols] uint8 (E4M3);
 *   scale  [rows] fp32.  rows = 0 is a no-op.  Inputs must be finite.
 * Any alignment works; 16-byte aligned rows of x (and 4-byte aligned rows of
 * codes) take the vector path.
 */
#define DSA_SCALE_AMAX 0
#define DSA_SCALE_POW2 1
int dsa_quantize_fp8(const float *x, int64_t rows, int64_t cols, int scale_mode,
                     void *codes, float *scale, dsa_stream_t stream);

/*
 * dsa_topk: fine-grained token selection (stage 2).
 *
 * For each row t with n = valid_len[t] candidates logits[t*ld + s], s in [0, n):
 * keeps the min(k, n) candidates ranked first by (score descending, index
 * ascending) and writes their indices to idx[t*k ...] in ASCENDING index
 * order, padded with -1 ("AMD Instinct MI355X GPUs Power DeepSeek-V3.2-Exp",
 * section "DeepSeek Sparse Attention (DSA)", item 2: top-2048 per query).
 * -0.0 and +0.0 compare equal.  Scores must be finite (a NaN makes that row's
 * result unspecified, never out of bounds).  n > ld is clamped to ld and
 * flagged DSA_DEV_BAD_POSITION; n < 0 counts as 0.
 *
 *   logits    [T, ld] fp32;  valid_len [T] int32;  idx [T, k] int32 output.
 * Supported: 1 <= k <= 4096, ld >= 1, ld <= 2^28.  Deterministic: the same
 * inputs give the same bytes.
 */
int dsa_topk(const float *logits, int64_t ld, int T, const int32_t *valid_len,
             int k, int32_t *idx, dsa_stream_t stream);

/*
 * dsa_indexer_topk: stages 1 and 2 in one call, without the index scores ever
 * reaching memory.
 *
 * Result: exactly what dsa_indexer_logits (contiguous keys) followed by
 * dsa_topk with valid_len[r] = min(q_pos[r] + 1, S) writes to idx, byte for
 * byte: for each query row r, the k keys s in [0, q_pos[r]] with the highest
 * index score (score descending, position ascending), in ascending order,
 * padded with -1 (release summary "DeepSeek-V3.2-Exp: Boosting Long-Context
 * Efficiency with DeepSeek Sparse Attention", section "Method"; "AMD Instinct
 * MI355X GPUs Power DeepSeek-V3.2-Exp", section "Computational Efficiency":
 * attention drops from O(L^2) to O(Lk), which leaves the indexer's L x L
 * scores as the long-context cost; here they are neither written nor read).
 *
 * How: a per-row threshold from the scores of keys sampled at a fixed stride
 * (2048 of them, or S/32 past 65536 keys), which about 1.25k + 256 of the
 * row's keys reach (rows of at most max(4096, 2k) keys take every key); the
 * indexer then appends only the keys at or above it to per-row lists, and an
 * exact top-k runs over each list.  A row whose list misses
 * [k, max(4096, 2k)] (a row unlike its samples) is redone from its full
 * scores, so the result never depends on the sample.
 *
 *   q8, q_scale, w, q_pos, k8, k_scale, S: as for dsa_indexer_logits with
 *             contiguous keys ([S, d_I] codes, [S] scales); (H_I, d_I) =
 *             (64, 128) or (32, 128); 1 <= S <= DSA_INDEXER_TOPK_MAX_KEYS.
 *   k         1 <= k <= 4096;   idx [T, k] int32 output.
 *   workspace a device buffer of dsa_indexer_topk_workspace_size(T, S, H_I,
 *             d_I, k) bytes, 256-byte aligned, owned by the caller, used only
 *             while the call's kernels run on `stream` (calls sharing one must
 *             be ordered).  It holds the sampled keys and scores, the per-row
 *             candidate lists (T x max(4096, 2k) entries of 8 bytes) and, for
 *             the rows redone from full scores, T x S fp32 scores: most of it
 *             stays untouched; callers with long rows pass rows in chunks.
 * A position q_pos[r] >= S is clamped to S-1 and flagged DSA_DEV_BAD_POSITION.
 */
#define DSA_INDEXER_TOPK_MAX_KEYS 262144
int dsa_indexer_topk(const void *q8, const float *q_scale, const float *w, int T, int H_I, int d_I,
                     const void *k8, const float *k_scale, int S, const int32_t *q_pos,
                     int k, int32_t *idx, void *workspace, size_t workspace_bytes, dsa_stream_t stream);

/* Bytes of workspace dsa_indexer_topk needs (0 on unsupported sizes). */
size_t dsa_indexer_topk_workspace_size(int T, int S, int H_I, int d_I, int k);

/*
 * dsa_indexer_warmup: the indexer's dense warm-up step, loss and gradients.
 *
 * Release summary "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency with
 * DeepSeek Sparse Attention", section "Method": before sparse training a dense
 * warm-up trains only the lightning indexer, against a KL-divergence-to-main-
 * attention target.  Readings (the pages give no formula): for query row t at
 * position q_pos[t] (clamped to S-1) over keys s <= q_pos[t]
 *   p[t,s]   = mean over the H heads of softmax_s(sm_scale * <q[t,h,:576], kv[s,:576]>)
 *              (the main attention's dense causal distribution, MQA mode)
 *   I[t,s]   = the index score of dsa_indexer_logits, a[t,j,s] = <q8[t,j]*q_scale[t], k8[s]*k_scale[s]>
 *   loss[t]  = sum_s p (ln p - ln softmax_s I[t,:])
 *   dw[t,j]  = d(sum loss)/dw = sum_s g ReLU(a),      g = softmax(I) - p
 *   dq[t,j,:] = sum_s g w[t,j] [a > 0] k[s,:] * k_scale[s]      (w.r.t. the dequantised q)
 *   dk[s,:]  = sum_t sum_j g w[t,j] [a > 0] q[t,j,:] * q_scale[t] (w.r.t. the dequantised k)
 * (the FP8 quantiser passes gradients straight through; ReLU'(0) = 0).
 *
 *   q [T, H, 576] bf16, kv [S, 576] bf16, 1 <= H <= 128, sm_scale > 0;
 *   q8, q_scale, w, q_pos, k8, k_scale: as for dsa_indexer_logits with
 *   contiguous keys, (H_I, d_I) = (64, 128) or (32, 128);
 *   outputs fp32: loss [T], dw [T, H_I], dq [T, H_I, d_I], dk [S, d_I].
 *   workspace: dsa_indexer_warmup_workspace_size(T, S, H_I, d_I) bytes, 256-byte
 *   aligned, owned by the caller (it holds p, I and then g, 8 T S bytes, and the
 *   FP8 codes as bf16 with per-row bounds, about 264 (T H_I + S) bytes).
 * Precision: the target's scores on BF16 tensor cores with fp32 accumulation,
 * the index scores as dsa_indexer_logits; the gradient contractions on BF16
 * tensor cores (the codes exact, the coefficients g w [a > 0] as bf16 hi + lo
 * pairs, fp32 accumulation); the ReLU decision [a > 0] exact (the sign of the
 * exact dot product of the codes).  dk is summed with atomics across chunks of
 * rows, so its last bits may differ from call to call.
 */
int dsa_indexer_warmup(const void *q, const void *kv, int H, float sm_scale,
                       const void *q8, const float *q_scale, const float *w, int H_I, int d_I,
                       const void *k8, const float *k_scale, const int32_t *q_pos, int T, int S,
                       float *loss, float *dw, float *dq, float *dk,
                       void *workspace, size_t workspace_bytes, dsa_stream_t stream);

/* Bytes of workspace dsa_indexer_warmup needs (0 on unsupported sizes). */
size_t dsa_indexer_warmup_workspace_size(int T, int S, int H_I, int d_I);

/*
 * dsa_sparse_mla_prefill: MQA-mode sparse MLA over the selected rows (stage 3).
 *
 * For query row t, head h and its valid selected rows s_i = idx[t*k + i]
 * (0 <= s_i < S; other entries are skipped wherever they stand):
 *     S_i      = sm_scale * sum_{d<576} q[t,h,d] * kv[s_i,d]
 *     out[t,h,v] = sum_i softmax(S)_i * kv[s_i,v]          (v < 512)
 *     lse[t,h] = ln sum_i exp(S_i)
 * ("DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency with DeepSeek Sparse
 * Attention", section "Method": main attention reads only the top-k entries,
 * in MLA's MQA mode so one latent row is shared by all heads of a token; the
 * first 512 columns are V, the last 64 are the RoPE part used only in scores.)
 * A row with no valid entry gets out = 0 and lse = -inf.
 *
 * Precision: scores accumulate in fp32 (each token runs on two SMs that each
 * hold half of the 576 score columns and exchange their fp32 partial scores,
 * so a score is off by a few fp32 ulps of its magnitude, however large); P is
 * rounded to bf16 before the PV product and out to bf16 (nearest even) at the
 * end.
 *
 *   q    [T, H, 576] bf16;  kv [S, 576] bf16;  idx [T, k] int32
 *   out  [T, H, 512] bf16 (rounded to nearest even);  lse [T, H] fp32
 * Supported: 1 <= H <= 128 (fewer than 128 heads run as zero-padded rows
 * that are never stored); D = 576, Dv = 512 fixed; 1 <= k <= 4096.  q, kv, out
 * 16-byte aligned.
 */
int dsa_sparse_mla_prefill(const void *q, const void *kv, int S,
                           const int32_t *idx, int T, int H, int k, float sm_scale,
                           void *out, float *lse, dsa_stream_t stream);

/*
 * dsa_sparse_mla_decode_paged: the same attention over a paged latent cache
 * (decode form of stage 3; "DeepSeek-V3.2-Exp: Boosting Long-Context
 * Efficiency with DeepSeek Sparse Attention", section "Key claims": the
 * released kernels are indexer-logit kernels, paged versions included, and
 * sparse-attention kernels; the attention itself is that of section "Method").
 *
 * Row b is one query: its token sits at position ctx_len[b]-1 of the sequence
 * whose pages block_table row b lists.  Rows are independent, so a batch may
 * hold one new token per sequence (decode), several positions of the same
 * sequence (multi-token decode), or every token of sequences of different
 * lengths (ragged batched prefill), all in one pool.  idx[b*k + i] holds
 * LOGICAL positions, read from slot s % page_size of pool page
 * block_table[b*max_pages + s/page_size].  Entries outside [0, ctx_len[b]) are
 * skipped; a page id outside [0, num_pages) is skipped and flagged
 * DSA_DEV_BAD_PAGE.
 *
 * Work split.  Attention runs on two-CTA clusters, one per pair of SMs.  With
 * more rows than two thirds of the clusters, each cluster takes whole rows, as
 * in prefill.  With fewer, the flattened (row, 64-entry block of idx) space is
 * cut into one contiguous share per cluster, so every SM works; a share that
 * holds only part of a row writes that part's softmax-normalised output and
 * LSE (fp32) to the workspace, and a second kernel merges the parts of each
 * row by their LSEs (LSE = ln sum exp LSE_p, O = sum exp(LSE_p - LSE) O_p)
 * into out and lse.  The split changes only the fp32 summation order.
 *
 *   q       [B, H, 576] bf16;  kv_pool [num_pages, page_size, 576] bf16
 *   block_table [B, max_pages] int32;  ctx_len [B] int32;  idx [B, k] int32
 *   out     [B, H, 512] bf16;  lse [B, H] fp32
 *   workspace: a device buffer of at least
 *           dsa_sparse_mla_decode_workspace_size(B, H, k) bytes, 256-byte
 *           aligned, owned by the caller, used only while the call's kernels
 *           run on `stream`; NULL is accepted when that size is 0.  Calls that
 *           share one workspace must be ordered on the GPU (same stream).
 *           A missing or short workspace returns DSA_ERR_WORKSPACE.
 */
int dsa_sparse_mla_decode_paged(const void *q, const void *kv_pool, int num_pages, int page_size,
                                const int32_t *block_table, int max_pages, const int32_t *ctx_len,
                                const int32_t *idx, int B, int H, int k, float sm_scale,
                                void *out, float *lse, void *workspace, size_t workspace_bytes,
                                dsa_stream_t stream);

/*
 * dsa_prefill_host: the whole prefill path (dsa_indexer_logits -> dsa_topk ->
 * dsa_sparse_mla_prefill, contiguous keys) on inputs in HOST memory, with the
 * outputs written back to HOST memory.  Row r is the query at position
 * q_pos[r] over keys [0, q_pos[r]] (release summary "DeepSeek-V3.2-Exp:
 * Boosting Long-Context Efficiency with DeepSeek Sparse Attention", section
 * "Method"); rows and their arguments mean what they mean for the three
 * device entry points, whose results this call reproduces byte for byte.
 *
 *   host: q8 [T, H_I, d_I] FP8, q_scale [T], w [T, H_I], q_pos [T] int32,
 *         k8 [S, d_I] FP8, k_scale [S], q [T, H, 576] bf16, kv [S, 576] bf16
 *         -> out [T, H, 512] bf16, lse [T, H] fp32.  0 <= q_pos[r] < S.
 *   workspace: device buffer of dsa_prefill_host_workspace_size(...) bytes,
 *         256-byte aligned, owned by the caller.
 *
 * Query rows go in chunks of at most chunk_rows (C): C/4 and C/2 rows first,
 * then C, and a last chunk of C/4, processed from the last chunk to the first
 * (short chunks at both ends: the kernels start after a short copy and little
 * is left to copy out after the last kernels; the first chunk processed brings
 * in the keys of every row, and the long rows' chunks, whose kernels outlast
 * their copies, come first).  The inputs of a chunk
 * are copied in on a copy stream, its kernels run on `stream`, its outputs are copied out on
 * a second copy stream, and four buffer slots let the copies run up to three
 * chunks ahead of the kernels.  The keys stay on the device for the call and are
 * copied in as far as each chunk's positions need them.  Host buffers should be
 * page-locked (cudaHostAlloc or cudaHostRegister) for the copies to overlap;
 * pageable memory gives the same results more slowly.  The call returns once
 * everything is enqueued; all of it is complete when `stream` reaches this
 * point, and the host buffers must stay untouched until then.  The first call
 * on a device creates the two copy streams and a few events, kept until exit;
 * calls from several host threads enqueue one at a time.  Errors of the three
 * stages are reported as they would be by their entry points.
 */
int dsa_prefill_host(const void *q8, const float *q_scale, const float *w, const int32_t *q_pos,
                     const void *k8, const float *k_scale, const void *q, const void *kv,
                     int T, int S, int H_I, int d_I, int H, int k, float sm_scale,
                     void *out, float *lse, int chunk_rows,
                     void *workspace, size_t workspace_bytes, dsa_stream_t stream);

/* Device workspace bytes dsa_prefill_host needs (0 on bad input). */
size_t dsa_prefill_host_workspace_size(int T, int S, int H_I, int d_I, int H, int k, int chunk_rows);

/*
 * dsa_prefill_host_trace: a per-chunk timeline of dsa_prefill_host calls on
 * the current device, to see which stream a slow call spent its time on (a
 * debugging record with no counterpart on the pages; off unless turned on).
 * max_chunks > 0 creates 6 * max_chunks + 1 timing events and starts an empty
 * record; every later call then records, for each of its chunks while the
 * record has room, an event on the input-copy stream before and after the
 * chunk's input copies, on `stream` before and after its three stages, and on
 * the output-copy stream before and after its output copies.  Each "before"
 * event follows the chunk's waits, so it marks when that stream began the
 * chunk.  max_chunks = 0 ends the record and destroys its events.  Returns
 * DSA_ERR_INVALID_ARG for max_chunks outside [0, 2^20], DSA_ERR_CUDA if the
 * events cannot be created (recording is then off).
 */
int dsa_prefill_host_trace(int max_chunks);

/*
 * dsa_prefill_host_trace_read: the record of dsa_prefill_host_trace.  Waits
 * for the recorded events and writes, for the first min(recorded, max_chunks)
 * chunks in enqueue order (HOST arrays): ms[6 j + e] = milliseconds from the
 * start of the first recorded call to event e of chunk j (0/1 input copies
 * begin/end, 2/3 stages begin/end, 4/5 output copies begin/end; NaN for an
 * event a failed call never reached), call[j] = the call the chunk belongs to
 * (0 = first recorded call), rows[j] = its query rows; *n_out = the chunks
 * written.  The record stays as it is. Returns DSA_ERR_INVALID_ARG for a null
 * pointer or max_chunks < 0.
 */
int dsa_prefill_host_trace_read(float *ms, int32_t *call, int32_t *rows, int max_chunks, int *n_out);

/*
 * dsa_sparse_mla_decode_paged_noalloc: dsa_sparse_mla_decode_paged without a
 * caller-provided workspace.  The pages have no counterpart to this entry
 * point: it is for callers that cannot allocate device memory while they
 * run, such as a plugin inside a host program that owns every device
 * allocation, or a service held to a fixed device-memory budget that must not
 * grow or wait on an allocator mid-request.  It allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library call): its workspace is a
 * static device buffer of DSA_DECODE_STATIC_WS_BYTES (40 MiB) built into the
 * library, which every GPU that loads libdsa.so holds until the process exits.
 *
 * Arguments, results and errors are those of dsa_sparse_mla_decode_paged.  A
 * call whose workspace need (dsa_sparse_mla_decode_workspace_size) exceeds the
 * buffer returns DSA_ERR_WORKSPACE with a message naming both sizes; with
 * H <= 128 that takes a device of 160 SMs or more.  The first call on each
 * device looks up the buffer's device address (cudaGetSymbolAddress, with
 * that device current) and keeps it; make that first call before any stream
 * capture.  All calls share the one buffer, which keeps the contents of the
 * last call (nothing in it needs to start at zero: each call writes every
 * part it reads), so calls whose kernels may overlap on the GPU (different
 * streams, or different host threads, on one device) race on it and must be
 * ordered by the caller.
 */
#define DSA_DECODE_STATIC_WS_BYTES (40u << 20)
int dsa_sparse_mla_decode_paged_noalloc(const void *q, const void *kv_pool, int num_pages, int page_size,
                                        const int32_t *block_table, int max_pages, const int32_t *ctx_len,
                                        const int32_t *idx, int B, int H, int k, float sm_scale,
                                        void *out, float *lse, dsa_stream_t stream);

/* Bytes of workspace dsa_sparse_mla_decode_paged needs for (B, H, k) on the
 * current device: 0 when the rows stay whole (3 B > 2 clusters), else
 * 2 * clusters * H * 513 * 4, with clusters = min(SM pairs, B * ceil(k / 64)).
 * 0 on bad input. */
size_t dsa_sparse_mla_decode_workspace_size(int B, int H, int k);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H */
