// Host-side interfaces between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace dsa {

// Encodes a 2-D tiled tensor map (dims/box in elements, row stride in bytes).
// Returns false and fills `err` on failure.
bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                    uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                    CUtensorMapSwizzle swizzle, char *err, size_t errlen);

int num_sms();

// Records a message for dsa_last_error() on this host thread and returns `code`.
int report_error(int code, const char *fmt, ...);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device (`done` holds one flag per device; a device past the
// table's end sets it on every call).  Two host threads may both find the flag
// clear and both set the attribute: the call is idempotent and the flag atomic.
template <typename... KArgs>
cudaError_t raise_smem_limit_once(void (*kernel)(KArgs...), int bytes, std::atomic<bool> (&done)[64])
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && done[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev < 64)
        done[dev].store(true, std::memory_order_release);
    if (e != cudaSuccess)
        cudaGetLastError(); // the failure is reported to the caller; leave no error behind for the next call
    return e;
}

// Launches `kernel` on `stream` with programmatic dependent launch allowed
// (the kernel must call grid_dep_wait() before touching global memory) and,
// when cluster_x > 1, thread-block clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned cluster_x, Args &&...args)
{
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}
unsigned *device_status_ptr(); // address of this device's status word, or null

struct QuantizeArgs {
    const float *x;  // [rows, cols] fp32
    int64_t rows, cols;
    int mode;        // 0: amax / 448, 1: power-of-two scale
    uint8_t *codes;  // [rows, cols] E4M3
    float *scale;    // [rows]
};
int launch_quantize(const QuantizeArgs &a, cudaStream_t stream, char *err, size_t errlen);

struct IndexerArgs {
    const void *q8;
    const float *q_scale;
    const float *w;
    int T, HI, dI;
    const void *k8;
    const float *k_scale;
    int S;
    const int32_t *block_table;
    int max_pages, num_pages, page_size;
    const int32_t *q_pos;
    float *logits;
    int64_t ld;
    // Candidate mode (cand != nullptr; contiguous keys, H_I in {32, 64}): no
    // logits are written; a key whose score is >= thr[r] is appended to row
    // r's list as {raw fp32 score bits, position}, in no particular order.  The
    // list is 128 regions of cap entries, one per epilogue lane scoring the row.
    const float *thr = nullptr;        // [T]
    uint2 *cand = nullptr;             // [T, 128, cap]
    int32_t *cand_cnt = nullptr;       // [T, 128] candidates each region found (only cap are stored)
    int cap = 0;
    const int32_t *row_flag = nullptr; // score only rows with row_flag[r] != 0 (nullptr: all rows)
};
// Returns 0 on success, else a dsa_status with `err` filled.
int launch_indexer(const IndexerArgs &a, cudaStream_t stream, char *err, size_t errlen);

struct TopkArgs {
    const float *logits;
    int64_t ld;
    int T;
    const int32_t *valid_len;
    int k;
    int32_t *idx;
    const int32_t *row_flag = nullptr; // only rows with row_flag[r] != 0 (nullptr: all rows)
};
int launch_topk(const TopkArgs &a, cudaStream_t stream, char *err, size_t errlen);

// Fused indexer -> top-k pieces (topk.cu): the per-row threshold from sampled
// scores, and the exact top-k over each row's candidate list.
int launch_topk_threshold(const float *samp, int ld_s, int T, const int32_t *q_pos, const int32_t *qpos_s, int S,
                          int k, int cap, float *thr, cudaStream_t stream, char *err, size_t errlen);
int launch_topk_candidates(const uint2 *cand, const int32_t *cand_cnt, int cap, int T, const int32_t *q_pos, int S,
                           int k, int32_t *idx, int32_t *flag, cudaStream_t stream, char *err, size_t errlen);
size_t topk_candidates_smem(int S, int cap);

struct IndexerTopkArgs {
    const void *q8;
    const float *q_scale;
    const float *w;
    int T, HI, dI;
    const void *k8;
    const float *k_scale;
    int S;
    const int32_t *q_pos;
    int k;
    int32_t *idx;
    void *workspace;
    size_t workspace_bytes;
};
int launch_indexer_topk(const IndexerTopkArgs &a, cudaStream_t stream, char *err, size_t errlen);
size_t indexer_topk_workspace_bytes(int T, int S, int dI, int k);

struct WarmupArgs {
    const void *q;       // [T, H, 576] bf16: main-attention queries
    const void *kv;      // [S, 576] bf16
    int H;
    float sm_scale;
    const void *q8;      // indexer inputs as for dsa_indexer_logits (contiguous keys)
    const float *q_scale;
    const float *w;
    int HI, dI;
    const void *k8;
    const float *k_scale;
    const int32_t *q_pos;
    int T, S;
    float *loss;         // [T]
    float *dw;           // [T, HI]
    float *dq;           // [T, HI, dI]
    float *dk;           // [S, dI]
    void *workspace;
    size_t workspace_bytes;
};
int launch_warmup(const WarmupArgs &a, cudaStream_t stream, char *err, size_t errlen);
size_t warmup_workspace_bytes(int T, int S, int HI);

struct MlaArgs {
    const void *q;      // [T, H, 576] bf16
    const void *kv;     // [S, 576] bf16, or pool [num_pages, page_size, 576]
    int S;              // rows of kv (prefill) / num_pages * page_size (paged)
    const int32_t *idx; // [T, k]
    int T, H, k;
    float sm_scale;
    void *out;          // [T, H, 512] bf16
    float *lse;         // [T, H]
    // paged decode
    const int32_t *block_table;
    int max_pages, num_pages, page_size;
    const int32_t *ctx_len;
    void *workspace;
    size_t workspace_bytes;
};
int launch_mla_prefill(const MlaArgs &a, cudaStream_t stream, char *err, size_t errlen);
int launch_mla_decode(const MlaArgs &a, cudaStream_t stream, char *err, size_t errlen);
size_t mla_decode_workspace_bytes(int B, int H, int k);

} // namespace dsa
