// C ABI of libdsa.so: host-side argument checks, then launches on the caller's
// stream.  See include/dsa.h for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "../../include/dsa.h"
#include "common.cuh"
#include "launch.h"

namespace dsa {

// Per-device status word (DSA_DEV_* bits); kernels receive its address.
__device__ unsigned g_device_status = 0u;

namespace {

thread_local char t_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok()
{
    t_err[0] = '\0';
    return DSA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device()
{
    int d = 0;
    cudaGetDevice(&d);
    return d;
}

} // namespace

int report_error(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return code;
}

unsigned *device_status_ptr()
{
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[d]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess)
            return nullptr;
        g_status_ptr[d] = static_cast<unsigned *>(p);
    }
    return g_status_ptr[d];
}

int num_sms()
{
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices)
        return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[d]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
        g_sms[d] = n > 0 ? n : 148;
    }
    return g_sms[d];
}

bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner, uint64_t rows,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                    char *err, size_t errlen)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn) {
                snprintf(err, errlen, "cuTensorMapEncodeTiled entry point unavailable");
                return false;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    cuuint64_t dims[2] = {inner, rows > 0 ? rows : 1};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(err, errlen, "cuTensorMapEncodeTiled failed (%d): inner=%llu rows=%llu stride=%llu box=%ux%u", (int)r,
                 (unsigned long long)inner, (unsigned long long)rows, (unsigned long long)row_stride_bytes, box_inner,
                 box_rows);
        return false;
    }
    return true;
}

} // namespace dsa

using namespace dsa;

extern "C" {

const char *dsa_last_error(void) { return t_err; }

int dsa_version(void) { return 100; }

int dsa_get_device_status(dsa_stream_t stream, uint32_t *status_out)
{
    if (!status_out)
        return fail(DSA_ERR_INVALID_ARG, "status_out is null");
    unsigned *dev = device_status_ptr();
    if (!dev)
        return fail(DSA_ERR_CUDA, "device status word unavailable");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, dev, sizeof host, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(dev, 0, sizeof(unsigned), s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return fail(DSA_ERR_CUDA, "reading device status: %s", cudaGetErrorString(e));
    *status_out = host;
    return ok();
}

int dsa_indexer_logits(const void *q8, const float *q_scale, const float *w, int T, int H_I, int d_I, const void *k8,
                       const float *k_scale, int S, const int32_t *block_table, int max_pages, int num_pages,
                       int page_size, const int32_t *q_pos, float *logits, int64_t ld_logits, dsa_stream_t stream)
{
    if (T < 0)
        return fail(DSA_ERR_INVALID_ARG, "T < 0");
    if (T == 0)
        return ok();
    if (!q8 || !q_scale || !w || !k8 || !k_scale || !q_pos || !logits)
        return fail(DSA_ERR_INVALID_ARG, "null pointer argument");
    if (H_I <= 0 || d_I <= 0 || ld_logits < 1)
        return fail(DSA_ERR_INVALID_ARG, "H_I, d_I and ld_logits must be positive");
    if (!aligned16(q8) || !aligned16(k8))
        return fail(DSA_ERR_ALIGNMENT, "q8 and k8 must be 16-byte aligned");
    if ((int64_t)T * H_I > (int64_t)INT32_MAX)
        return fail(DSA_ERR_UNSUPPORTED, "T * H_I too large");
    if (block_table) {
        if (max_pages <= 0 || num_pages <= 0)
            return fail(DSA_ERR_INVALID_ARG, "paged: max_pages and num_pages must be positive");
        if (page_size != 32 && page_size != 64 && page_size != 128)
            return fail(DSA_ERR_UNSUPPORTED, "paged: page_size must be 32, 64 or 128");
    } else {
        if (S <= 0)
            return fail(DSA_ERR_INVALID_ARG, "S must be positive");
    }
    IndexerArgs a{q8, q_scale, w, T, H_I, d_I, k8, k_scale, S, block_table, max_pages, num_pages, page_size,
                  q_pos, logits, ld_logits};
    int rc = launch_indexer(a, reinterpret_cast<cudaStream_t>(stream), t_err, sizeof t_err);
    return rc == DSA_OK ? ok() : rc;
}

size_t dsa_indexer_topk_workspace_size(int T, int S, int H_I, int d_I, int k)
{
    if (T < 0 || S < 1 || S > DSA_INDEXER_TOPK_MAX_KEYS || k < 1 || k > 4096 || d_I != 128 ||
        (H_I != 64 && H_I != 32))
        return 0;
    return indexer_topk_workspace_bytes(T, S, d_I, k);
}

int dsa_indexer_topk(const void *q8, const float *q_scale, const float *w, int T, int H_I, int d_I, const void *k8,
                     const float *k_scale, int S, const int32_t *q_pos, int k, int32_t *idx, void *workspace,
                     size_t workspace_bytes, dsa_stream_t stream)
{
    if (T < 0)
        return fail(DSA_ERR_INVALID_ARG, "T < 0");
    if (T == 0)
        return ok();
    if (!q8 || !q_scale || !w || !k8 || !k_scale || !q_pos || !idx)
        return fail(DSA_ERR_INVALID_ARG, "null pointer argument");
    if (d_I != 128 || (H_I != 64 && H_I != 32))
        return fail(DSA_ERR_UNSUPPORTED, "fused indexer -> top-k: (H_I, d_I) must be (64, 128) or (32, 128)");
    if (S < 1 || S > DSA_INDEXER_TOPK_MAX_KEYS)
        return fail(DSA_ERR_UNSUPPORTED, "fused indexer -> top-k: S must be in [1, %d]", DSA_INDEXER_TOPK_MAX_KEYS);
    if (k < 1 || k > 4096)
        return fail(DSA_ERR_UNSUPPORTED, "k must be in [1, 4096]");
    if (!aligned16(q8) || !aligned16(k8))
        return fail(DSA_ERR_ALIGNMENT, "q8 and k8 must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(DSA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    if (!workspace || workspace_bytes < indexer_topk_workspace_bytes(T, S, d_I, k))
        return fail(DSA_ERR_WORKSPACE, "workspace missing or smaller than dsa_indexer_topk_workspace_size");
    IndexerTopkArgs a{q8, q_scale, w, T, H_I, d_I, k8, k_scale, S, q_pos, k, idx, workspace, workspace_bytes};
    int rc = launch_indexer_topk(a, reinterpret_cast<cudaStream_t>(stream), t_err, sizeof t_err);
    return rc == DSA_OK ? ok() : rc;
}

size_t dsa_indexer_warmup_workspace_size(int T, int S, int H_I, int d_I)
{
    if (T < 0 || S < 1 || d_I != 128 || (H_I != 64 && H_I != 32))
        return 0;
    return warmup_workspace_bytes(T, S, H_I);
}

int dsa_indexer_warmup(const void *q, const void *kv, int H, float sm_scale, const void *q8, const float *q_scale,
                       const float *w, int H_I, int d_I, const void *k8, const float *k_scale, const int32_t *q_pos,
                       int T, int S, float *loss, float *dw, float *dq, float *dk, void *workspace,
                       size_t workspace_bytes, dsa_stream_t stream)
{
    if (T < 0 || S < 1)
        return fail(DSA_ERR_INVALID_ARG, "T < 0 or S < 1");
    if (T == 0)
        return ok();
    if (!q || !kv || !q8 || !q_scale || !w || !k8 || !k_scale || !q_pos || !loss || !dw || !dq || !dk)
        return fail(DSA_ERR_INVALID_ARG, "null pointer argument");
    if (H < 1 || H > 128)
        return fail(DSA_ERR_UNSUPPORTED, "H must be in [1, 128]");
    if (d_I != 128 || (H_I != 64 && H_I != 32))
        return fail(DSA_ERR_UNSUPPORTED, "warm-up: (H_I, d_I) must be (64, 128) or (32, 128)");
    if (!(sm_scale > 0.f) || sm_scale > 1e30f)
        return fail(DSA_ERR_INVALID_ARG, "sm_scale must be positive and finite");
    if (!aligned16(q) || !aligned16(kv) || !aligned16(q8) || !aligned16(k8) || !aligned16(dq))
        return fail(DSA_ERR_ALIGNMENT, "q, kv, q8, k8 and dq must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(DSA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    if (!workspace || workspace_bytes < warmup_workspace_bytes(T, S, H_I))
        return fail(DSA_ERR_WORKSPACE, "workspace missing or smaller than dsa_indexer_warmup_workspace_size");
    WarmupArgs a{q, kv, H, sm_scale, q8, q_scale, w, H_I, d_I, k8, k_scale, q_pos, T, S, loss, dw, dq, dk,
                 workspace, workspace_bytes};
    int rc = launch_warmup(a, reinterpret_cast<cudaStream_t>(stream), t_err, sizeof t_err);
    return rc == DSA_OK ? ok() : rc;
}

int dsa_quantize_fp8(const float *x, int64_t rows, int64_t cols, int scale_mode, void *codes, float *scale,
                     dsa_stream_t stream)
{
    if (rows < 0 || cols < 1)
        return fail(DSA_ERR_INVALID_ARG, "rows must be >= 0 and cols >= 1");
    if (scale_mode != DSA_SCALE_AMAX && scale_mode != DSA_SCALE_POW2)
        return fail(DSA_ERR_INVALID_ARG, "scale_mode must be DSA_SCALE_AMAX or DSA_SCALE_POW2");
    if (rows == 0)
        return ok();
    if (!x || !codes || !scale)
        return fail(DSA_ERR_INVALID_ARG, "null pointer argument");
    if (rows > (int64_t(1) << 40) / cols)
        return fail(DSA_ERR_UNSUPPORTED, "rows * cols too large");
    QuantizeArgs a{x, rows, cols, scale_mode, static_cast<uint8_t *>(codes), scale};
    int rc = launch_quantize(a, reinterpret_cast<cudaStream_t>(stream), t_err, sizeof t_err);
    return rc == DSA_OK ? ok() : rc;
}

int dsa_topk(const float *logits, int64_t ld, int T, const int32_t *valid_len, int k, int32_t *idx,
             dsa_stream_t stream)
{
    if (T < 0)
        return fail(DSA_ERR_INVALID_ARG, "T < 0");
    if (T == 0)
        return ok();
    if (!logits || !valid_len || !idx)
        return fail(DSA_ERR_INVALID_ARG, "null pointer argument");
    if (k < 1 || k > 4096)
        return fail(DSA_ERR_UNSUPPORTED, "k must be in [1, 4096]");
    if (ld < 1 || ld > (int64_t(1) << 28))
        return fail(DSA_ERR_UNSUPPORTED, "ld must be in [1, 2^28]");
    TopkArgs a{logits, ld, T, valid_len, k, idx};
    int rc = launch_topk(a, reinterpret_cast<cudaStream_t>(stream), t_err, sizeof t_err);
    return rc == DSA_OK ? ok() : rc;
}

int dsa_sparse_mla_prefill(const void *q, const void *kv, int S, const int32_t *idx, int T, int H, int k,
                           float sm_scale, void *out, float *lse, dsa_stream_t stream)
{
    if (T < 0 || S < 0)
        return fail(DSA_ERR_INVALID_ARG, "T < 0 or S < 0");
    if (T == 0)
        return ok();
    if (!q || !kv || !idx || !out || !lse)
        return fail(DSA_ERR_INVALID_ARG, "null pointer argument");
    if (H < 1 || H > 128)
        return fail(DSA_ERR_UNSUPPORTED, "H must be in [1, 128]");
    if (k < 1 || k > 4096)
        return fail(DSA_ERR_UNSUPPORTED, "k must be in [1, 4096]");
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out))
        return fail(DSA_ERR_ALIGNMENT, "q, kv and out must be 16-byte aligned");
    if (!(sm_scale > 0.f) || sm_scale > 1e30f)
        return fail(DSA_ERR_INVALID_ARG, "sm_scale must be positive and finite");
    MlaArgs a{};
    a.q = q;
    a.kv = kv;
    a.S = S;
    a.idx = idx;
    a.T = T;
    a.H = H;
    a.k = k;
    a.sm_scale = sm_scale;
    a.out = out;
    a.lse = lse;
    int rc = launch_mla_prefill(a, reinterpret_cast<cudaStream_t>(stream), t_err, sizeof t_err);
    return rc == DSA_OK ? ok() : rc;
}

size_t dsa_sparse_mla_decode_workspace_size(int B, int H, int k)
{
    if (B < 0 || H < 1 || H > 128 || k < 1 || k > 4096)
        return 0;
    return mla_decode_workspace_bytes(B, H, k);
}

int dsa_sparse_mla_decode_paged(const void *q, const void *kv_pool, int num_pages, int page_size,
                                const int32_t *block_table, int max_pages, const int32_t *ctx_len, const int32_t *idx,
                                int B, int H, int k, float sm_scale, void *out, float *lse, void *workspace,
                                size_t workspace_bytes, dsa_stream_t stream)
{
    if (B < 0)
        return fail(DSA_ERR_INVALID_ARG, "B < 0");
    if (B == 0)
        return ok();
    if (!q || !kv_pool || !block_table || !ctx_len || !idx || !out || !lse)
        return fail(DSA_ERR_INVALID_ARG, "null pointer argument");
    if (H < 1 || H > 128)
        return fail(DSA_ERR_UNSUPPORTED, "H must be in [1, 128]");
    if (k < 1 || k > 4096)
        return fail(DSA_ERR_UNSUPPORTED, "k must be in [1, 4096]");
    if (num_pages <= 0 || max_pages <= 0 || page_size <= 0)
        return fail(DSA_ERR_INVALID_ARG, "num_pages, max_pages and page_size must be positive");
    if ((int64_t)num_pages * page_size > (int64_t)INT32_MAX)
        return fail(DSA_ERR_UNSUPPORTED, "pool too large");
    if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out))
        return fail(DSA_ERR_ALIGNMENT, "q, kv_pool and out must be 16-byte aligned");
    if (!(sm_scale > 0.f) || sm_scale > 1e30f)
        return fail(DSA_ERR_INVALID_ARG, "sm_scale must be positive and finite");
    const size_t need = mla_decode_workspace_bytes(B, H, k);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(DSA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    MlaArgs a{};
    a.q = q;
    a.kv = kv_pool;
    a.S = num_pages * page_size;
    a.idx = idx;
    a.T = B;
    a.H = H;
    a.k = k;
    a.sm_scale = sm_scale;
    a.out = out;
    a.lse = lse;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.page_size = page_size;
    a.ctx_len = ctx_len;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    int rc = launch_mla_decode(a, reinterpret_cast<cudaStream_t>(stream), t_err, sizeof t_err);
    return rc == DSA_OK ? ok() : rc;
}

} // extern "C"

// ---------------------------------------------------------------------------
// Self-test of the failure detection: one CTA waits, through the same bounded
// mbarrier wait every pipeline uses, on a barrier that nothing arrives on.
namespace dsa {
namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, unsigned *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    grid_dep_wait();
    grid_dep_launch();
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // phase 0 never completes: the wait gives up after limit_ns, sets
    // DSA_DEV_TIMEOUT and the kernel returns
    mbar_wait_warp(b, 0, &abort_flag, status, limit_ns);
}

} // namespace
} // namespace dsa

extern "C" int dsa_selftest_wait_timeout(uint32_t limit_us, dsa_stream_t stream)
{
    if (limit_us == 0 || limit_us > 1000000u)
        return fail(DSA_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
    unsigned *status = device_status_ptr();
    if (!status)
        return fail(DSA_ERR_CUDA, "device status word unavailable");
    cudaError_t e = launch_pdl(wait_timeout_kernel, dim3(1), dim3(32), 0, reinterpret_cast<cudaStream_t>(stream), 1,
                               (uint64_t)limit_us * 1000u, status);
    if (e != cudaSuccess)
        return fail(DSA_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
    return ok();
}

// ---------------------------------------------------------------------------
// Allocation-free decode attention.  The workspace lives in this file-scope
// device array, which every device that loads the library holds until the
// process exits.  In host code the array's name only stands for it: the
// device address comes from cudaGetSymbolAddress, looked up once per device
// (with that device current) on the first call and kept.
namespace dsa {
namespace {

static __device__ __align__(256) unsigned char g_decode_static_ws[DSA_DECODE_STATIC_WS_BYTES];
void *g_decode_static_ws_ptr[kMaxDevices] = {};

// Device address of this device's static decode workspace, or null (message in *why).
void *decode_static_workspace(cudaError_t *why)
{
    *why = cudaSuccess;
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_decode_static_ws_ptr[d]) {
        void *p = nullptr;
        *why = cudaGetSymbolAddress(&p, g_decode_static_ws);
        if (*why != cudaSuccess || !p)
            return nullptr;
        g_decode_static_ws_ptr[d] = p;
    }
    return g_decode_static_ws_ptr[d];
}

} // namespace
} // namespace dsa

extern "C" int dsa_sparse_mla_decode_paged_noalloc(const void *q, const void *kv_pool, int num_pages, int page_size,
                                                   const int32_t *block_table, int max_pages, const int32_t *ctx_len,
                                                   const int32_t *idx, int B, int H, int k, float sm_scale, void *out,
                                                   float *lse, dsa_stream_t stream)
{
    // 0 for bad arguments too: those are then reported by the call below
    const size_t need = dsa_sparse_mla_decode_workspace_size(B, H, k);
    if (need > (size_t)DSA_DECODE_STATIC_WS_BYTES)
        return fail(DSA_ERR_WORKSPACE,
                    "decode with B=%d, H=%d, k=%d needs %zu bytes of workspace on this device, more than the "
                    "%zu-byte static buffer of the allocation-free entry point",
                    B, H, k, need, (size_t)DSA_DECODE_STATIC_WS_BYTES);
    cudaError_t why;
    void *ws = decode_static_workspace(&why);
    if (!ws)
        return fail(DSA_ERR_CUDA, "address of the static decode workspace: %s",
                    why == cudaSuccess ? "no current device" : cudaGetErrorString(why));
    return dsa_sparse_mla_decode_paged(q, kv_pool, num_pages, page_size, block_table, max_pages, ctx_len, idx, B, H, k,
                                       sm_scale, out, lse, ws, (size_t)DSA_DECODE_STATIC_WS_BYTES, stream);
}
