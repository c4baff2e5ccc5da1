// Prefill from host memory: the whole hot path (indexer -> top-k -> sparse MLA)
// on inputs that sit in host memory, with the outputs returned to host memory.
//
// Query rows go in chunks (short ones at both ends, see chunk_starts), taken
// from the last rows to the first: the first chunk processed brings in the keys
// of every row (a few tens of MB against GBs of queries), and the chunks whose
// kernels outlast their input copies (long rows) run while the copies of the
// next ones proceed; the short rows at the end are copy-bound but few.
// Chunk c's inputs are copied host -> device on one
// stream, its three kernels run on the caller's stream, and its outputs are
// copied device -> host on a third stream; four buffer slots let the input
// copies run up to three chunks ahead of the kernels (two: 35.3 ms per call at
// L = 32768 against 34.9 ms, the copy-bound chunks at the end waiting on their
// inputs) and the output copies of earlier chunks overlap them.  The key-side tensors (k8, k_scale, kv) stay on the device for the
// whole call and are copied in as far as each chunk's positions need them.
// Per row the work and its order are those of the device entry points, so the
// results are the same bytes.
#include <cuda_runtime.h>

#include <algorithm>
#include <limits>
#include <mutex>
#include <vector>
#include <stdio.h>

#include "common.cuh"
#include "launch.h"

namespace dsa {
namespace {

constexpr int kMaxDev = 64;
constexpr int kSlots = 4;

// valid_len of the top-k stage: the query position plus one (the query itself
// is a candidate).
__global__ void pos_to_len_kernel(const int32_t *__restrict__ q_pos, int n, int32_t *__restrict__ len)
{
    grid_dep_wait();
    grid_dep_launch();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n)
        len[i] = q_pos[i] + 1;
}

// Events of a chunk's timeline (dsa_prefill_host_trace), in this order.
enum { kInBegin, kInEnd, kKernBegin, kKernEnd, kOutBegin, kOutEnd, kTraceEvents };

// Copy streams and events of one device, created on its first call and kept;
// the timeline record only while dsa_prefill_host_trace has it on.
struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_ready[kSlots] = {}, slot_done[kSlots] = {}, out_copied[kSlots] = {};
    int trace_cap = 0, trace_n = 0, trace_calls = 0; // chunks the record holds, has, calls recorded
    cudaEvent_t trace_t0 = nullptr;                  // start of the first recorded call
    std::vector<cudaEvent_t> trace_ev;               // kTraceEvents per chunk
    std::vector<int32_t> trace_call, trace_rows;     // per chunk: call number, query rows
};
HostPipe g_pipe[kMaxDev];
std::mutex g_pipe_mu[kMaxDev];

// Releases what a partly built pipe holds, so that the next call starts clean.
void drop_pipe(HostPipe &p)
{
    for (cudaStream_t *st : {&p.h2d, &p.d2h}) {
        if (*st)
            cudaStreamDestroy(*st);
        *st = nullptr;
    }
    for (cudaEvent_t *e : {&p.start, &p.end}) {
        if (*e)
            cudaEventDestroy(*e);
        *e = nullptr;
    }
    for (int s = 0; s < kSlots; ++s)
        for (cudaEvent_t *e : {&p.in_ready[s], &p.slot_done[s], &p.out_copied[s]}) {
            if (*e)
                cudaEventDestroy(*e);
            *e = nullptr;
        }
    p.ready = false;
}

bool make_pipe(HostPipe &p)
{
    if (p.ready)
        return true;
    auto ev = [](cudaEvent_t *e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
    bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess && ev(&p.start) && ev(&p.end);
    for (int s = 0; ok && s < kSlots; ++s)
        ok = ev(&p.in_ready[s]) && ev(&p.slot_done[s]) && ev(&p.out_copied[s]);
    if (!ok) {
        drop_pipe(p);
        return false;
    }
    p.ready = true;
    return true;
}

void free_trace(HostPipe &p)
{
    for (cudaEvent_t e : p.trace_ev)
        cudaEventDestroy(e);
    if (p.trace_t0)
        cudaEventDestroy(p.trace_t0);
    p.trace_ev.clear();
    p.trace_call.clear();
    p.trace_rows.clear();
    p.trace_t0 = nullptr;
    p.trace_cap = p.trace_n = p.trace_calls = 0;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Chunk starts for T rows in chunks of at most C: C/4 and C/2 first, then C,
// and a last chunk of C/4.  Taken in reverse, the first chunk processed is
// short (the kernels start after a short copy) and so is the last (little is
// left to copy out after the last kernels).  Returns the starts and T.
std::vector<int> chunk_starts(int T, int C)
{
    std::vector<int> st;
    const int q = std::max(1, C / 4), h = std::max(1, C / 2);
    int r = 0;
    for (int first : {q, h}) {
        if (r < T) {
            st.push_back(r);
            r += std::min(first, T - r);
        }
    }
    while (T - r > C + q) {
        st.push_back(r);
        r += C;
    }
    if (T - r > q) {
        st.push_back(r);
        r = T - q;
    }
    if (r < T)
        st.push_back(r);
    st.push_back(T);
    return st;
}

// Workspace layout; every region starts on a 256-byte boundary.
struct Layout {
    size_t k8, ks, kv, logits, idx;              // shared regions
    size_t q8[kSlots], qs[kSlots], w[kSlots], qpos[kSlots], len[kSlots], q[kSlots], out[kSlots], lse[kSlots];
    size_t total;
};

Layout layout(int S, int H_I, int d_I, int H, int k, int C)
{
    Layout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += up256(bytes);
        return at;
    };
    L.k8 = take((size_t)S * d_I);
    L.ks = take((size_t)S * 4);
    L.kv = take((size_t)S * 576 * 2);
    L.logits = take((size_t)C * S * 4);
    L.idx = take((size_t)C * k * 4);
    for (int s = 0; s < kSlots; ++s) {
        L.q8[s] = take((size_t)C * H_I * d_I);
        L.qs[s] = take((size_t)C * 4);
        L.w[s] = take((size_t)C * H_I * 4);
        L.qpos[s] = take((size_t)C * 4);
        L.len[s] = take((size_t)C * 4);
        L.q[s] = take((size_t)C * H * 576 * 2);
        L.out[s] = take((size_t)C * H * 512 * 2);
        L.lse[s] = take((size_t)C * H * 4);
    }
    L.total = o;
    return L;
}

} // namespace
} // namespace dsa

using namespace dsa;

extern "C" size_t dsa_prefill_host_workspace_size(int T, int S, int H_I, int d_I, int H, int k, int chunk_rows)
{
    if (T < 1 || S < 1 || H_I < 1 || d_I < 1 || H < 1 || H > 128 || k < 1 || k > 4096 || chunk_rows < 1)
        return 0;
    return layout(S, H_I, d_I, H, k, std::min(T, chunk_rows)).total;
}

extern "C" int dsa_prefill_host(const void *q8, const float *q_scale, const float *w, const int32_t *q_pos,
                                const void *k8, const float *k_scale, const void *q, const void *kv, int T, int S,
                                int H_I, int d_I, int H, int k, float sm_scale, void *out, float *lse,
                                int chunk_rows, void *workspace, size_t workspace_bytes, dsa_stream_t stream)
{
    // Argument errors are reported by the entry points called below, except
    // those only this call can see.
    if (T < 0 || chunk_rows < 1)
        return report_error(DSA_ERR_INVALID_ARG, "T < 0 or chunk_rows < 1");
    if (T == 0)
        return DSA_OK;
    if (!q8 || !q_scale || !w || !q_pos || !k8 || !k_scale || !q || !kv || !out || !lse || !workspace)
        return report_error(DSA_ERR_INVALID_ARG, "null pointer argument");
    if (S < 1 || H_I < 1 || d_I < 1 || H < 1 || H > 128 || k < 1 || k > 4096)
        return report_error(DSA_ERR_INVALID_ARG, "bad shape (S, H_I, d_I, H or k)");
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return report_error(DSA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    const int C = std::min(T, chunk_rows);
    const Layout L = layout(S, H_I, d_I, H, k, C);
    if (workspace_bytes < L.total)
        return report_error(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", L.total,
                                workspace_bytes);
    for (int r = 0; r < T; ++r)
        if (q_pos[r] < 0 || q_pos[r] >= S)
            return report_error(DSA_ERR_INVALID_ARG, "q_pos[%d] = %d outside [0, S = %d)", r, q_pos[r], S);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return report_error(DSA_ERR_CUDA, "no current device");
    std::lock_guard<std::mutex> lk(g_pipe_mu[dev]); // one call enqueues at a time per device
    HostPipe &P = g_pipe[dev];
    if (!make_pipe(P))
        return report_error(DSA_ERR_CUDA, "creating the copy streams and events failed");
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const char *hq8 = static_cast<const char *>(q8), *hk8 = static_cast<const char *>(k8);
    const char *hq = static_cast<const char *>(q), *hkv = static_cast<const char *>(kv);
    char *hout = static_cast<char *>(out);

    cudaError_t e = cudaSuccess;
    auto chk = [&](cudaError_t x) {
        if (e == cudaSuccess && x != cudaSuccess)
            e = x;
    };
    // the workspace may still be in use by earlier work on the caller's stream
    if (P.trace_cap > 0 && P.trace_calls == 0)
        chk(cudaEventRecord(P.trace_t0, cs)); // before the copy streams are released
    chk(cudaEventRecord(P.start, cs));
    chk(cudaStreamWaitEvent(P.h2d, P.start, 0));
    chk(cudaStreamWaitEvent(P.d2h, P.start, 0));
    // the chunk's timeline events while the record has room, else none
    auto mark = [&](int j, int which, cudaStream_t st) {
        if (j >= 0)
            chk(cudaEventRecord(P.trace_ev[static_cast<size_t>(j) * kTraceEvents + which], st));
    };

    int keys_in = 0; // key rows [0, keys_in) already on the device
    const std::vector<int> starts = chunk_starts(T, C);
    const int nchunks = static_cast<int>(starts.size()) - 1;
    int rc = DSA_OK;
    for (int c = 0; c < nchunks && rc == DSA_OK && e == cudaSuccess; ++c) {
        const int s = c % kSlots;
        // last rows first: their chunk brings in the keys of every row at once (a few
        // tens of MB), and the chunks whose kernels outlast their copies come first
        const int cr = nchunks - 1 - c;
        const int r0 = starts[cr], n = starts[cr + 1] - r0; // 1 <= n <= C
        int kmax = 0;
        for (int r = r0; r < r0 + n; ++r)
            kmax = std::max(kmax, q_pos[r] + 1);
        int tj = -1; // this chunk's slot in the timeline record
        if (P.trace_n < P.trace_cap) {
            tj = P.trace_n++;
            P.trace_call[tj] = P.trace_calls;
            P.trace_rows[tj] = n;
        }
        // ---- inputs (the slot's previous chunk must be done with them)
        if (c >= kSlots)
            chk(cudaStreamWaitEvent(P.h2d, P.slot_done[s], 0));
        mark(tj, kInBegin, P.h2d);
        if (kmax > keys_in) {
            const size_t a = keys_in, b = kmax;
            chk(cudaMemcpyAsync(ws + L.k8 + a * d_I, hk8 + a * d_I, (b - a) * d_I, cudaMemcpyHostToDevice, P.h2d));
            chk(cudaMemcpyAsync(ws + L.ks + a * 4, k_scale + a, (b - a) * 4, cudaMemcpyHostToDevice, P.h2d));
            chk(cudaMemcpyAsync(ws + L.kv + a * 1152, hkv + a * 1152, (b - a) * 1152, cudaMemcpyHostToDevice,
                                P.h2d));
            keys_in = kmax;
        }
        chk(cudaMemcpyAsync(ws + L.q8[s], hq8 + (size_t)r0 * H_I * d_I, (size_t)n * H_I * d_I,
                            cudaMemcpyHostToDevice, P.h2d));
        chk(cudaMemcpyAsync(ws + L.qs[s], q_scale + r0, (size_t)n * 4, cudaMemcpyHostToDevice, P.h2d));
        chk(cudaMemcpyAsync(ws + L.w[s], w + (size_t)r0 * H_I, (size_t)n * H_I * 4, cudaMemcpyHostToDevice, P.h2d));
        chk(cudaMemcpyAsync(ws + L.qpos[s], q_pos + r0, (size_t)n * 4, cudaMemcpyHostToDevice, P.h2d));
        chk(cudaMemcpyAsync(ws + L.q[s], hq + (size_t)r0 * H * 1152, (size_t)n * H * 1152, cudaMemcpyHostToDevice,
                            P.h2d));
        mark(tj, kInEnd, P.h2d);
        chk(cudaEventRecord(P.in_ready[s], P.h2d));
        // ---- kernels (the slot's previous outputs must have been copied out)
        chk(cudaStreamWaitEvent(cs, P.in_ready[s], 0));
        if (c >= kSlots)
            chk(cudaStreamWaitEvent(cs, P.out_copied[s], 0));
        mark(tj, kKernBegin, cs);
        if (e != cudaSuccess)
            break;
        const int32_t *qpos_d = reinterpret_cast<const int32_t *>(ws + L.qpos[s]);
        int32_t *len_d = reinterpret_cast<int32_t *>(ws + L.len[s]);
        chk(launch_pdl(pos_to_len_kernel, dim3((n + 255) / 256), dim3(256), 0, cs, 1, qpos_d, n, len_d));
        float *logits = reinterpret_cast<float *>(ws + L.logits);
        int32_t *idx = reinterpret_cast<int32_t *>(ws + L.idx);
        rc = dsa_indexer_logits(ws + L.q8[s], reinterpret_cast<const float *>(ws + L.qs[s]),
                                reinterpret_cast<const float *>(ws + L.w[s]), n, H_I, d_I, ws + L.k8,
                                reinterpret_cast<const float *>(ws + L.ks), kmax, nullptr, 0, 0, 0, qpos_d, logits, S,
                                stream);
        if (rc == DSA_OK)
            rc = dsa_topk(logits, S, n, len_d, k, idx, stream);
        if (rc == DSA_OK)
            rc = dsa_sparse_mla_prefill(ws + L.q[s], ws + L.kv, kmax, idx, n, H, k, sm_scale, ws + L.out[s],
                                        reinterpret_cast<float *>(ws + L.lse[s]), stream);
        if (rc != DSA_OK)
            break;
        mark(tj, kKernEnd, cs);
        chk(cudaEventRecord(P.slot_done[s], cs));
        // ---- outputs
        chk(cudaStreamWaitEvent(P.d2h, P.slot_done[s], 0));
        mark(tj, kOutBegin, P.d2h);
        chk(cudaMemcpyAsync(hout + (size_t)r0 * H * 1024, ws + L.out[s], (size_t)n * H * 1024,
                            cudaMemcpyDeviceToHost, P.d2h));
        chk(cudaMemcpyAsync(lse + (size_t)r0 * H, ws + L.lse[s], (size_t)n * H * 4, cudaMemcpyDeviceToHost, P.d2h));
        mark(tj, kOutEnd, P.d2h);
        chk(cudaEventRecord(P.out_copied[s], P.d2h));
    }
    if (P.trace_cap > 0)
        ++P.trace_calls;
    // the call is complete on the caller's stream once every copy has landed
    chk(cudaEventRecord(P.end, P.d2h));
    chk(cudaEventRecord(P.start, P.h2d));
    chk(cudaStreamWaitEvent(cs, P.end, 0));
    chk(cudaStreamWaitEvent(cs, P.start, 0));
    if (rc != DSA_OK)
        return rc;
    if (e != cudaSuccess)
        return report_error(DSA_ERR_CUDA, "host prefill: %s", cudaGetErrorString(e));
    return DSA_OK;
}

extern "C" int dsa_prefill_host_trace(int max_chunks)
{
    if (max_chunks < 0 || max_chunks > (1 << 20))
        return report_error(DSA_ERR_INVALID_ARG, "max_chunks = %d outside [0, 2^20]", max_chunks);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return report_error(DSA_ERR_CUDA, "no current device");
    std::lock_guard<std::mutex> lk(g_pipe_mu[dev]);
    HostPipe &P = g_pipe[dev];
    free_trace(P);
    if (max_chunks == 0)
        return DSA_OK;
    bool ok = cudaEventCreate(&P.trace_t0) == cudaSuccess;
    P.trace_ev.assign(static_cast<size_t>(max_chunks) * kTraceEvents, nullptr);
    for (size_t i = 0; ok && i < P.trace_ev.size(); ++i)
        ok = cudaEventCreate(&P.trace_ev[i]) == cudaSuccess;
    if (!ok) {
        free_trace(P);
        return report_error(DSA_ERR_CUDA, "creating the timeline events failed");
    }
    P.trace_call.assign(max_chunks, 0);
    P.trace_rows.assign(max_chunks, 0);
    P.trace_cap = max_chunks;
    return DSA_OK;
}

extern "C" int dsa_prefill_host_trace_read(float *ms, int32_t *call, int32_t *rows, int max_chunks, int *n_out)
{
    if (!ms || !call || !rows || !n_out || max_chunks < 0)
        return report_error(DSA_ERR_INVALID_ARG, "null pointer or max_chunks < 0");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return report_error(DSA_ERR_CUDA, "no current device");
    std::lock_guard<std::mutex> lk(g_pipe_mu[dev]);
    HostPipe &P = g_pipe[dev];
    const int n = std::min(P.trace_n, max_chunks);
    for (int j = 0; j < n; ++j) {
        for (int ev = 0; ev < kTraceEvents; ++ev) {
            cudaEvent_t x = P.trace_ev[static_cast<size_t>(j) * kTraceEvents + ev];
            float t = 0.f;
            // an event a failed call never recorded reads as NaN
            if (cudaEventSynchronize(x) != cudaSuccess || cudaEventElapsedTime(&t, P.trace_t0, x) != cudaSuccess) {
                cudaGetLastError();
                t = std::numeric_limits<float>::quiet_NaN();
            }
            ms[static_cast<size_t>(j) * kTraceEvents + ev] = t;
        }
        call[j] = P.trace_call[j];
        rows[j] = P.trace_rows[j];
    }
    *n_out = n;
    return DSA_OK;
}
