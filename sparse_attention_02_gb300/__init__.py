"""Python binding of libdsa.so, the GB300 (sm_103a) DSA hot path.

Argument marshalling only: each function checks dtypes/shapes, passes raw
device pointers and the current CUDA stream to the C entry point of the same
name (declared in include/dsa.h) and raises ``DsaError`` on a non-zero status.
Every step of the computation runs in the library's CUDA kernels; there is no
host or PyTorch fallback, and importing this package fails loudly when the
library has not been built.

PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_OK = 0
DSA_DEV_TIMEOUT = 0x1
DSA_DEV_BAD_POSITION = 0x2
DSA_DEV_BAD_PAGE = 0x4

_lib = None


class DsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dsa error {code}: {msg}")
        self.code = code


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libdsa.so (built by ``sparse_attention_02_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with `python -m sparse_attention_02_gb300.build` "
                           "(or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(p)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.dsa_last_error.restype = ctypes.c_char_p
    lib.dsa_version.restype = i32
    lib.dsa_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.dsa_quantize_fp8.argtypes = [P, i64, i64, i32, P, P, P]
    lib.dsa_indexer_logits.argtypes = [P, P, P, i32, i32, i32, P, P, i32, P, i32, i32, i32, P, P, i64, P]
    lib.dsa_topk.argtypes = [P, i64, i32, P, i32, P, P]
    lib.dsa_sparse_mla_prefill.argtypes = [P, P, i32, P, i32, i32, i32, f32, P, P, P]
    lib.dsa_sparse_mla_decode_paged.argtypes = [P, P, i32, i32, P, i32, P, P, i32, i32, i32, f32, P, P, P, sz, P]
    lib.dsa_sparse_mla_decode_paged_noalloc.argtypes = [P, P, i32, i32, P, i32, P, P, i32, i32, i32, f32, P, P, P]
    lib.dsa_prefill_host.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P, i32, P, sz, P]
    lib.dsa_prefill_host_workspace_size.restype = sz
    lib.dsa_prefill_host_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.dsa_prefill_host_trace.argtypes = [i32]
    lib.dsa_prefill_host_trace_read.argtypes = [P, P, P, i32, ctypes.POINTER(i32)]
    lib.dsa_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
    lib.dsa_selftest_wait_timeout.restype = i32
    lib.dsa_sparse_mla_decode_workspace_size.restype = sz
    lib.dsa_sparse_mla_decode_workspace_size.argtypes = [i32, i32, i32]
    lib.dsa_indexer_topk.argtypes = [P, P, P, i32, i32, i32, P, P, i32, P, i32, P, P, sz, P]
    lib.dsa_indexer_warmup.argtypes = [P, P, i32, f32, P, P, P, i32, i32, P, P, P, i32, i32, P, P, P, P, P, sz, P]
    lib.dsa_indexer_warmup_workspace_size.restype = sz
    lib.dsa_indexer_warmup_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.dsa_indexer_topk_workspace_size.restype = sz
    lib.dsa_indexer_topk_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    for name in ("dsa_quantize_fp8", "dsa_indexer_logits", "dsa_topk", "dsa_indexer_topk", "dsa_indexer_warmup",
                 "dsa_sparse_mla_prefill",
                 "dsa_sparse_mla_decode_paged",
                 "dsa_sparse_mla_decode_paged_noalloc", "dsa_prefill_host", "dsa_prefill_host_trace",
                 "dsa_prefill_host_trace_read", "dsa_get_device_status"):
        getattr(lib, name).restype = i32
    if path is None:
        _lib = lib
    return lib


def _check(rc: int):
    if rc != DSA_OK:
        raise DsaError(rc, load_library().dsa_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _same_device(t: torch.Tensor, name: str):
    # the library runs on the current device (cudaGetDevice); a tensor elsewhere would
    # hand it another GPU's pointer
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{cur}")


def _need(t: torch.Tensor, dtype, name: str, dim: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    _same_device(t, name)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name}: expected {dim} dims, got {t.dim()}")


def _need_rows(t: torch.Tensor, dtype, name: str):
    """A 2-D tensor whose rows may be strided (leading dimension >= width)."""
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or t.dim() != 2:
        raise TypeError(f"{name}: expected a 2-D CUDA {dtype} tensor")
    _same_device(t, name)
    if t.stride(1) != 1 or t.stride(0) < t.shape[1]:
        raise ValueError(f"{name}: rows must be contiguous with a leading dimension >= width")


DSA_SCALE_AMAX = 0
DSA_SCALE_POW2 = 1


def dsa_quantize_fp8(x, codes, scale, mode: int = DSA_SCALE_AMAX, stream=None):
    """Per-row FP8 quantisation: x fp32 [rows, ...] -> codes uint8 (E4M3, same shape), scale fp32 [rows].

    mode DSA_SCALE_AMAX: scale = amax / 448; DSA_SCALE_POW2: the smallest power of two >= that.
    """
    _need(x, torch.float32, "x")
    _need(codes, torch.uint8, "codes")
    _need(scale, torch.float32, "scale", 1)
    if x.dim() < 1 or tuple(codes.shape) != tuple(x.shape) or scale.shape[0] != x.shape[0]:
        raise ValueError("codes must match x's shape and scale must have one entry per row")
    rows = x.shape[0]
    cols = x.numel() // rows if rows > 0 else 1
    _check(load_library().dsa_quantize_fp8(_ptr(x), rows, cols, int(mode), _ptr(codes), _ptr(scale),
                                           _stream(stream)))
    return codes, scale


def dsa_indexer_logits(q8, q_scale, w, k8, k_scale, q_pos, logits, block_table=None, stream=None):
    """Lightning-indexer scores into ``logits`` [T, ld] (fp32).

    q8 uint8 [T, H_I, d_I] (E4M3 codes), q_scale fp32 [T], w fp32 [T, H_I], q_pos int32 [T].
    Contiguous keys: k8 uint8 [S, d_I], k_scale fp32 [S].  Paged keys: k8 uint8
    [num_pages, page_size, d_I], k_scale fp32 [num_pages, page_size] and
    block_table int32 [T, max_pages].  ``logits`` rows may be strided
    (leading dimension = logits.stride(0)).
    """
    _need(q8, torch.uint8, "q8", 3)
    T, HI, dI = q8.shape
    _need(q_scale, torch.float32, "q_scale", 1)
    _need(w, torch.float32, "w", 2)
    _need(q_pos, torch.int32, "q_pos", 1)
    _need_rows(logits, torch.float32, "logits")
    _need(k8, torch.uint8, "k8")
    _need(k_scale, torch.float32, "k_scale")
    if q_scale.shape[0] != T or tuple(w.shape) != (T, HI) or q_pos.shape[0] != T or logits.shape[0] != T:
        raise ValueError("inconsistent query shapes")
    if block_table is None:
        if k8.dim() != 2 or k8.shape[1] != dI or k_scale.shape != (k8.shape[0],):
            raise ValueError("k8 must be [S, d_I] and k_scale [S]")
        S, mp, npg, ps = k8.shape[0], 0, 0, 0
    else:
        _need(block_table, torch.int32, "block_table", 2)
        if k8.dim() != 3 or k8.shape[2] != dI or tuple(k_scale.shape) != tuple(k8.shape[:2]):
            raise ValueError("paged: k8 must be [P, page, d_I] and k_scale [P, page]")
        if block_table.shape[0] != T:
            raise ValueError("block_table must have one row per query")
        S, mp, npg, ps = 0, block_table.shape[1], k8.shape[0], k8.shape[1]
    lib = load_library()
    _check(lib.dsa_indexer_logits(_ptr(q8), _ptr(q_scale), _ptr(w), T, HI, dI, _ptr(k8), _ptr(k_scale), S,
                                  _ptr(block_table), mp, npg, ps, _ptr(q_pos), _ptr(logits), logits.stride(0),
                                  _stream(stream)))
    return logits


def dsa_topk(logits, valid_len, k: int, idx, stream=None):
    """Top-k indices (ascending, -1 padded) of each row of ``logits`` [T, >= max valid_len]
    (rows may be strided) into ``idx`` [T, k]."""
    _need_rows(logits, torch.float32, "logits")
    _need(valid_len, torch.int32, "valid_len", 1)
    _need(idx, torch.int32, "idx", 2)
    T = logits.shape[0]
    if valid_len.shape[0] != T or tuple(idx.shape) != (T, k):
        raise ValueError("inconsistent shapes")
    _check(load_library().dsa_topk(_ptr(logits), logits.stride(0), T, _ptr(valid_len), k, _ptr(idx),
                                   _stream(stream)))
    return idx


def dsa_indexer_topk_workspace_size(T: int, S: int, H_I: int, d_I: int, k: int) -> int:
    return int(load_library().dsa_indexer_topk_workspace_size(T, S, H_I, d_I, k))


def dsa_indexer_topk(q8, q_scale, w, k8, k_scale, q_pos, k: int, idx, workspace=None, stream=None):
    """Fused indexer -> top-k: the top-k key positions of each query row into ``idx`` [T, k]
    (ascending, -1 padded) without writing the index scores.  Inputs as for
    dsa_indexer_logits with contiguous keys.  ``workspace``: a uint8 CUDA tensor of at least
    dsa_indexer_topk_workspace_size(T, S, H_I, d_I, k) bytes; taken from PyTorch's
    allocator when None."""
    _need(q8, torch.uint8, "q8", 3)
    T, HI, dI = q8.shape
    _need(q_scale, torch.float32, "q_scale", 1)
    _need(w, torch.float32, "w", 2)
    _need(q_pos, torch.int32, "q_pos", 1)
    _need(k8, torch.uint8, "k8", 2)
    _need(k_scale, torch.float32, "k_scale", 1)
    _need(idx, torch.int32, "idx", 2)
    S = k8.shape[0]
    if q_scale.shape[0] != T or tuple(w.shape) != (T, HI) or q_pos.shape[0] != T or tuple(idx.shape) != (T, k) \
            or k8.shape[1] != dI or k_scale.shape[0] != S:
        raise ValueError("inconsistent shapes")
    if workspace is None:
        need = dsa_indexer_topk_workspace_size(T, S, HI, dI, k)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q8.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    _same_device(workspace, "workspace")
    _check(load_library().dsa_indexer_topk(_ptr(q8), _ptr(q_scale), _ptr(w), T, HI, dI, _ptr(k8), _ptr(k_scale), S,
                                           _ptr(q_pos), k, _ptr(idx), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream)))
    return idx


def dsa_indexer_warmup_workspace_size(T: int, S: int, H_I: int, d_I: int) -> int:
    return int(load_library().dsa_indexer_warmup_workspace_size(T, S, H_I, d_I))


def dsa_indexer_warmup(q, kv, sm_scale: float, q8, q_scale, w, k8, k_scale, q_pos, loss, dw, dq, dk,
                       workspace=None, stream=None):
    """Indexer warm-up: the KL loss of the index scores' softmax against the main attention's
    head-averaged dense distribution, and its gradients.  q bf16 [T, H, 576], kv bf16 [S, 576];
    indexer inputs as for dsa_indexer_logits (contiguous keys); outputs fp32 loss [T],
    dw [T, H_I], dq [T, H_I, d_I], dk [S, d_I].  ``workspace``: a uint8 CUDA tensor of at least
    dsa_indexer_warmup_workspace_size(T, S, H_I, d_I) bytes; taken from PyTorch when None."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv", 2)
    _need(q8, torch.uint8, "q8", 3)
    _need(q_scale, torch.float32, "q_scale", 1)
    _need(w, torch.float32, "w", 2)
    _need(k8, torch.uint8, "k8", 2)
    _need(k_scale, torch.float32, "k_scale", 1)
    _need(q_pos, torch.int32, "q_pos", 1)
    for t, name, dim in ((loss, "loss", 1), (dw, "dw", 2), (dq, "dq", 3), (dk, "dk", 2)):
        _need(t, torch.float32, name, dim)
    T, H, D = q.shape
    S = kv.shape[0]
    _, HI, dI = q8.shape
    if D != 576 or kv.shape[1] != 576 or q8.shape[0] != T or q_scale.shape[0] != T or tuple(w.shape) != (T, HI) \
            or tuple(k8.shape) != (S, dI) or k_scale.shape[0] != S or q_pos.shape[0] != T \
            or loss.shape[0] != T or tuple(dw.shape) != (T, HI) or tuple(dq.shape) != (T, HI, dI) \
            or tuple(dk.shape) != (S, dI):
        raise ValueError("inconsistent shapes")
    if workspace is None:
        need = dsa_indexer_warmup_workspace_size(T, S, HI, dI)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    _same_device(workspace, "workspace")
    _check(load_library().dsa_indexer_warmup(_ptr(q), _ptr(kv), H, float(sm_scale), _ptr(q8), _ptr(q_scale),
                                             _ptr(w), HI, dI, _ptr(k8), _ptr(k_scale), _ptr(q_pos), T, S, _ptr(loss),
                                             _ptr(dw), _ptr(dq), _ptr(dk), _ptr(workspace),
                                             workspace.numel() * workspace.element_size(), _stream(stream)))
    return loss, dw, dq, dk


def dsa_sparse_mla_prefill(q, kv, idx, sm_scale: float, out, lse, stream=None):
    """Sparse MQA-mode MLA: q bf16 [T, H, 576], kv bf16 [S, 576], idx int32 [T, k]
    -> out bf16 [T, H, 512], lse fp32 [T, H]."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv, torch.bfloat16, "kv", 2)
    _need(idx, torch.int32, "idx", 2)
    _need(out, torch.bfloat16, "out", 3)
    _need(lse, torch.float32, "lse", 2)
    T, H, D = q.shape
    S = kv.shape[0]
    k = idx.shape[1]
    if D != 576 or kv.shape[1] != 576 or idx.shape[0] != T or tuple(out.shape) != (T, H, 512) \
            or tuple(lse.shape) != (T, H):
        raise ValueError("inconsistent shapes (D must be 576, Dv 512)")
    _check(load_library().dsa_sparse_mla_prefill(_ptr(q), _ptr(kv), S, _ptr(idx), T, H, k, float(sm_scale),
                                                 _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def dsa_sparse_mla_decode_workspace_size(B: int, H: int, k: int) -> int:
    return int(load_library().dsa_sparse_mla_decode_workspace_size(B, H, k))


def dsa_sparse_mla_decode_paged(q, kv_pool, block_table, ctx_len, idx, sm_scale: float, out, lse,
                                workspace=None, stream=None):
    """Paged decode attention: q bf16 [B, H, 576], kv_pool bf16 [P, page, 576],
    block_table int32 [B, max_pages], ctx_len int32 [B], idx int32 [B, k] (logical positions).
    ``workspace``: a uint8 CUDA tensor of at least dsa_sparse_mla_decode_workspace_size(B, H, k)
    bytes; when None and the call needs one, it is taken from PyTorch's allocator."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_pool, torch.bfloat16, "kv_pool", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    _need(idx, torch.int32, "idx", 2)
    _need(out, torch.bfloat16, "out", 3)
    _need(lse, torch.float32, "lse", 2)
    B, H, D = q.shape
    P, ps, D2 = kv_pool.shape
    k = idx.shape[1]
    if D != 576 or D2 != 576 or block_table.shape[0] != B or ctx_len.shape[0] != B or idx.shape[0] != B \
            or tuple(out.shape) != (B, H, 512) or tuple(lse.shape) != (B, H):
        raise ValueError("inconsistent shapes")
    ws_bytes = 0
    if workspace is None:
        need = dsa_sparse_mla_decode_workspace_size(B, H, k)
        if need:  # device memory from PyTorch's caching allocator (256-byte aligned)
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().dsa_sparse_mla_decode_paged(_ptr(q), _ptr(kv_pool), P, ps, _ptr(block_table),
                                                      block_table.shape[1], _ptr(ctx_len), _ptr(idx), B, H, k,
                                                      float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                                      ws_bytes, _stream(stream)))
    return out, lse


def dsa_sparse_mla_decode_paged_noalloc(q, kv_pool, block_table, ctx_len, idx, sm_scale: float, out, lse,
                                        stream=None):
    """dsa_sparse_mla_decode_paged for callers that cannot allocate device memory:
    the library's static device buffer serves as the workspace, and this wrapper
    allocates nothing either.  Same arguments, minus the workspace."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_pool, torch.bfloat16, "kv_pool", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    _need(idx, torch.int32, "idx", 2)
    _need(out, torch.bfloat16, "out", 3)
    _need(lse, torch.float32, "lse", 2)
    B, H, D = q.shape
    P, ps, D2 = kv_pool.shape
    k = idx.shape[1]
    if D != 576 or D2 != 576 or block_table.shape[0] != B or ctx_len.shape[0] != B or idx.shape[0] != B \
            or tuple(out.shape) != (B, H, 512) or tuple(lse.shape) != (B, H):
        raise ValueError("inconsistent shapes")
    _check(load_library().dsa_sparse_mla_decode_paged_noalloc(_ptr(q), _ptr(kv_pool), P, ps, _ptr(block_table),
                                                              block_table.shape[1], _ptr(ctx_len), _ptr(idx), B, H,
                                                              k, float(sm_scale), _ptr(out), _ptr(lse),
                                                              _stream(stream)))
    return out, lse


def _host(t: torch.Tensor, dtype, name: str, dim: int):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.is_cuda or not t.is_contiguous() or t.dim() != dim:
        raise ValueError(f"{name}: expected a contiguous {dim}-d host tensor of {dtype}")


def dsa_prefill_host_workspace_size(T: int, S: int, H_I: int, d_I: int, H: int, k: int, chunk_rows: int) -> int:
    return int(load_library().dsa_prefill_host_workspace_size(T, S, H_I, d_I, H, k, chunk_rows))


def dsa_prefill_host(q8, q_scale, w, q_pos, k8, k_scale, q, kv, sm_scale: float, k: int, out, lse,
                     chunk_rows: int = 4096, workspace=None, stream=None):
    """The whole prefill path on HOST tensors (pinned for overlapped copies): q8 uint8 [T, H_I, d_I],
    q_scale f32 [T], w f32 [T, H_I], q_pos i32 [T], k8 uint8 [S, d_I], k_scale f32 [S], q bf16 [T, H, 576],
    kv bf16 [S, 576] -> out bf16 [T, H, 512], lse f32 [T, H] (host).  ``workspace``: a uint8 CUDA tensor of
    dsa_prefill_host_workspace_size(...) bytes, taken from PyTorch's allocator when None."""
    _host(q8, torch.uint8, "q8", 3)
    _host(q_scale, torch.float32, "q_scale", 1)
    _host(w, torch.float32, "w", 2)
    _host(q_pos, torch.int32, "q_pos", 1)
    _host(k8, torch.uint8, "k8", 2)
    _host(k_scale, torch.float32, "k_scale", 1)
    _host(q, torch.bfloat16, "q", 3)
    _host(kv, torch.bfloat16, "kv", 2)
    _host(out, torch.bfloat16, "out", 3)
    _host(lse, torch.float32, "lse", 2)
    T, H_I, d_I = q8.shape
    S = k8.shape[0]
    H = q.shape[1]
    need = dsa_prefill_host_workspace_size(T, S, H_I, d_I, H, k, chunk_rows)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=torch.cuda.current_device())
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().dsa_prefill_host(_ptr(q8), _ptr(q_scale), _ptr(w), _ptr(q_pos), _ptr(k8), _ptr(k_scale),
                                           _ptr(q), _ptr(kv), T, S, H_I, d_I, H, k, float(sm_scale), _ptr(out),
                                           _ptr(lse), chunk_rows, _ptr(workspace), ws_bytes, _stream(stream)))
    return out, lse


def dsa_prefill_host_trace(max_chunks: int):
    """Start (max_chunks > 0) or end (0) the per-chunk timeline record of dsa_prefill_host calls."""
    _check(load_library().dsa_prefill_host_trace(int(max_chunks)))


def dsa_prefill_host_trace_read(max_chunks: int):
    """The recorded timeline: (ms [n, 6] float32 from the first recorded call's start to each chunk's
    input-copy begin/end, stages begin/end, output-copy begin/end; call [n]; rows [n])."""
    ms = np.full((max_chunks, 6), np.nan, dtype=np.float32)
    call = np.zeros(max_chunks, dtype=np.int32)
    rows = np.zeros(max_chunks, dtype=np.int32)
    n = ctypes.c_int(0)
    _check(load_library().dsa_prefill_host_trace_read(ms.ctypes.data, call.ctypes.data, rows.ctypes.data,
                                                       int(max_chunks), ctypes.byref(n)))
    return ms[:n.value], call[:n.value], rows[:n.value]


def dsa_selftest_wait_timeout(limit_us: int, stream=None):
    """Run one bounded pipeline wait that nothing completes; it sets DSA_DEV_TIMEOUT after limit_us."""
    _check(load_library().dsa_selftest_wait_timeout(int(limit_us), _stream(stream)))


def dsa_get_device_status(stream=None) -> int:
    """Read and clear the device status word (DSA_DEV_* bits)."""
    v = ctypes.c_uint32(0)
    _check(load_library().dsa_get_device_status(_stream(stream), ctypes.byref(v)))
    return int(v.value)
