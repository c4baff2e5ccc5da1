"""fp64 CPU oracle for the DSA hot path: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline
leg and ``--impl reference``) may import this package.  The product library in
``sparse_attention_02_gb300`` never does, and the two share no code.

The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64, OpenMP over rows); this
module builds it with gcc and wraps each function with numpy arguments.  See the
C file's header for the passages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdsa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libdsa_oracle.so`` (portable C, no ISA flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.dsa_oracle_e4m3.restype = f64
        lib.dsa_oracle_e4m3.argtypes = [ctypes.c_uint8]
        lib.dsa_oracle_bf16.restype = f64
        lib.dsa_oracle_bf16.argtypes = [ctypes.c_uint16]
        lib.dsa_oracle_num_threads.restype = i32
        lib.dsa_oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.dsa_oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.dsa_oracle_quantize_fp8.argtypes = [P, i64, i64, i32, P, P]
        lib.dsa_oracle_indexer.argtypes = [P, P, P, P, i32, i32, i32, P, P, i32, P, i64]
        lib.dsa_oracle_indexer_paged.argtypes = [P, P, P, P, i32, i32, i32, P, P, i32, i32, P, i32, P, i64]
        lib.dsa_oracle_topk.argtypes = [P, i64, i32, P, i32, P]
        lib.dsa_oracle_sparse_mla.argtypes = [P, P, i32, P, i32, i32, i32, i32, i32, f64, P, P]
        lib.dsa_oracle_sparse_mla_paged.argtypes = [P, P, i32, i32, P, i32, P, P, i32, i32, i32, i32, i32, f64, P, P]
        lib.dsa_oracle_attn_target.argtypes = [P, P, i32, P, i32, i32, i32, f64, P, i64]
        lib.dsa_oracle_indexer_kl.argtypes = [P, P, P, i32, i32, i32, P, i32, P, i64, P, P, P, P]
        _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_L().dsa_oracle_num_threads())


def e4m3(code: int) -> float:
    return float(_L().dsa_oracle_e4m3(int(code) & 0xFF))


def bf16(bits: int) -> float:
    return float(_L().dsa_oracle_bf16(int(bits) & 0xFFFF))


def e4m3_encode(v: float) -> int:
    """E4M3 code of one fp32 value (nearest, ties to even, saturating at +-448)."""
    return int(_L().dsa_oracle_e4m3_encode(float(v)))


def quantize_fp8(x, mode: int = 0):
    """Per-row FP8 quantisation of fp32 ``x`` [rows, cols] (leading dims flattened into rows).

    mode 0: scale = fp32(amax / 448); mode 1: the smallest power of two not below it
    (1 for an all-zero row).  Returns (codes uint8 shaped like x, scale float32 [rows]).
    """
    x = np.asarray(x, dtype=np.float32)
    shape = x.shape
    rows = shape[0]
    cols = int(np.prod(shape[1:])) if x.ndim > 1 else 1
    xf = _c(x.reshape(rows, cols), np.float32)
    codes = np.empty((rows, cols), dtype=np.uint8)
    scale = np.empty(rows, dtype=np.float32)
    _L().dsa_oracle_quantize_fp8(_p(xf), rows, cols, int(mode), _p(codes), _p(scale))
    return codes.reshape(shape), scale


def indexer(q8, q_scale, w, q_pos, k8, k_scale, ld: int | None = None, fill=np.nan) -> np.ndarray:
    """Index scores for contiguous keys.

    q8: uint8 [n, HI, dI] E4M3 codes; q_scale: [n]; w: [n, HI]; q_pos: int [n];
    k8: uint8 [S, dI]; k_scale: [S].  Returns float64 [n, ld] with I[r, s] for
    s <= q_pos[r] and ``fill`` elsewhere.
    """
    q8 = _c(q8, np.uint8)
    n, HI, dI = q8.shape
    k8 = _c(k8, np.uint8)
    S = k8.shape[0]
    ld = S if ld is None else ld
    out = np.full((n, ld), fill, dtype=np.float64)
    qs, ww, qp, ks = _c(q_scale, np.float32), _c(w, np.float32), _c(q_pos, np.int32), _c(k_scale, np.float32)
    _L().dsa_oracle_indexer(_p(q8), _p(qs), _p(ww), _p(qp), n, HI, dI, _p(k8), _p(ks), S, _p(out), ld)
    return out


def indexer_paged(q8, q_scale, w, ctx_len, k8_pool, k_scale_pool, block_table, ld: int, fill=np.nan) -> np.ndarray:
    """Index scores over a paged key pool (k8_pool [P, page, dI], k_scale_pool [P, page])."""
    q8 = _c(q8, np.uint8)
    n, HI, dI = q8.shape
    k8_pool = _c(k8_pool, np.uint8)
    num_pages, page_size, _ = k8_pool.shape
    bt = _c(block_table, np.int32)
    out = np.full((n, ld), fill, dtype=np.float64)
    qs, ww, cl, ks = _c(q_scale, np.float32), _c(w, np.float32), _c(ctx_len, np.int32), _c(k_scale_pool, np.float32)
    _L().dsa_oracle_indexer_paged(_p(q8), _p(qs), _p(ww), _p(cl), n, HI, dI, _p(k8_pool), _p(ks),
                                  num_pages, page_size, _p(bt), bt.shape[1], _p(out), ld)
    return out


def topk(vals, valid_len, k: int) -> np.ndarray:
    """Top-k indices per row of ``vals`` [rows, ld] (any real dtype, compared exactly in fp64)."""
    v = _c(vals, np.float64)
    rows, ld = v.shape
    vl = _c(valid_len, np.int32)
    idx = np.empty((rows, k), dtype=np.int32)
    _L().dsa_oracle_topk(_p(v), ld, rows, _p(vl), k, _p(idx))
    return idx


def sparse_mla(q_bits, kv_bits, idx, sm_scale: float, Dv: int = 512):
    """Sparse MQA-mode MLA.  q_bits uint16 [n, H, D], kv_bits uint16 [S, D], idx int [n, k]."""
    q = _c(q_bits, np.uint16)
    n, H, D = q.shape
    kv = _c(kv_bits, np.uint16)
    S = kv.shape[0]
    ix = _c(idx, np.int32)
    k = ix.shape[1]
    out = np.empty((n, H, Dv), dtype=np.float64)
    lse = np.empty((n, H), dtype=np.float64)
    _L().dsa_oracle_sparse_mla(_p(q), _p(kv), S, _p(ix), n, H, D, Dv, k, float(sm_scale), _p(out), _p(lse))
    return out, lse


def sparse_mla_paged(q_bits, kv_pool_bits, block_table, ctx_len, idx, sm_scale: float, Dv: int = 512):
    """Paged sparse MLA for decode.  kv_pool_bits uint16 [P, page, D]."""
    q = _c(q_bits, np.uint16)
    n, H, D = q.shape
    pool = _c(kv_pool_bits, np.uint16)
    num_pages, page_size, _ = pool.shape
    bt = _c(block_table, np.int32)
    cl = _c(ctx_len, np.int32)
    ix = _c(idx, np.int32)
    k = ix.shape[1]
    out = np.empty((n, H, Dv), dtype=np.float64)
    lse = np.empty((n, H), dtype=np.float64)
    _L().dsa_oracle_sparse_mla_paged(_p(q), _p(pool), num_pages, page_size, _p(bt), bt.shape[1], _p(cl),
                                     _p(ix), n, H, D, Dv, k, float(sm_scale), _p(out), _p(lse))
    return out, lse


def attn_target(q_bits, kv_bits, q_pos, sm_scale: float, ld: int | None = None, fill=np.nan) -> np.ndarray:
    """Warm-up target: the main attention's dense causal distribution over keys s <= q_pos[r],
    averaged over heads.  q_bits uint16 [n, H, D], kv_bits uint16 [S, D].  Returns float64 [n, ld]."""
    q = _c(q_bits, np.uint16)
    n, H, D = q.shape
    kv = _c(kv_bits, np.uint16)
    S = kv.shape[0]
    ld = S if ld is None else ld
    out = np.full((n, ld), fill, dtype=np.float64)
    qp = _c(q_pos, np.int32)
    _L().dsa_oracle_attn_target(_p(q), _p(kv), S, _p(qp), n, H, D, float(sm_scale), _p(out), ld)
    return out


def indexer_kl(q, w, q_pos, k, p):
    """Warm-up loss and gradients from dequantised fp64 q [n, HI, dI], k [S, dI], w [n, HI]
    and the target p [n, >= S].  Returns (loss [n], dw [n, HI], dq [n, HI, dI], dk [S, dI]).
    The gradients' ReLU decisions are taken on the fp64 dot products (ReLU'(0) = 0)."""
    q = _c(q, np.float64)
    n, HI, dI = q.shape
    k = _c(k, np.float64)
    S = k.shape[0]
    w = _c(w, np.float64)
    pp = _c(p, np.float64)
    qp = _c(q_pos, np.int32)
    loss = np.empty(n, dtype=np.float64)
    dw = np.empty((n, HI), dtype=np.float64)
    dq = np.empty((n, HI, dI), dtype=np.float64)
    dk = np.empty((S, dI), dtype=np.float64)
    _L().dsa_oracle_indexer_kl(_p(q), _p(w), _p(qp), n, HI, dI, _p(k), S, _p(pp), pp.shape[1], _p(loss), _p(dw),
                               _p(dq), _p(dk))
    return loss, dw, dq, dk
