"""C ABI checks that need no GPU: every declared symbol is exported, and bad
arguments are rejected on the host (before any CUDA call) with a message."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_02_gb300 import build

    path = build.build()
    import sparse_attention_02_gb300 as dsa

    return dsa.load_library(path)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"dsa_indexer_logits", "dsa_topk", "dsa_sparse_mla_prefill", "dsa_sparse_mla_decode_paged"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dsa.h but not exported"


def test_version_and_workspace_query(lib):
    assert lib.dsa_version() >= 100
    # at most two thirds as many rows as SM pairs: rows are split, 2 slots per
    # cluster of H x (512 + 1) fp32
    n = lib.dsa_sparse_mla_decode_workspace_size(32, 128, 2048)
    assert n > 0 and n % (2 * 128 * 513 * 4) == 0
    assert lib.dsa_sparse_mla_decode_workspace_size(32, 16, 2048) == n // 8
    assert lib.dsa_sparse_mla_decode_workspace_size(1024, 128, 2048) == 0  # whole rows: none
    assert lib.dsa_sparse_mla_decode_workspace_size(1, 128, 64) == 0       # one block: nothing to split
    assert lib.dsa_sparse_mla_decode_workspace_size(64, 129, 2048) == 0  # unsupported H: 0


def _err(lib):
    return lib.dsa_last_error().decode()


def test_host_validation_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: every call below fails its host checks first
    # top-k: k out of range, null pointers, T < 0; T == 0 is a no-op
    assert lib.dsa_topk(fake, 16, 4, fake, 0, fake, None) == 2
    assert "k must be" in _err(lib)
    assert lib.dsa_topk(None, 16, 4, fake, 8, fake, None) == 1
    assert lib.dsa_topk(fake, 16, -1, fake, 8, fake, None) == 1
    assert lib.dsa_topk(fake, 16, 0, fake, 8, fake, None) == 0
    assert lib.dsa_topk(fake, 1 << 29, 4, fake, 8, fake, None) == 2
    # quantiser: bad mode, bad sizes, null pointers; rows == 0 is a no-op
    i64 = ctypes.c_int64
    assert lib.dsa_quantize_fp8(fake, i64(4), i64(128), 2, fake, fake, None) == 1
    assert "scale_mode" in _err(lib)
    assert lib.dsa_quantize_fp8(fake, i64(-1), i64(128), 0, fake, fake, None) == 1
    assert lib.dsa_quantize_fp8(fake, i64(4), i64(0), 0, fake, fake, None) == 1
    assert lib.dsa_quantize_fp8(None, i64(4), i64(128), 1, fake, fake, None) == 1
    assert lib.dsa_quantize_fp8(fake, i64(0), i64(128), 0, None, None, None) == 0
    assert lib.dsa_quantize_fp8(fake, i64(1 << 40), i64(1 << 20), 0, fake, fake, None) == 2
    # indexer: misaligned q8, bad page size, missing S
    assert lib.dsa_indexer_logits(P(4097), fake, fake, 4, 64, 128, fake, fake, 16, None, 0, 0, 0, fake, fake, 16,
                                  None) == 3
    assert lib.dsa_indexer_logits(fake, fake, fake, 4, 64, 128, fake, fake, 16, fake, 4, 4, 48, fake, fake, 16,
                                  None) == 2
    assert lib.dsa_indexer_logits(fake, fake, fake, 4, 64, 128, fake, fake, 0, None, 0, 0, 0, fake, fake, 16,
                                  None) == 1
    assert lib.dsa_indexer_logits(fake, fake, fake, 0, 64, 128, fake, fake, 16, None, 0, 0, 0, fake, fake, 16,
                                  None) == 0
    # sparse MLA: heads out of range, non-positive scale, misaligned output
    f = ctypes.c_float
    assert lib.dsa_sparse_mla_prefill(fake, fake, 8, fake, 4, 129, 64, f(0.04), fake, fake, None) == 2
    assert lib.dsa_sparse_mla_prefill(fake, fake, 8, fake, 4, 128, 64, f(0.0), fake, fake, None) == 1
    assert lib.dsa_sparse_mla_prefill(fake, fake, 8, fake, 4, 128, 64, f(0.04), P(4098), fake, None) == 3
    assert lib.dsa_sparse_mla_prefill(fake, fake, 8, fake, 0, 128, 64, f(0.04), fake, fake, None) == 0
    # paged decode: workspace check and misaligned pool
    assert lib.dsa_sparse_mla_decode_paged(fake, P(4100), 4, 64, fake, 2, fake, fake, 2, 128, 64, f(0.04), fake,
                                           fake, None, 0, None) == 3
    assert lib.dsa_sparse_mla_decode_paged(fake, fake, 0, 64, fake, 2, fake, fake, 2, 128, 64, f(0.04), fake,
                                           fake, None, 0, None) == 1


def test_host_prefill_validation(lib):
    """dsa_prefill_host's own checks, all taken on the host before any CUDA call (no call
    here passes them all, so nothing reaches the device)."""
    import numpy as np

    P = ctypes.c_void_p
    fake = P(4096)
    T, S, HI, dI, H, k, C = 4, 8, 64, 128, 128, 64, 4
    need = lib.dsa_prefill_host_workspace_size(T, S, HI, dI, H, k, C)
    assert need > 0 and lib.dsa_prefill_host_workspace_size(T, S, HI, dI, 129, k, C) == 0
    q_pos = np.arange(T, dtype=np.int32)
    qp = q_pos.ctypes.data_as(P)

    def call(t=T, h=H, chunk=C, ws=P(1 << 20), ws_bytes=need, pos=qp):
        return lib.dsa_prefill_host(fake, fake, fake, pos, fake, fake, fake, fake, t, S, HI, dI, h, k,
                                    ctypes.c_float(0.04), fake, fake, chunk, ws, ws_bytes, None)

    assert call(t=-1) == 1
    assert call(chunk=0) == 1
    assert call(t=0) == 0                       # no rows: nothing to do
    assert call(ws=None) == 1                   # null workspace
    assert call(h=129) == 1                     # heads out of range
    assert call(ws=P((1 << 20) + 16)) == 3      # workspace not 256-byte aligned
    assert call(ws_bytes=need - 1) == 4         # workspace short by one byte
    assert "workspace" in _err(lib)
    bad = np.array([0, 1, S, 3], dtype=np.int32)
    assert call(pos=bad.ctypes.data_as(P)) == 1  # a query position past the keys
    assert "q_pos[2]" in _err(lib)


def test_host_prefill_timeline_validation(lib):
    """The timeline calls' argument checks, taken before any CUDA call."""
    import numpy as np

    P = ctypes.c_void_p
    assert lib.dsa_prefill_host_trace(-1) == 1
    assert lib.dsa_prefill_host_trace((1 << 20) + 1) == 1
    n = ctypes.c_int(0)
    buf = np.zeros(6, dtype=np.float32)
    ib = np.zeros(1, dtype=np.int32)
    assert lib.dsa_prefill_host_trace_read(None, P(ib.ctypes.data), P(ib.ctypes.data), 1, ctypes.byref(n)) == 1
    assert lib.dsa_prefill_host_trace_read(P(buf.ctypes.data), P(ib.ctypes.data), P(ib.ctypes.data), -1,
                                           ctypes.byref(n)) == 1
    assert lib.dsa_prefill_host_trace_read(P(buf.ctypes.data), P(ib.ctypes.data), P(ib.ctypes.data), 1, None) == 1


def test_binding_raises_without_the_library(tmp_path):
    import sparse_attention_02_gb300 as dsa

    with pytest.raises(RuntimeError, match="missing"):
        dsa.load_library(str(tmp_path / "nope.so"))


def test_every_declaration_is_documented_and_cites_its_page():
    """Each function in dsa.h has a comment right above it (or above its macro); the
    entry points of the method's steps cite the page that defines them."""
    text = open(HEADER).read()
    pages = ("AMD Instinct MI355X GPUs Power DeepSeek-V3.2-Exp", "DeepSeek-V3.2-Exp: Boosting Long-Context")
    steps = {"dsa_indexer_logits", "dsa_quantize_fp8", "dsa_topk", "dsa_sparse_mla_prefill",
             "dsa_sparse_mla_decode_paged"}
    for name in declared_functions():
        m = re.search(r"^[A-Za-z_][\w\s\*]*\b" + name + r"\s*\(", text, flags=re.M)
        assert m, f"{name}: declaration not found"
        before = text[: m.start()].rstrip()
        while before.endswith(")") or re.search(r"#define [^\n]*$", before):  # macros placed between
            before = before[: before.rfind("\n")].rstrip()
        assert before.endswith("*/"), f"{name} has no comment above its declaration"
        comment = before[before.rfind("/*"):]
        if name in steps:
            flat = " ".join(comment.replace("*", " ").split())
            assert any(" ".join(pg.split()) in flat for pg in pages), f"{name}: no page cited"


def test_fused_indexer_topk_validation(lib):
    """dsa_indexer_topk's host checks and its workspace query (nothing reaches the device)."""
    P = ctypes.c_void_p
    fake = P(4096)
    T, S, k = 8, 1000, 64
    need = lib.dsa_indexer_topk_workspace_size(T, S, 64, 128, k)
    # sampled keys, per-row positions and thresholds, T x max(4096, 4k) candidates of 8 bytes,
    # T x S fp32 scores for rows redone from full scores
    assert need >= T * 4096 * 8 + T * S * 4 + T * min(S, 2048) * 4
    assert lib.dsa_indexer_topk_workspace_size(T, S, 64, 128, 4096) > need  # the list cap grows with k past 2048
    assert lib.dsa_indexer_topk_workspace_size(T, S, 4, 32, k) == 0        # unsupported head shape
    assert lib.dsa_indexer_topk_workspace_size(T, 262145, 64, 128, k) == 0  # past the key limit
    assert lib.dsa_indexer_topk_workspace_size(T, S, 64, 128, 4097) == 0

    def call(t=T, hi=64, di=128, s=S, kk=k, q8=fake, ws=P(1 << 20), ws_bytes=need):
        return lib.dsa_indexer_topk(q8, fake, fake, t, hi, di, fake, fake, s, fake, kk, fake, ws, ws_bytes, None)

    assert call(t=-1) == 1
    assert call(t=0) == 0
    assert call(hi=4, di=32) == 2
    assert call(s=0) == 2 and call(s=262145) == 2
    assert call(kk=0) == 2
    assert call(q8=P(4097)) == 3
    assert call(ws=P((1 << 20) + 64)) == 3
    assert call(ws_bytes=need - 1) == 4
    assert "workspace" in _err(lib)


def test_warmup_workspace_size(lib):
    """The warm-up's workspace: p and I/g (T x S fp32 each), the FP8 codes as bf16 with one
    bound and one w q_scale per (t, j) row and one bound per key: no per-(t, j, s) buffer."""
    lib.dsa_indexer_warmup_workspace_size.restype = ctypes.c_size_t
    ws = lib.dsa_indexer_warmup_workspace_size
    T, S, HI = 4096, 4096, 64
    need = ws(T, S, HI, 128)
    floor = 8 * T * S + 256 * T * HI + 8 * T * HI + 256 * S + 4 * S
    assert floor <= need <= floor + 6 * 256                        # each region rounded up to 256 bytes
    assert need < 4 * HI * T * S // 8                              # far below a coefficient buffer
    assert ws(T, 2 * S, HI, 128) > need and ws(T, S, 32, 128) < need
    assert ws(T, S, 48, 128) == 0 and ws(T, S, 64, 64) == 0 and ws(-1, S, HI, 128) == 0 and ws(T, 0, HI, 128) == 0
