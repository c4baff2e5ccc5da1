"""GPU tests of dsa_prefill_host: the prefill path on host buffers, in chunks of
query rows whose copies overlap the kernels of neighbouring chunks.  Each case
checks the host-path outputs byte for byte against the three device entry
points run on the same inputs (the rows' work is the same, only the copies and
the chunking differ), with ragged last chunks, rows that start mid-sequence and
a single row."""
import numpy as np
import pytest
import torch

import dsa_workloads as W
from tests.gpu_util import lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _device_path(dsa, x, rows, cfg):
    """Indexer -> top-k -> sparse MLA on the device for query rows `rows`."""
    q_pos = x["q_pos"][rows].contiguous()
    T, S = q_pos.numel(), x["k8"].shape[0]
    logits = torch.full((T, S), float("nan"), device=DEV)
    dsa.dsa_indexer_logits(x["q8"][rows].contiguous(), x["qs"][rows].contiguous(), x["w"][rows].contiguous(),
                           x["k8"], x["ks"], q_pos, logits)
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device=DEV)
    dsa.dsa_topk(logits, q_pos + 1, cfg.k, idx)
    out = torch.empty((T, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((T, cfg.H), dtype=torch.float32, device=DEV)
    dsa.dsa_sparse_mla_prefill(x["q"][rows].contiguous(), x["kv"], idx, cfg.sm_scale, out, lse)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def _host_path(dsa, x, rows, cfg, chunk_rows):
    h = {n: x[n][rows].contiguous().cpu().pin_memory() for n in ("q8", "qs", "w", "q_pos", "q")}
    hk = {n: x[n].cpu().pin_memory() for n in ("k8", "ks", "kv")}
    T = h["q_pos"].numel()
    out = torch.full((T, cfg.H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
    lse = torch.full((T, cfg.H), float("nan"), dtype=torch.float32).pin_memory()
    dsa.dsa_prefill_host(h["q8"], h["qs"], h["w"], h["q_pos"], hk["k8"], hk["ks"], h["q"], hk["kv"], cfg.sm_scale,
                         cfg.k, out, lse, chunk_rows=chunk_rows)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("name,rows,chunk_rows", [
    ("tiny", slice(None), 100),          # 256 rows: chunks of 100, 100, 56
    ("tiny", slice(200, 201), 64),       # one row mid-sequence
    ("prefill_4k", slice(None), 1000),   # 4096 rows: four chunks of 1000 and one of 96
    ("prefill_4k", slice(2048, 4096), 4096),  # the second half in one chunk
])
def test_prefill_host_matches_device_path(name, rows, chunk_rows):
    dsa = lib()
    cfg = W.CONFIGS[name]
    x = W.prefill_inputs(cfg, DEV)
    o_ref, l_ref = _device_path(dsa, x, rows, cfg)
    o, l = _host_path(dsa, x, rows, cfg, chunk_rows)
    assert dsa.dsa_get_device_status() == 0
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(l, l_ref)


def test_prefill_host_two_calls_back_to_back():
    """Two calls enqueued without a host sync in between share the copy streams and
    buffer slots; the second must not overwrite what the first still uses."""
    dsa = lib()
    cfg = W.CONFIGS["tiny"]
    x = W.prefill_inputs(cfg, DEV)
    o_ref, l_ref = _device_path(dsa, x, slice(None), cfg)
    h = {n: x[n].cpu().pin_memory() for n in ("q8", "qs", "w", "q_pos", "q", "k8", "ks", "kv")}
    outs = []
    for _ in range(2):
        out = torch.full((cfg.L, cfg.H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
        lse = torch.full((cfg.L, cfg.H), float("nan"), dtype=torch.float32).pin_memory()
        dsa.dsa_prefill_host(h["q8"], h["qs"], h["w"], h["q_pos"], h["k8"], h["ks"], h["q"], h["kv"], cfg.sm_scale,
                             cfg.k, out, lse, chunk_rows=64)
        outs.append((out, lse))
    torch.cuda.synchronize()
    for out, lse in outs:
        assert torch.equal(out.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, l_ref)


def test_prefill_host_timeline():
    """The per-chunk timeline of two calls: one entry per chunk in enqueue order, rows that
    add up to the calls' rows, each chunk's input copies before its stages before its
    output copies, the stages of successive chunks in stream order, and outputs unchanged
    by the recording; a record of fewer chunks keeps the first ones."""
    dsa = lib()
    cfg = W.CONFIGS["tiny"]
    x = W.prefill_inputs(cfg, DEV)
    o_ref, l_ref = _device_path(dsa, x, slice(None), cfg)
    dsa.dsa_prefill_host_trace(64)
    try:
        outs = [_host_path(dsa, x, slice(None), cfg, 64) for _ in range(2)]
        t, call, rows = dsa.dsa_prefill_host_trace_read(64)
    finally:
        dsa.dsa_prefill_host_trace(0)
    for o, l in outs:
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)) and torch.equal(l, l_ref)
    # 256 rows in chunks of at most 64 (16, 32, 64, 64, 64, 16), processed last rows first
    per_call = [16, 64, 64, 64, 32, 16]
    assert call.tolist() == [0] * 6 + [1] * 6 and rows.tolist() == per_call * 2
    assert np.all(np.isfinite(t)) and np.all(t >= 0)
    assert np.all(np.diff(t, axis=1) >= 0)               # in begin <= in end <= stages ... <= out end
    assert np.all(t[1:, 2] >= t[:-1, 3])                 # stages of successive chunks in order
    assert t[6, 0] >= t[5, 5]                            # the second call starts after the first ends
    dsa.dsa_prefill_host_trace(3)
    try:
        _host_path(dsa, x, slice(None), cfg, 64)
        t, call, rows = dsa.dsa_prefill_host_trace_read(64)
    finally:
        dsa.dsa_prefill_host_trace(0)
    assert rows.tolist() == per_call[:3] and call.tolist() == [0, 0, 0]
