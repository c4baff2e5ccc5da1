"""GPU parity at the workloads' full sizes, in the launch configuration bench.py
times: exact oracle comparison on sampled rows (rows are independent, so any
row can be computed by the oracle alone), plus properties checked on every row.

* prefill L=32768: indexer rows, top-k on every row (validity, ordering, and the
  selection threshold with its tie rule) plus exact oracle top-k on sampled
  rows from the GPU's own logits, sparse MLA rows;
* paged decode, 64 sequences with contexts in [8192, 65536];
* chunked prefill L=131072 in chunks of 4096 over the full prefix, and the
  invariant that chunked and unchunked prefill agree bit for bit at L=8192.
"""
import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from tests.gpu_util import bits16, check_attention, check_logits, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def check_topk_all_rows(logits: torch.Tensor, valid: torch.Tensor, idx: torch.Tensor, k: int, chunk: int = 2048):
    """Every row: k ascending in-range indices (or 0..n-1 then -1), and no
    unselected candidate outranks a selected one under (score desc, index asc)."""
    T, ld = logits.shape
    cols = torch.arange(ld, device=logits.device)
    for r0 in range(0, T, chunk):
        r1 = min(T, r0 + chunk)
        lg = logits[r0:r1]
        n = valid[r0:r1].long()
        ix = idx[r0:r1].long()
        m = torch.minimum(n, torch.tensor(k, device=n.device))
        pos = torch.arange(k, device=n.device)[None, :]
        used = pos < m[:, None]
        assert torch.all(ix[~used] == -1), "padding must be -1"
        small = n <= k
        if small.any():
            assert torch.all((ix[small] == torch.where(used[small], pos.expand_as(ix)[small], -1))), "n <= k rows"
        big = ~small
        if not big.any():
            continue
        lg, ix, n = lg[big], ix[big], n[big]
        assert torch.all(ix[:, 1:] > ix[:, :-1]), "indices must be strictly ascending"
        assert torch.all(ix >= 0) and torch.all(ix < n[:, None]), "indices in range"
        sel_vals = lg.gather(1, ix)
        thr = sel_vals.min(1).values
        in_range = cols[None, :] < n[:, None]
        selected = torch.zeros_like(lg, dtype=torch.bool).scatter_(1, ix, True)
        rest = lg.masked_fill(selected | ~in_range, float("-inf"))
        rest_max = rest.max(1).values
        assert torch.all(rest_max <= thr), "an unselected score beats a selected one"
        # ties at the threshold: every selected index with that score precedes every unselected one
        tie = rest_max == thr
        if tie.any():
            lt, it_, ct = lg[tie], selected[tie], thr[tie]
            eq = lt == ct[:, None]
            big_idx = torch.where(eq & it_, cols[None, :], -1).max(1).values
            small_idx = torch.where(eq & ~it_ & (cols[None, :] < n[tie][:, None]), cols[None, :], ld).min(1).values
            assert torch.all(big_idx < small_idx), "tie rule (smaller index first) violated"


def test_prefill_32k_full_size():
    cfg = W.CONFIGS["prefill_32k"]
    dsa = lib()
    L = cfg.L
    x = W.prefill_inputs(cfg, DEV)
    logits = torch.empty((L, L), dtype=torch.float32, device=DEV)
    idx = torch.empty((L, cfg.k), dtype=torch.int32, device=DEV)
    out = torch.empty((L, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((L, cfg.H), dtype=torch.float32, device=DEV)
    valid = x["q_pos"] + 1
    dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], logits)
    dsa.dsa_topk(logits, valid, cfg.k, idx)
    dsa.dsa_sparse_mla_prefill(x["q"], x["kv"], idx, cfg.sm_scale, out, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    check_topk_all_rows(logits, valid, idx, cfg.k)
    rows = np.array([0, 1, 2046, 2047, 2048, 12345, 32766, 32767])
    r = torch.as_tensor(rows, device=DEV)
    ref = oracle.indexer(x["q8"][r].cpu().numpy(), x["qs"][r].cpu().numpy(), x["w"][r].cpu().numpy(), rows,
                         x["k8"].cpu().numpy(), x["ks"].cpu().numpy(), ld=L)
    got = logits[r].cpu().double().numpy()
    check_logits(got, ref, rows)
    ref_idx = oracle.topk(np.nan_to_num(got, nan=0.0), rows + 1, cfg.k)
    assert np.array_equal(idx[r].cpu().numpy(), ref_idx)
    o_ref, l_ref = oracle.sparse_mla(bits16(x["q"][r]), bits16(x["kv"]), ref_idx, cfg.sm_scale)
    check_attention(out[r].cpu().double().numpy(), lse[r].cpu().double().numpy(), o_ref, l_ref)


def test_decode_paged_full_size():
    cfg = W.CONFIGS["decode_paged"]
    dsa = lib()
    d = W.decode_inputs(cfg, DEV)
    B = d["ctx"].shape[0]
    ctx = d["ctx"].cpu().numpy()
    ld = int(ctx.max())
    logits = torch.empty((B, ld), dtype=torch.float32, device=DEV)
    idx = torch.empty((B, cfg.k), dtype=torch.int32, device=DEV)
    out = torch.empty((B, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, cfg.H), dtype=torch.float32, device=DEV)
    dsa.dsa_indexer_logits(d["q8"], d["qs"], d["w"], d["k8_pool"], d["ks_pool"], d["q_pos"], logits,
                           block_table=d["block_table"])
    dsa.dsa_topk(logits, d["ctx"], cfg.k, idx)
    dsa.dsa_sparse_mla_decode_paged(d["q"], d["kv_pool"], d["block_table"], d["ctx"], idx, cfg.sm_scale, out, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    bt = d["block_table"].cpu().numpy()
    rows = np.unique(np.array([0, int(np.argmax(ctx)), int(np.argmin(ctx)), B - 1]))
    ref = oracle.indexer_paged(d["q8"][rows].cpu().numpy(), d["qs"][rows].cpu().numpy(), d["w"][rows].cpu().numpy(),
                               ctx[rows], d["k8_pool"].cpu().numpy(), d["ks_pool"].cpu().numpy(), bt[rows], ld)
    check_logits(logits.cpu().double().numpy()[rows], ref, ctx[rows] - 1)
    # top-k and attention exactly on every sequence
    lg = logits.cpu().double().numpy()
    for b in range(B):
        lg[b, ctx[b]:] = 0.0
    ref_idx = oracle.topk(lg, ctx, cfg.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    o_ref, l_ref = oracle.sparse_mla_paged(bits16(d["q"]), bits16(d["kv_pool"]), bt, ctx, ref_idx, cfg.sm_scale)
    check_attention(out.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, l_ref)


def run_chunked(dsa, x, cfg, L, chunk):
    """Chunked prefill: rows [c, c+chunk) scored and attended over the prefix [0, c+chunk)."""
    idx = torch.empty((L, cfg.k), dtype=torch.int32, device=DEV)
    out = torch.empty((L, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((L, cfg.H), dtype=torch.float32, device=DEV)
    logits = torch.empty((chunk, L), dtype=torch.float32, device=DEV)
    last_logits = None
    for c0 in range(0, L, chunk):
        c1 = min(L, c0 + chunk)
        S = c1
        lg = logits[: c1 - c0, :S] if S == L else torch.empty((c1 - c0, S), dtype=torch.float32, device=DEV)
        dsa.dsa_indexer_logits(x["q8"][c0:c1], x["qs"][c0:c1], x["w"][c0:c1], x["k8"][:S], x["ks"][:S],
                               x["q_pos"][c0:c1], lg)
        dsa.dsa_topk(lg, x["q_pos"][c0:c1] + 1, cfg.k, idx[c0:c1])
        dsa.dsa_sparse_mla_prefill(x["q"][c0:c1], x["kv"][:S], idx[c0:c1], cfg.sm_scale, out[c0:c1], lse[c0:c1])
        last_logits = lg
    return idx, out, lse, last_logits


def test_chunked_equals_unchunked_8k():
    cfg = W.CONFIGS["chunked_128k"]
    dsa = lib()
    L = 8192
    x = W.prefill_inputs(cfg, DEV, L=L)
    idx_c, out_c, lse_c, _ = run_chunked(dsa, x, cfg, L, 4096)
    logits = torch.empty((L, L), dtype=torch.float32, device=DEV)
    idx = torch.empty((L, cfg.k), dtype=torch.int32, device=DEV)
    out = torch.empty((L, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((L, cfg.H), dtype=torch.float32, device=DEV)
    dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], logits)
    dsa.dsa_topk(logits, x["q_pos"] + 1, cfg.k, idx)
    dsa.dsa_sparse_mla_prefill(x["q"], x["kv"], idx, cfg.sm_scale, out, lse)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_c)
    assert torch.equal(out.view(torch.int16), out_c.view(torch.int16))
    assert torch.equal(lse, lse_c)


def test_chunked_128k_full_size():
    cfg = W.CONFIGS["chunked_128k"]
    dsa = lib()
    L, chunk = cfg.L, cfg.chunk
    x = W.prefill_inputs(cfg, DEV)
    idx, out, lse, last_logits = run_chunked(dsa, x, cfg, L, chunk)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    rows = np.array([L - chunk, L - chunk + 777, L - 1])  # last chunk: full 131072-key prefix
    r = torch.as_tensor(rows, device=DEV)
    ref = oracle.indexer(x["q8"][r].cpu().numpy(), x["qs"][r].cpu().numpy(), x["w"][r].cpu().numpy(), rows,
                         x["k8"].cpu().numpy(), x["ks"].cpu().numpy(), ld=L)
    got = last_logits[r - (L - chunk)].cpu().double().numpy()
    check_logits(got, ref, rows)
    ref_idx = oracle.topk(np.nan_to_num(got, nan=0.0), rows + 1, cfg.k)
    assert np.array_equal(idx[r].cpu().numpy(), ref_idx)
    o_ref, l_ref = oracle.sparse_mla(bits16(x["q"][r]), bits16(x["kv"]), ref_idx, cfg.sm_scale)
    check_attention(out[r].cpu().double().numpy(), lse[r].cpu().double().numpy(), o_ref, l_ref)
