"""GPU parity for ragged batches through the paged entry points: a varlen batched
prefill (every token of several different-length sequences is a query row) and a
multi-token decode (the last few positions of each sequence), all rows sharing one
permuted page pool.  Each query row carries its own position, context length and
block-table row.  Checked against the oracle (indexer rows, top-k on every row
from the GPU's logits, attention rows) and against the contiguous entry point on
the same latent rows concatenated per sequence: bit-identical output when the
decode keeps whole rows (at least as many rows as SM pairs), equal up to fp32
summation order when it cuts fewer rows into pieces over the SMs."""
import dataclasses

import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from tests.gpu_util import bits16, check_attention, check_logits, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_paged(dsa, v, k, sm_scale):
    T = v["q8"].shape[0]
    ld = int(v["seq_lens"].max())
    logits = torch.full((T, ld), float("nan"), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    H = v["q"].shape[1]
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((T, H), dtype=torch.float32, device=DEV)
    dsa.dsa_indexer_logits(v["q8"], v["qs"], v["w"], v["k8_pool"], v["ks_pool"], v["q_pos"], logits,
                           block_table=v["block_table"])
    dsa.dsa_topk(logits, v["ctx"], k, idx)
    dsa.dsa_sparse_mla_decode_paged(v["q"], v["kv_pool"], v["block_table"], v["ctx"], idx, sm_scale, out, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    return logits, idx, out, lse


def check_against_oracle(v, logits, idx, out, lse, k, sm_scale, rows):
    ctx = v["ctx"].cpu().numpy()
    bt = v["block_table"].cpu().numpy()
    ld = logits.shape[1]
    ref = oracle.indexer_paged(v["q8"][rows].cpu().numpy(), v["qs"][rows].cpu().numpy(), v["w"][rows].cpu().numpy(),
                               ctx[rows], v["k8_pool"].cpu().numpy(), v["ks_pool"].cpu().numpy(), bt[rows], ld)
    check_logits(logits.cpu().double().numpy()[rows], ref, ctx[rows] - 1)
    lg = logits.cpu().double().numpy()
    for r in range(lg.shape[0]):
        lg[r, ctx[r]:] = 0.0
    ref_idx = oracle.topk(lg, ctx, k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    o_ref, l_ref = oracle.sparse_mla_paged(bits16(v["q"][rows]), bits16(v["kv_pool"]), bt[rows], ctx[rows],
                                           ref_idx[rows], sm_scale)
    check_attention(out[rows].cpu().double().numpy(), lse[rows].cpu().double().numpy(), o_ref, l_ref)


def check_contiguous_equivalence(dsa, v, idx, out, lse, sm_scale):
    """The same rows through the contiguous entry point: latent rows concatenated per
    sequence, selected positions offset by the sequence start."""
    starts = v["seq_starts"][v["seq"]].to(DEV).to(torch.int32)[:, None]
    gidx = torch.where(idx >= 0, idx + starts, idx)
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    S = v["kv_concat"].shape[0]
    dsa.dsa_sparse_mla_prefill(v["q"], v["kv_concat"], gidx, sm_scale, out2, lse2)
    torch.cuda.synchronize()
    assert S == int(v["seq_lens"].sum())
    T, H = lse.shape
    if dsa.dsa_sparse_mla_decode_workspace_size(T, H, idx.shape[1]) == 0:  # whole rows: same kernel path
        assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
        assert torch.equal(lse2, lse)
    else:  # rows merged from pieces: fp32 rounding, then one bf16 rounding of O
        assert (out2.float() - out.float()).abs().max().item() <= 2e-3
        assert (lse2 - lse).abs().max().item() <= 1e-4


def boundary_rows(v, extra=()):
    seq = v["seq"].numpy()
    first = np.flatnonzero(np.r_[True, seq[1:] != seq[:-1]])
    last = np.r_[first[1:] - 1, len(seq) - 1]
    return np.unique(np.r_[first, last, np.asarray(extra, dtype=np.int64)])


def test_varlen_batched_prefill():
    dsa = lib()
    cfg = dataclasses.replace(W.CONFIGS["decode_paged"], seed=7)
    k = 256
    v = W.varlen_inputs(cfg, DEV, [300, 1000, 77, 513, 64, 1250])
    logits, idx, out, lse = run_paged(dsa, v, k, cfg.sm_scale)
    rows = boundary_rows(v, extra=[255, 256, 257, 1299, 1600, 2500])
    check_against_oracle(v, logits, idx, out, lse, k, cfg.sm_scale, rows)
    check_contiguous_equivalence(dsa, v, idx, out, lse, cfg.sm_scale)


def test_multi_token_decode():
    dsa = lib()
    cfg = dataclasses.replace(W.CONFIGS["decode_paged"], seed=8)
    v = W.varlen_inputs(cfg, DEV, [3000, 5000, 4097, 8192, 2049], [3, 2, 4, 1, 2])
    logits, idx, out, lse = run_paged(dsa, v, cfg.k, cfg.sm_scale)
    rows = np.arange(v["q8"].shape[0])
    check_against_oracle(v, logits, idx, out, lse, cfg.k, cfg.sm_scale, rows)
    check_contiguous_equivalence(dsa, v, idx, out, lse, cfg.sm_scale)
