"""GPU tests of failure detection: data problems only the device can see never
fault, they skip the offending element and set a bit of the device status word,
and a pipeline wait that runs out sets DSA_DEV_TIMEOUT and returns.  Every case
checks the status bits and that the other results still match the oracle; no
case can fault or hang (out-of-range pages are zero-filled copies that are then
masked, and the timed-out wait is bounded)."""
import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
import sparse_attention_02_gb300 as dsa_mod
from tests.gpu_util import bits16, check_attention, check_logits, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_timed_out_wait_sets_status_and_context_stays_usable():
    dsa = lib()
    assert dsa.dsa_get_device_status() == 0
    dsa.dsa_selftest_wait_timeout(2000)  # 2 ms
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == dsa_mod.DSA_DEV_TIMEOUT
    assert dsa.dsa_get_device_status() == 0  # reading cleared it
    # the context still runs the hot path
    cfg = W.CONFIGS["tiny"]
    x = W.prefill_inputs(cfg, DEV)
    logits = torch.full((cfg.L, cfg.L), float("nan"), device=DEV)
    dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], logits)
    idx = torch.empty((cfg.L, cfg.k), dtype=torch.int32, device=DEV)
    dsa.dsa_topk(logits, x["q_pos"] + 1, cfg.k, idx)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    ref = oracle.topk(np.nan_to_num(logits.cpu().double().numpy(), nan=0.0), np.arange(1, cfg.L + 1), cfg.k)
    assert np.array_equal(idx.cpu().numpy(), ref)


@pytest.mark.parametrize("T", [8, 400])  # cluster kernel, row kernel
def test_topk_valid_length_past_ld_is_clamped_and_flagged(T):
    dsa = lib()
    ld, k = 5000, 2048
    g = torch.Generator(device=DEV).manual_seed(11)
    vals = torch.randn((T, ld), generator=g, device=DEV)
    n = torch.full((T,), ld, dtype=torch.int32, device=DEV)
    n_bad = n.clone()
    n_bad[T // 2] = ld + 7
    a = torch.empty((T, k), dtype=torch.int32, device=DEV)
    b = torch.empty_like(a)
    dsa.dsa_topk(vals, n, k, a)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    dsa.dsa_topk(vals, n_bad, k, b)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == dsa_mod.DSA_DEV_BAD_POSITION
    assert torch.equal(a, b)


def test_indexer_position_past_keys_is_clamped_and_flagged():
    dsa = lib()
    cfg = W.CONFIGS["tiny"]
    x = W.prefill_inputs(cfg, DEV)
    S = 200
    q_pos = x["q_pos"].clone()
    q_pos[250] = S + 30  # past the 200 keys given
    logits = torch.full((cfg.L, cfg.L), float("nan"), device=DEV)
    dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"][:S], x["ks"][:S], q_pos, logits)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == dsa_mod.DSA_DEV_BAD_POSITION
    rows = np.array([0, 100, 199, 250])
    h = {n: x[n].cpu().numpy() for n in ("q8", "qs", "w", "k8", "ks")}
    pos = np.minimum(rows, S - 1)  # the flagged row is scored as if at the last key
    ref = oracle.indexer(h["q8"][rows], h["qs"][rows], h["w"][rows], pos, h["k8"][:S], h["ks"][:S], ld=cfg.L)
    check_logits(logits.cpu().double().numpy()[rows], ref, pos)


def _bad_page_case():
    """Decode rows over a permuted page pool; one page of row 1 and one of row 5
    point outside the pool (past the end, and negative)."""
    cfg = W.CONFIGS["decode_paged"]
    ctx = [700, 3001, 64, 2100, 130, 5000]
    d = W.decode_inputs(cfg, DEV, ctx=ctx, seed=21)
    bt = d["block_table"].clone()
    bt[1, 3] = d["num_pages"] + 5
    bt[5, 40] = -3
    return cfg, d, bt, np.array(ctx, dtype=np.int32)


def test_paged_indexer_bad_page_is_skipped_and_flagged():
    dsa = lib()
    cfg, d, bt, ctx = _bad_page_case()
    B, ld = len(ctx), int(ctx.max())
    sentinel = -12345.0
    logits = torch.full((B, ld), sentinel, device=DEV)
    dsa.dsa_indexer_logits(d["q8"], d["qs"], d["w"], d["k8_pool"], d["ks_pool"], d["q_pos"], logits,
                           block_table=bt)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == dsa_mod.DSA_DEV_BAD_PAGE
    got = logits.cpu().double().numpy()
    ref = oracle.indexer_paged(d["q8"].cpu().numpy(), d["qs"].cpu().numpy(), d["w"].cpu().numpy(), ctx,
                               d["k8_pool"].cpu().numpy(), d["ks_pool"].cpu().numpy(), bt.cpu().numpy(), ld)
    ps = cfg.page_size
    for r in range(B):
        bad = np.zeros(ld, dtype=bool)
        for lp in range(bt.shape[1]):
            p = int(bt[r, lp])
            if p < 0 or p >= d["num_pages"]:
                bad[lp * ps:(lp + 1) * ps] = True
        n = int(ctx[r])
        good = ~bad[:n]
        # keys on a bad page keep whatever the buffer held; the rest match the oracle
        assert np.all(got[r, :n][bad[:n]] == sentinel)
        m = np.abs(ref[r, :n][good]).max()
        assert np.abs(got[r, :n][good] - ref[r, :n][good]).max() <= 1e-3 * m


@pytest.mark.parametrize("B_keep", [6, 64])  # rows split over the clusters, and whole rows
def test_decode_attention_bad_page_is_skipped_and_flagged(B_keep):
    dsa = lib()
    cfg, d, bt, ctx = _bad_page_case()
    B, k = len(ctx), cfg.k
    g = np.random.default_rng(5)
    idx = np.full((B, k), -1, np.int32)
    for b in range(B):
        m = min(k, int(ctx[b]))
        idx[b, :m] = np.sort(g.choice(int(ctx[b]), size=m, replace=False))
    if B_keep > B:  # tile the rows so the batch keeps whole rows per cluster
        reps = (B_keep + B - 1) // B
        sel = np.tile(np.arange(B), reps)[:B_keep]
    else:
        sel = np.arange(B)
    q = d["q"][torch.as_tensor(sel, device=DEV)].contiguous()
    bt_s = bt[torch.as_tensor(sel, device=DEV)].contiguous()
    ctx_s = torch.as_tensor(ctx[sel], device=DEV)
    idx_s = torch.as_tensor(idx[sel], device=DEV)
    n = len(sel)
    out = torch.empty((n, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((n, cfg.H), dtype=torch.float32, device=DEV)
    dsa.dsa_sparse_mla_decode_paged(q, d["kv_pool"], bt_s, ctx_s, idx_s, cfg.sm_scale, out, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == dsa_mod.DSA_DEV_BAD_PAGE
    o_ref, l_ref = oracle.sparse_mla_paged(bits16(q), bits16(d["kv_pool"]), bt_s.cpu().numpy(), ctx[sel], idx[sel],
                                           cfg.sm_scale)
    check_attention(out.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, l_ref)
