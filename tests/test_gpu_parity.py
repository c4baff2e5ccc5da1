"""GPU parity of each stage against the fp64 oracle, through the C ABI.

Sizes are chosen so the oracle finishes in seconds while still spanning several
tiles and a ragged tail (query rows, key tiles of 128, attention blocks of 64,
pages of 64).  Seeded synthetic inputs only.
"""
import dataclasses

import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from tests.gpu_util import bits16, check_attention, check_logits, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _indexer_case(cfg, L, rows=None):
    dsa = lib()
    x = W.prefill_inputs(cfg, DEV, L=L)
    logits = torch.full((L, L + 3), float("nan"), device=DEV)  # ld not a multiple of 4
    dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], logits)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    rows = np.arange(L) if rows is None else np.asarray(rows)
    h = {k: v.cpu() for k, v in x.items()}
    ref = oracle.indexer(h["q8"][rows].numpy(), h["qs"][rows].numpy(), h["w"][rows].numpy(), rows,
                         h["k8"].numpy(), h["ks"].numpy(), ld=L + 3)
    got = logits.cpu().double().numpy()[rows]
    check_logits(got, ref, rows)
    return x, logits


def test_indexer_tiny_all_rows():
    _indexer_case(W.CONFIGS["tiny"], 256)


@pytest.mark.parametrize("L", [1, 7, 129, 700])
def test_indexer_h64_ragged(L):
    rng = np.random.default_rng(L)
    rows = np.unique(np.concatenate([[0, L - 1, min(127, L - 1), min(128, L - 1)], rng.integers(0, L, 40)]))
    _indexer_case(W.CONFIGS["prefill_4k"], L, rows)


@pytest.mark.parametrize("L", [129, 700])
def test_indexer_h32_ragged(L):
    """The H_I = 32 instantiation of the contiguous indexer (half the heads per token)."""
    cfg = dataclasses.replace(W.CONFIGS["prefill_4k"], HI=32)
    rng = np.random.default_rng(L + 32)
    rows = np.unique(np.concatenate([[0, L - 1, min(127, L - 1), min(128, L - 1)], rng.integers(0, L, 40)]))
    _indexer_case(cfg, L, rows)


def test_paged_indexer_h32():
    """The H_I = 32 instantiation of the paged indexer over a shuffled page pool."""
    cfg = dataclasses.replace(W.CONFIGS["decode_paged"], HI=32)
    dsa = lib()
    ctx = [1, 64, 65, 2047, 3001, 5000]
    d = W.decode_inputs(cfg, DEV, ctx=ctx)
    B, ld = len(ctx), max(ctx) + 3
    logits = torch.full((B, ld), float("nan"), device=DEV)
    dsa.dsa_indexer_logits(d["q8"], d["qs"], d["w"], d["k8_pool"], d["ks_pool"], d["q_pos"], logits,
                           block_table=d["block_table"])
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    h = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}
    ref = oracle.indexer_paged(h["q8"].numpy(), h["qs"].numpy(), h["w"].numpy(), h["ctx"].numpy(),
                               h["k8_pool"].numpy(), h["ks_pool"].numpy(), h["block_table"].numpy(), ld)
    check_logits(logits.cpu().double().numpy(), ref, h["q_pos"].numpy())


def test_topk_from_gpu_logits_bit_exact():
    cfg = W.CONFIGS["tiny"]
    dsa = lib()
    x, logits = _indexer_case(cfg, 256)
    for k in (1, 64, 100, 256, 300):
        idx = torch.empty((256, k), dtype=torch.int32, device=DEV)
        dsa.dsa_topk(logits, x["q_pos"] + 1, k, idx)
        torch.cuda.synchronize()
        ref = oracle.topk(np.nan_to_num(logits.cpu().double().numpy(), nan=0.0), np.arange(1, 257), k)
        assert np.array_equal(idx.cpu().numpy(), ref), f"k={k}"


# At most two rows per SM run on the cluster kernel (one cluster per row), more rows on
# the one-CTA-per-row kernel; tiling the same rows REPS_MANY_ROWS times (more than 304
# rows) sends them through the latter.  Both fall back to the four histogram passes for
# rows whose candidates miss [k, cap] (the all-ties row below, the planted rows after it).
REPS_MANY_ROWS = 40


@pytest.mark.parametrize("reps", [1, REPS_MANY_ROWS])
@pytest.mark.parametrize("ld", [4099, 4096])
def test_topk_edge_rows_and_ties(ld, reps):
    """Valid lengths 0, 1, k-1, k, k+1, ld; tie-heavy integer scores with -0/+0;
    ld both aligned and unaligned (vector and scalar paths); few rows and many."""
    dsa = lib()
    g = torch.Generator(device=DEV).manual_seed(3)
    T = 24
    vals = torch.randint(-20, 21, (T, ld), generator=g, device=DEV).float() * 0.5
    vals[vals == 0] = torch.where(torch.rand((T, ld), generator=g, device=DEV) < 0.5, -0.0, 0.0)[vals == 0]
    vals[5:10] = torch.randn((5, ld), generator=g, device=DEV)
    k = 2048
    n = torch.tensor([0, 1, k - 1, k, k + 1, ld, ld, 3000, 2049, 4000, 7, ld - 1] * 2, dtype=torch.int32)
    # poison past the valid length: any read of it would change the result
    for r in range(T):
        vals[r, int(n[r]):] = float("nan")
    idx = torch.empty((T * reps, k), dtype=torch.int32, device=DEV)
    dsa.dsa_topk(vals.repeat(reps, 1), n.repeat(reps).to(DEV), k, idx)
    torch.cuda.synchronize()
    v = vals.cpu().double().numpy()
    ref = oracle.topk(np.nan_to_num(v, nan=-np.inf), n.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), np.tile(ref, (reps, 1)))
    assert dsa.dsa_get_device_status() == 0


@pytest.mark.parametrize("reps", [1, REPS_MANY_ROWS])
def test_topk_deterministic_large_row(reps):
    dsa = lib()
    T, ld = 8, 131072
    g = torch.Generator(device=DEV).manual_seed(4)
    vals = torch.randn((T, ld), generator=g, device=DEV)
    vals[:, ::7] = 0.25  # a large tie block straddling the threshold
    vals[7] = 1.0        # one tie over the whole row: every key passes the sampled threshold
    n = torch.tensor([ld, ld - 5, 70000, 2049, 65536, 131071, 4096, 100000], dtype=torch.int32, device=DEV)
    a = torch.empty((T * reps, 2048), dtype=torch.int32, device=DEV)
    b = torch.empty_like(a)
    vals_r, n_r = vals.repeat(reps, 1), n.repeat(reps)
    dsa.dsa_topk(vals_r, n_r, 2048, a)
    dsa.dsa_topk(vals_r, n_r, 2048, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    ref = oracle.topk(vals.cpu().double().numpy(), n.cpu().numpy(), 2048)
    assert np.array_equal(a.cpu().numpy(), np.tile(ref, (reps, 1)))


@pytest.mark.parametrize("k", [1000, 2048, 2049])
def test_topk_many_rows_planted_and_ties(k):
    """More rows than two per SM.  Rows 0-1 hold scores that grow along the row with the
    row's largest scores planted at 512 evenly spaced positions, so a sampled threshold can
    miss the k-th key (those rows then take the four histogram passes); row 2 is integer
    ties, the rest random; unaligned rows; k below, at and above the workload's 2048."""
    dsa = lib()
    g = torch.Generator(device=DEV).manual_seed(9)
    ld = 32771
    n = torch.tensor([ld, 32768, 20000, 9000, 5000, 3500, 3073, ld - 2], dtype=torch.int32)
    vals = torch.randn((len(n), ld), generator=g, device=DEV)
    for r in (0, 1):
        nr = int(n[r])
        vals[r, :nr] = torch.arange(nr, device=DEV, dtype=torch.float32) * 1e-3
        pos = (torch.arange(512, device=DEV, dtype=torch.int64) * nr) // 512
        vals[r, pos] = 1e6 + torch.arange(512, device=DEV, dtype=torch.float32)
    vals[2] = torch.randint(-8, 9, (ld,), generator=g, device=DEV).float()
    for r in range(len(n)):
        vals[r, int(n[r]):] = float("nan")
    reps = REPS_MANY_ROWS
    idx = torch.empty((len(n) * reps, k), dtype=torch.int32, device=DEV)
    dsa.dsa_topk(vals.repeat(reps, 1), n.repeat(reps).to(DEV), k, idx)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    ref = oracle.topk(np.nan_to_num(vals.cpu().double().numpy(), nan=-np.inf), n.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), np.tile(ref, (reps, 1)))


def _mla_case(T, S, H, k, seed, invalid_frac=0.0, rows=None):
    dsa = lib()
    g = torch.Generator(device=DEV).manual_seed(seed)
    q = torch.randn((T, H, 576), generator=g, device=DEV).to(torch.bfloat16)
    kv = torch.randn((S, 576), generator=g, device=DEV).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(S, generator=g, device=DEV)[:k] for _ in range(T)]).int()
    idx = torch.sort(idx, dim=1).values
    if invalid_frac > 0:
        drop = torch.rand((T, k), generator=g, device=DEV) < invalid_frac
        idx[drop] = -1
        idx[0, :] = -1          # a row with nothing valid
        idx[1, 1:] = -1         # a row with a single valid entry
        idx[2, 5] = S + 7       # out of range: skipped
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((T, H), dtype=torch.float32, device=DEV)
    dsa.dsa_sparse_mla_prefill(q, kv, idx, 1 / 24, out, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    rows = np.arange(T) if rows is None else np.asarray(rows)
    o_ref, l_ref = oracle.sparse_mla(bits16(q)[rows], bits16(kv), idx.cpu().numpy()[rows], 1 / 24)
    o = out.cpu().double().numpy()[rows]
    l = lse.cpu().double().numpy()[rows]
    if invalid_frac > 0:
        assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    return check_attention(o, l, o_ref, l_ref)


@pytest.mark.parametrize("H", [128, 16, 64])
def test_mla_prefill_small(H):
    _mla_case(T=6, S=300, H=H, k=64, seed=H)


def test_mla_prefill_ragged_k_and_invalid():
    _mla_case(T=5, S=1000, H=128, k=200, seed=1, invalid_frac=0.3)


def test_mla_prefill_k2048():
    _mla_case(T=9, S=5000, H=128, k=2048, seed=2, rows=[0, 4, 8])


def test_pipeline_tiny_end_to_end():
    """indexer -> top-k -> sparse MLA on the tiny workload, every row."""
    cfg = W.CONFIGS["tiny"]
    dsa = lib()
    x, logits = _indexer_case(cfg, 256)
    idx = torch.empty((256, cfg.k), dtype=torch.int32, device=DEV)
    dsa.dsa_topk(logits, x["q_pos"] + 1, cfg.k, idx)
    out = torch.empty((256, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((256, cfg.H), dtype=torch.float32, device=DEV)
    dsa.dsa_sparse_mla_prefill(x["q"], x["kv"], idx, cfg.sm_scale, out, lse)
    torch.cuda.synchronize()
    ref_idx = oracle.topk(np.nan_to_num(logits.cpu().double().numpy(), nan=0.0), np.arange(1, 257), cfg.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    o_ref, l_ref = oracle.sparse_mla(bits16(x["q"]), bits16(x["kv"]), ref_idx, cfg.sm_scale)
    check_attention(out.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, l_ref)
    # rows t <= 63 select every prior token: sparse equals dense there (checked in the oracle pins)


def test_decode_paged_pipeline():
    """Paged indexer -> top-k -> paged sparse MLA for one new token per sequence.

    Context lengths cover one token, page boundaries, fewer than k and more
    than k candidates; pages are a shuffled pool and unused slots hold NaN."""
    cfg = W.CONFIGS["decode_paged"]
    dsa = lib()
    ctx = [1, 64, 65, 2047, 2048, 2049, 3001, 5000]
    d = W.decode_inputs(cfg, DEV, ctx=ctx)
    B = len(ctx)
    ld = max(ctx) + 5
    logits = torch.full((B, ld), float("nan"), device=DEV)
    dsa.dsa_indexer_logits(d["q8"], d["qs"], d["w"], d["k8_pool"], d["ks_pool"], d["q_pos"], logits,
                           block_table=d["block_table"])
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    h = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}
    ref = oracle.indexer_paged(h["q8"].numpy(), h["qs"].numpy(), h["w"].numpy(), h["ctx"].numpy(),
                               h["k8_pool"].numpy(), h["ks_pool"].numpy(), h["block_table"].numpy(), ld)
    got = logits.cpu().double().numpy()
    check_logits(got, ref, h["q_pos"].numpy())
    idx = torch.empty((B, cfg.k), dtype=torch.int32, device=DEV)
    dsa.dsa_topk(logits, d["ctx"], cfg.k, idx)
    torch.cuda.synchronize()
    ref_idx = oracle.topk(np.nan_to_num(got, nan=0.0), h["ctx"].numpy(), cfg.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    out = torch.empty((B, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, cfg.H), dtype=torch.float32, device=DEV)
    ws_n = dsa.dsa_sparse_mla_decode_workspace_size(B, cfg.H, cfg.k)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=DEV) if ws_n else None
    dsa.dsa_sparse_mla_decode_paged(d["q"], d["kv_pool"], d["block_table"], d["ctx"], idx, cfg.sm_scale,
                                    out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    o_ref, l_ref = oracle.sparse_mla_paged(bits16(d["q"]), bits16(d["kv_pool"]), h["block_table"].numpy(),
                                           h["ctx"].numpy(), ref_idx, cfg.sm_scale)
    check_attention(out.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, l_ref)


@pytest.mark.parametrize("H", [16, 64])
@pytest.mark.parametrize("B", [5, 96])  # rows split over the clusters, and whole rows
def test_decode_fewer_heads(H, B):
    """Paged decode attention with fewer than 128 query heads (the MMA rows past H are
    zero and never stored), split and whole rows, against the oracle."""
    cfg = W.CONFIGS["decode_paged"]
    dsa = lib()
    k = 256
    g = np.random.default_rng(7 * H + B)
    ctx = g.integers(1, 3 * k, size=B)
    d = W.decode_inputs(cfg, DEV, ctx=ctx.tolist(), seed=H + B)
    idx_np = np.full((B, k), -1, np.int32)
    for b in range(B):
        c = int(ctx[b])
        m = min(k, c)
        idx_np[b, :m] = g.choice(c, size=m, replace=False)
    idx = torch.from_numpy(idx_np).to(DEV)
    q = d["q"][:, :H].contiguous()
    out = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
    dsa.dsa_sparse_mla_decode_paged(q, d["kv_pool"], d["block_table"], d["ctx"], idx, cfg.sm_scale, out, lse)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    o_ref, l_ref = oracle.sparse_mla_paged(bits16(q), bits16(d["kv_pool"]), d["block_table"].cpu().numpy(),
                                           ctx.astype(np.int32), idx_np, cfg.sm_scale)
    check_attention(out.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, l_ref)


@pytest.mark.parametrize("B,k", [(1, 2048), (3, 100), (5, 64), (17, 2048), (64, 2048), (75, 256), (100, 300)])
def test_decode_split_pieces(B, k):
    """Decode batches with fewer rows than SM pairs cut each row into pieces over
    the clusters (partial output and LSE per piece in the workspace, then a merge
    by LSE); larger batches keep whole rows.  Selections are unsorted and hold
    -1 and out-of-context entries; some contexts are shorter than k, so whole
    pieces see nothing valid."""
    cfg = W.CONFIGS["decode_paged"]
    dsa = lib()
    g = np.random.default_rng(1000 * B + k)
    ctx = g.integers(1, 3 * k, size=B)
    ctx[0] = 1
    d = W.decode_inputs(cfg, DEV, ctx=ctx.tolist(), seed=B + k)
    idx_np = np.full((B, k), -1, np.int32)
    for b in range(B):
        c = int(ctx[b])
        m = min(k, c + 2)
        idx_np[b, :m] = g.choice(np.arange(-1, c + 1), size=m, replace=False)
    idx = torch.from_numpy(idx_np).to(DEV)
    out = torch.empty((B, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, cfg.H), dtype=torch.float32, device=DEV)
    ws_n = dsa.dsa_sparse_mla_decode_workspace_size(B, cfg.H, k)
    ws = torch.full((max(ws_n, 1),), 0xFF, dtype=torch.uint8, device=DEV)  # NaN-filled: stale data shows
    dsa.dsa_sparse_mla_decode_paged(d["q"], d["kv_pool"], d["block_table"], d["ctx"], idx, cfg.sm_scale,
                                    out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    o_ref, l_ref = oracle.sparse_mla_paged(bits16(d["q"]), bits16(d["kv_pool"]), d["block_table"].cpu().numpy(),
                                           ctx.astype(np.int32), idx_np, cfg.sm_scale)
    check_attention(out.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, l_ref)
