"""GPU parity of the fused indexer -> top-k (dsa_indexer_topk), through the C ABI.

The fused call never writes the index scores, so its output is checked two ways:
byte for byte against the two-call path on the same inputs (dsa_indexer_logits
then dsa_topk, whose scores are the same fp32 values), and against the oracle's
top-k of the GPU's own scores on sampled rows (the oracle's top-k is the
definition; it runs on the GPU scores so that both sides rank the same values).
Cases cover rows short enough to keep every key, rows long enough to take the
sampled threshold, chunked rows over a longer prefix, both head counts, k below,
at and above 2048, and rows built so their samples mislead the threshold (too
few candidates, and ties that overflow the candidate list), which take the
full-score path.
"""
import dataclasses

import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from tests.gpu_util import lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _two_call(dsa, x, k, rows_pos, S):
    T = rows_pos.shape[0]
    logits = torch.full((T, S), float("nan"), device=DEV)
    dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], rows_pos, logits)
    vlen = torch.clamp(rows_pos + 1, max=S).int()
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    dsa.dsa_topk(logits, vlen, k, idx)
    return logits, vlen, idx


def _check(x, k, q_pos, S, sample_rows=16, seed=0):
    dsa = lib()
    T = q_pos.shape[0]
    logits, vlen, ref = _two_call(dsa, x, k, q_pos, S)
    got = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    dsa.dsa_indexer_topk(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], q_pos, k, got)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    assert torch.equal(got, ref), f"{(got != ref).any(1).sum().item()} rows differ from the two-call path"
    g = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, T - 1], g.integers(0, T, sample_rows)]))
    lg = logits[torch.as_tensor(rows, device=DEV)].cpu().double().numpy()
    o = oracle.topk(np.nan_to_num(lg, nan=-np.inf), vlen.cpu().numpy()[rows], k)
    assert np.array_equal(got.cpu().numpy()[rows], o)
    return got


@pytest.mark.parametrize("L", [1, 700, 5000, 9000, 20000])
def test_fused_causal_prefill(L):
    """Every row of a causal prefill: rows up to 4096 keys keep every key, longer rows
    take the sampled threshold."""
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=L, seed=L)
    _check(x, 2048, x["q_pos"], L, seed=L)


@pytest.mark.parametrize("k", [64, 1000, 3000, 4096])
def test_fused_k_range(k):
    L = 20000  # rows past max(4096, 2k) keys take the threshold
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=L, seed=k)
    _check(x, k, x["q_pos"], L, seed=k)


def test_fused_h32():
    cfg = dataclasses.replace(W.CONFIGS["prefill_4k"], HI=32)
    L = 10000
    x = W.prefill_inputs(cfg, DEV, L=L, seed=32)
    _check(x, 2048, x["q_pos"], L, seed=32)


def test_fused_chunk_over_longer_prefix():
    """A chunk of rows [S - 3000, S) over keys [0, S), as in chunked prefill; rows sit at
    unaligned positions and the last row count is not a multiple of the row group."""
    S = 40000
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=S, seed=7)
    r0 = S - 3001
    xc = dict(x)
    for key in ("q8", "qs", "w"):
        xc[key] = x[key][r0:].contiguous()
    q_pos = x["q_pos"][r0:].contiguous()
    _check(xc, 2048, q_pos, S, seed=7)


def _planted(S, seed):
    """Keys at the sample positions floor(j S / 2048) get a scale 10^4 times the others',
    so the samples put the threshold where only ~k/4 keys of a row reach it: those rows
    collect fewer than k candidates and take the full-score path."""
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=S, seed=seed)
    ks = x["ks"].clone()
    ks.mul_(1e-2)
    pos = (torch.arange(2048, dtype=torch.int64) * S // 2048).to(DEV)
    ks[pos] = ks[pos] * 1e4
    x["ks"] = ks
    return x


def test_fused_fallback_too_few_candidates():
    S = 16384
    x = _planted(S, 11)
    _check(x, 2048, x["q_pos"], S, seed=11)


def test_fused_fallback_ties_overflow():
    """Every key identical: all scores of a row tie, every key reaches the threshold,
    the candidate list overflows and the rows are redone; the tie rule keeps the
    smallest positions."""
    S = 12000
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=S, seed=5)
    x["k8"] = x["k8"][:1].expand(S, -1).contiguous()
    x["ks"] = torch.full_like(x["ks"], float(x["ks"][0]))
    got = _check(x, 2048, x["q_pos"], S, seed=5)
    # rows longer than k that score anything above zero keep the first k positions
    n = x["q_pos"].cpu().numpy() + 1
    g = got.cpu().numpy()
    long_rows = np.nonzero(n > 2048)[0]
    assert np.array_equal(g[long_rows[-1]], np.arange(2048))


def test_fused_position_past_keys_is_clamped_and_flagged():
    dsa = lib()
    S = 3000
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=S, seed=3)
    q_pos = x["q_pos"].clone()
    q_pos[5] = S + 100
    idx = torch.empty((S, 256), dtype=torch.int32, device=DEV)
    dsa.dsa_indexer_topk(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], q_pos, 256, idx)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() & 0x2  # DSA_DEV_BAD_POSITION
    q_pos[5] = S - 1
    _, _, ref = _two_call(dsa, x, 256, q_pos, S)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_status() == 0
    assert torch.equal(idx, ref)
