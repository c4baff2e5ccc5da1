"""GPU parity of the indexer warm-up path (dsa_indexer_warmup) against the fp64 oracle,
through the C ABI.

The oracle computes the target (the main attention's head-averaged dense causal
distribution) from the bf16 bits of q and kv, and the loss and gradients from the
dequantised FP8 indexer inputs (codes decoded by the oracle's own E4M3 decoder,
times their scales).  The kernels take each gradient's ReLU decision on the exact
dot product of the codes, as the oracle does; a planted row pair whose products
cancel to a tiny or zero sum checks that where fp32 would lose the sign.  Sizes
span several 128-row and 128-key backward tiles with ragged tails; a chunk of rows
over a longer prefix, fewer heads, both indexer head counts, and positions past the
keys are covered.  Tolerances: loss per row within 1e-4 + 1e-3 |loss|; each
gradient tensor within 1e-3 of its largest magnitude, element by element (fp32
arithmetic after the tensor-core products).
"""
import dataclasses

import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from tests.gpu_util import bits16, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL = 1e-3


def _e4m3_table():
    return np.array([oracle.e4m3(c) for c in range(256)], dtype=np.float64)


def _run(x, q_pos, S, H):
    dsa = lib()
    T, HI, dI = x["q8"].shape
    loss = torch.full((T,), float("nan"), device=DEV)
    dw = torch.full((T, HI), float("nan"), device=DEV)
    dq = torch.full((T, HI, dI), float("nan"), device=DEV)
    dk = torch.full((S, dI), float("nan"), device=DEV)
    q = x["q"][:, :H].contiguous()
    dsa.dsa_indexer_warmup(q, x["kv"][:S].contiguous(), 1 / 24, x["q8"], x["qs"], x["w"], x["k8"][:S].contiguous(),
                           x["ks"][:S].contiguous(), q_pos, loss, dw, dq, dk)
    torch.cuda.synchronize()
    status = dsa.dsa_get_device_status()
    tab = _e4m3_table()
    qd = tab[x["q8"].cpu().numpy()] * x["qs"].cpu().double().numpy()[:, None, None]
    kd = tab[x["k8"][:S].cpu().numpy()] * x["ks"][:S].cpu().double().numpy()[:, None]
    qp = q_pos.cpu().numpy()
    p = oracle.attn_target(bits16(q), bits16(x["kv"][:S]), qp, 1 / 24, ld=S)
    ref = oracle.indexer_kl(qd, x["w"].cpu().double().numpy(), qp, kd, p)
    got = [t.cpu().double().numpy() for t in (loss, dw, dq, dk)]
    return status, got, ref


def _check(got, ref):
    loss, dw, dq, dk = got
    rl, rdw, rdq, rdk = ref
    assert np.all(np.isfinite(loss)) and np.all(loss >= -1e-5)
    assert np.all(np.abs(loss - rl) <= 1e-4 + 1e-3 * np.abs(rl)), np.abs(loss - rl).max()
    for name, g, r in (("dw", dw, rdw), ("dq", dq, rdq), ("dk", dk, rdk)):
        assert np.all(np.isfinite(g)), name
        m = np.abs(r).max()
        err = np.abs(g - r).max()
        assert err <= REL * m + 1e-12, f"{name}: err {err} vs max {m}"


@pytest.mark.parametrize("L,H", [(300, 128), (700, 16)])
def test_warmup_causal_prefill(L, H):
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=L, seed=L)
    status, got, ref = _run(x, x["q_pos"], L, H)
    assert status == 0
    _check(got, ref)


def test_warmup_chunk_over_longer_prefix_h32():
    """Rows [S - 130, S) over keys [0, S), 32 indexer heads."""
    cfg = dataclasses.replace(W.CONFIGS["prefill_4k"], HI=32)
    S = 450
    x = W.prefill_inputs(cfg, DEV, L=S, seed=9)
    r0 = S - 130
    xc = dict(x)
    for key in ("q8", "qs", "w", "q"):
        xc[key] = x[key][r0:].contiguous()
    status, got, ref = _run(xc, x["q_pos"][r0:].contiguous(), S, 128)
    assert status == 0
    _check(got, ref)


def test_warmup_position_past_keys_is_clamped_and_flagged():
    S = 200
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=S, seed=4)
    q_pos = x["q_pos"].clone()
    q_pos[-1] = S + 50
    status, got, ref = _run(x, q_pos, S, 64)
    assert status & 0x2  # DSA_DEV_BAD_POSITION
    _check(got, ref)     # the oracle clamps the same way


def test_warmup_exact_relu_decision_at_cancellation():
    """Rows whose code products cancel: (448, 448, 2^-9) . (448, -448, +-2^-9) is +-2^-18 and
    (448, 448) . (448, -448) is 0, all of which an fp32 sum of the products in the wrong order
    rounds to 0, and a three-term sum that is exactly 0.  The gradient terms of those (row, key)
    pairs are included exactly when the exact sum is positive."""
    L = 300
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=L, seed=12)
    q8, k8 = x["q8"].clone(), x["k8"].clone()
    big, tiny, neg = 0x7E, 0x01, 0x80  # E4M3 codes of 448 and 2^-9; the sign bit
    for (t, j, s, sign) in [(250, 3, 40, 0), (250, 7, 41, neg), (251, 60, 42, None), (299, 0, 298, 0)]:
        q8[t, j].zero_()
        q8[t, j, :3] = torch.tensor([big, big, tiny], dtype=torch.uint8)
        k8[s].zero_()
        k8[s, :2] = torch.tensor([big, big | neg], dtype=torch.uint8)
        if sign is not None:
            k8[s, 2] = tiny | sign
    # (15, 15, 15) . (15, -16, 1) = 225 - 240 + 15 = 0 exactly, which a plain fp64 sum of the
    # dequantised products need not return
    q8[200, 9].zero_()
    q8[200, 9, :3] = torch.tensor([0x57, 0x57, 0x57], dtype=torch.uint8)
    k8[77].zero_()
    k8[77, :3] = torch.tensor([0x57, 0xD8, 0x38], dtype=torch.uint8)
    x = dict(x, q8=q8, k8=k8)
    status, got, ref = _run(x, x["q_pos"], L, 128)
    assert status == 0
    _check(got, ref)


def test_warmup_tiny_rows_and_a_row_with_no_keys():
    """Three rows over a 5-key prefix: positions -1 (no keys: zero loss and gradients), 0 (one
    key) and 4 (all five): single partial row and key tiles, most of them past the data."""
    S = 5
    x = W.prefill_inputs(W.CONFIGS["prefill_4k"], DEV, L=S, seed=21)
    rows = torch.tensor([0, 1, 4], device=DEV)
    xc = dict(x)
    for key in ("q8", "qs", "w", "q"):
        xc[key] = x[key][rows].contiguous()
    q_pos = torch.tensor([-1, 0, 4], dtype=torch.int32, device=DEV)
    status, got, ref = _run(xc, q_pos, S, 128)
    assert status == 0
    loss, dw, dq, dk = got
    assert loss[0] == 0.0 and np.all(dw[0] == 0.0) and np.all(dq[0] == 0.0)
    _check(got, ref)
