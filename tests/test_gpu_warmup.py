"""GPU parity of the indexer warm-up path (dsa_indexer_warmup) against the fp64 oracle,
through the C ABI.

The oracle computes the target (the main attention's head-averaged dense causal
distribution) from the bf16 bits of q and kv, and the loss and gradients from the
dequantised FP8 indexer inputs (codes decoded by the oracle's own E4M3 decoder,
times their scales; the gradients' ReLU decisions are taken on the dot products
formed as the kernel forms them in fp32, since rounding can flip a decision near
a = 0).  Sizes span several 128-key target tiles and 64-key backward
tiles with ragged tails; a chunk of rows over a longer prefix, fewer heads, both
indexer head counts, and positions past the keys are covered.  Tolerances: loss
per row within 1e-4 + 1e-3 |loss|; each gradient tensor within 1e-3 of its largest
magnitude, element by element (fp32 arithmetic after the tensor-core products).
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
    # ReLU decisions on the fp32 dot products the kernel forms (a discrete outcome that rounding
    # can flip near a = 0); every value of the oracle stays fp64
    ref = oracle.indexer_kl(qd, x["w"].cpu().double().numpy(), qp, kd, p, mask_fp32=True)
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
