"""Pins of the oracle's indexer warm-up (training) path, CPU only.

The pages give the warm-up only in words (release summary "DeepSeek-V3.2-Exp:
Boosting Long-Context Efficiency with DeepSeek Sparse Attention", section
"Method": the indexer alone is trained against a KL-divergence-to-main-attention
target); the oracle's readings are stated in its source.  What pins them here:
central finite differences of the loss (every gradient element), the minimum
(target = the indexer's own distribution, taken from the already-pinned
indexer oracle, gives loss 0 and zero gradients), a closed form (w = 0 makes the
indexer uniform: loss = ln n - entropy(target)), and for the target its
reduction to a library softmax with one head, head-permutation invariance and
rows that sum to one."""
import numpy as np
import pytest
import torch

import oracle


def _bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def _bf(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def _case(seed, n=5, HI=3, dI=4, S=7, q_pos=(0, 2, 3, 6, 6)):
    g = np.random.default_rng(seed)
    q = g.standard_normal((n, HI, dI))
    k = g.standard_normal((S, dI))
    w = g.standard_normal((n, HI))
    qp = np.array(q_pos, dtype=np.int32)
    p = np.full((n, S), np.nan)
    for r in range(n):
        x = g.random(qp[r] + 1) + 0.1
        p[r, :qp[r] + 1] = x / x.sum()
    return q, w, qp, k, p


def _total(q, w, qp, k, p):
    return oracle.indexer_kl(q, w, qp, k, p)[0].sum()


def test_gradients_match_central_differences():
    q, w, qp, k, p = _case(1)
    loss, dw, dq, dk = oracle.indexer_kl(q, w, qp, k, p)
    eps = 1e-6
    for arr, grad in ((w, dw), (q, dq), (k, dk)):
        flat = arr.reshape(-1)
        num = np.empty(flat.size)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            up = _total(q, w, qp, k, p)
            flat[i] = keep - eps
            dn = _total(q, w, qp, k, p)
            flat[i] = keep
            num[i] = (up - dn) / (2 * eps)
        assert np.allclose(grad.reshape(-1), num, rtol=1e-5, atol=1e-7), (grad.reshape(-1), num)


def test_minimum_at_the_indexers_own_distribution():
    """Target = softmax of the scores the pinned FP8 indexer oracle computes: loss 0, gradients 0."""
    g = np.random.default_rng(2)
    n, HI, dI, S = 4, 4, 32, 9
    q8 = g.integers(0, 0x7E, (n, HI, dI), dtype=np.uint8) | (g.integers(0, 2, (n, HI, dI), dtype=np.uint8) << 7)
    k8 = g.integers(0, 0x7E, (S, dI), dtype=np.uint8) | (g.integers(0, 2, (S, dI), dtype=np.uint8) << 7)
    qs = g.random(n).astype(np.float32) * 0.01 + 0.001
    ks = g.random(S).astype(np.float32) * 0.01 + 0.001
    w = g.standard_normal((n, HI)).astype(np.float32)
    qp = np.array([0, 3, 8, 8], dtype=np.int32)
    I = oracle.indexer(q8, qs, w, qp, k8, ks, ld=S)
    p = np.full((n, S), np.nan)
    for r in range(n):
        x = np.exp(I[r, :qp[r] + 1] - I[r, :qp[r] + 1].max())
        p[r, :qp[r] + 1] = x / x.sum()
    dec = np.vectorize(oracle.e4m3)
    qd = dec(q8) * qs[:, None, None].astype(np.float64)
    kd = dec(k8) * ks[:, None].astype(np.float64)
    loss, dw, dq, dk = oracle.indexer_kl(qd, w.astype(np.float64), qp, kd, p)
    assert np.allclose(loss, 0.0, atol=1e-12)
    assert np.allclose(dw, 0.0, atol=1e-10) and np.allclose(dq, 0.0, atol=1e-10) and np.allclose(dk, 0.0, atol=1e-10)


def test_uniform_indexer_closed_form():
    """w = 0: the indexer's distribution is uniform over the n = t + 1 keys, so the loss is
    ln n - entropy(p); dq and dk vanish (every path to them carries a factor w)."""
    q, w, qp, k, p = _case(3)
    w[:] = 0.0
    loss, dw, dq, dk = oracle.indexer_kl(q, w, qp, k, p)
    for r in range(len(qp)):
        pr = p[r, :qp[r] + 1]
        assert np.isclose(loss[r], np.log(qp[r] + 1) + np.sum(pr * np.log(pr)), rtol=1e-12)
    assert np.allclose(dq, 0.0) and np.allclose(dk, 0.0)
    assert np.any(np.abs(dw) > 1e-3)  # w still receives a gradient


def test_target_one_head_is_the_library_softmax():
    g = np.random.default_rng(4)
    n, S, D = 3, 11, 576
    qb = _bits(g.standard_normal((n, 1, D)))
    kvb = _bits(g.standard_normal((S, D)))
    qp = np.array([0, 5, 10], dtype=np.int32)
    p = oracle.attn_target(qb, kvb, qp, 1 / 24)
    qf, kf = torch.from_numpy(_bf(qb)[:, 0]), torch.from_numpy(_bf(kvb))
    for r in range(n):
        ref = torch.softmax(qf[r] @ kf[:qp[r] + 1].T / 24, dim=0).numpy()
        assert np.allclose(p[r, :qp[r] + 1], ref, rtol=1e-12, atol=1e-15)
        assert np.all(np.isnan(p[r, qp[r] + 1:]))  # past the row: untouched


def test_target_is_the_head_mean_and_sums_to_one():
    g = np.random.default_rng(5)
    n, H, S, D = 2, 6, 9, 576
    qb = _bits(g.standard_normal((n, H, D)) * 2)
    kvb = _bits(g.standard_normal((S, D)))
    qp = np.array([4, 8], dtype=np.int32)
    p = oracle.attn_target(qb, kvb, qp, 1 / 24)
    for r in range(n):
        assert np.isclose(np.nansum(p[r]), 1.0, rtol=1e-12)
    perm = g.permutation(H)
    assert np.allclose(oracle.attn_target(qb[:, perm], kvb, qp, 1 / 24), p, rtol=1e-12, equal_nan=True)
    heads = [oracle.attn_target(qb[:, h:h + 1], kvb, qp, 1 / 24) for h in range(H)]
    assert np.allclose(np.mean(heads, axis=0), p, rtol=1e-12, equal_nan=True)


def test_relu_decision_is_exact_at_cancellation():
    """[a > 0] is taken on the exact dot product (ReLU'(0) = 0).  Codes (15, 15, 15) . (15, -16, 1)
    cancel to exactly 0 (225 - 240 + 15); times the fp32 scales 0.3 and 0.7 the fp64 products
    round so that their plain fp64 sum is +3.6e-15.  That key must be masked, so dq and dk come
    from the other key alone, by hand."""
    qs, ks = float(np.float32(0.3)), float(np.float32(0.7))
    dI = 128
    qrow = np.zeros(dI)
    qrow[:3] = 15 * qs
    k0 = np.zeros(dI)
    k0[:3] = np.array([15.0, -16.0, 1.0]) * ks
    naive = 0.0
    for d in range(3):
        naive += qrow[d] * k0[d]
    assert naive > 0.0  # the plain fp64 sum would switch the term on
    k1 = np.zeros(dI)
    k1[0] = 2.0 * ks
    w = np.array([[0.5]])
    p = np.array([[0.3, 0.7]])
    loss, dw, dq, dk = oracle.indexer_kl(qrow[None, None, :], w, np.array([1], dtype=np.int32), np.stack([k0, k1]), p)
    a1 = float(qrow @ k1)
    I = np.array([0.0, 0.5 * a1])
    sm = np.exp(I - I.max()) / np.exp(I - I.max()).sum()
    g = sm - p[0]
    assert np.allclose(dq[0, 0], g[1] * 0.5 * k1, rtol=1e-12, atol=0.0)
    assert np.array_equal(dk[0], np.zeros(dI))
    assert np.allclose(dk[1], g[1] * 0.5 * qrow, rtol=1e-12, atol=0.0)
    assert np.isclose(dw[0, 0], g[1] * a1, rtol=1e-12)
