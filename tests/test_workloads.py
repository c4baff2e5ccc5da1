"""Seeded input generators: determinism, shapes and the FP8 fixture quantiser (CPU)."""
import numpy as np
import torch

import dsa_workloads as W


def test_prefill_inputs_are_deterministic_and_shaped():
    cfg = W.CONFIGS["tiny"]
    a = W.prefill_inputs(cfg, "cpu")
    b = W.prefill_inputs(cfg, "cpu")
    for key in a:
        assert torch.equal(a[key], b[key]), key
    L = cfg.L
    assert a["q8"].shape == (L, cfg.HI, cfg.dI) and a["q8"].dtype == torch.uint8
    assert a["k8"].shape == (L, cfg.dI) and a["ks"].shape == (L,)
    assert a["q"].shape == (L, cfg.H, 576) and a["q"].dtype == torch.bfloat16
    assert a["kv"].shape == (L, 576)
    c = W.prefill_inputs(cfg, "cpu", seed=cfg.seed + 1)
    assert not torch.equal(a["q"], c["q"])


def test_fp8_quantiser_per_token_amax():
    x = torch.randn(33, 4, 32, generator=torch.Generator().manual_seed(0))
    x[5] = 0
    codes, scale = W.quantize_fp8_per_token(x)
    deq = codes.view(torch.float8_e4m3fn).float() * scale[:, None, None]
    amax = x.reshape(33, -1).abs().amax(1)
    assert scale[5] == 1 and torch.all(codes[5] == 0)
    nz = amax > 0
    assert torch.allclose(scale[nz], amax[nz] / 448)
    # the largest magnitude of every token maps to code +-448
    top = codes.view(torch.float8_e4m3fn).float().reshape(33, -1).abs().amax(1)
    assert torch.all(top[nz] == 448)
    # E4M3 has 3 mantissa bits: relative error <= 2^-4 for normal values
    big = x.abs() > scale[:, None, None] * 2 ** -6 * 8
    rel = ((deq - x).abs() / x.abs())[big]
    assert rel.max() <= 2 ** -4 + 1e-6


def test_decode_layout_pool_is_a_permutation():
    cfg = W.CONFIGS["decode_paged"]
    ctx, bt, P = W.decode_layout(cfg, B=8, ctx_lo=1, ctx_hi=300)
    pages = bt[bt >= 0]
    assert sorted(pages.tolist()) == list(range(P))
    for b in range(8):
        n = (int(ctx[b]) + 63) // 64
        assert torch.all(bt[b, :n] >= 0) and torch.all(bt[b, n:] == -1)
    d = W.decode_inputs(cfg, "cpu", B=4, ctx_lo=70, ctx_hi=130)
    for b in range(4):
        c = int(d["ctx"][b])
        if c % 64:
            page = int(d["block_table"][b, (c - 1) // 64])
            assert torch.isnan(d["kv_pool"][page, c % 64:].float()).all()
            assert torch.isnan(d["ks_pool"][page, c % 64:]).all()
            assert torch.isfinite(d["kv_pool"][page, : c % 64].float()).all()


def test_prefill_rows_match_the_full_draw(monkeypatch):
    """prefill_rows gives the bytes of prefill_inputs at the chosen rows, also when the
    rows fall in several generator chunks (chunk size shrunk so that they do)."""
    monkeypatch.setattr(W, "_CHUNK_ELEMS", 1 << 14)
    cfg = W.CONFIGS["tiny"]
    full = W.prefill_inputs(cfg, "cpu")
    rows = np.array([0, 3, 70, 71, 128, 200, 255])
    part = W.prefill_rows(cfg, "cpu", rows)
    for key in ("q8", "qs", "w", "q", "q_pos"):
        assert torch.equal(part[key], full[key][rows]), key
    for key in ("k8", "ks", "kv"):
        assert torch.equal(part[key], full[key]), key
