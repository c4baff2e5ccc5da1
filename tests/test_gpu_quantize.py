"""GPU parity of the per-token FP8 quantiser (a0) against the oracle: codes and
scales bit-exact (an integer decided by fp32 divisions on both sides), on ragged,
misaligned and edge-case rows, and at the full L=32768 indexer size against the
input fixture and sampled oracle rows."""
import numpy as np
import pytest
import torch

import dsa_workloads as W
import oracle
from tests.gpu_util import lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def edge_rows(cols: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    rows = [
        g.standard_normal(cols),                          # ordinary
        np.zeros(cols),                                   # all zero: scale 1
        -np.zeros(cols),                                  # negative zeros keep their sign bit
        g.standard_normal(cols) * 1e-30,                  # tiny: subnormal quotients round in E4M3
        g.standard_normal(cols) * 1e30,                   # huge magnitudes
        np.full(cols, 3.0),                               # constant row
        g.integers(-448, 449, cols).astype(np.float64),   # exact integers (ties at the E4M3 steps)
        g.standard_normal(cols) * 10 ** g.uniform(-3, 3, cols),
    ]
    return np.stack(rows).astype(np.float32)


def run(dsa, x: torch.Tensor, mode: int):
    rows = x.shape[0]
    codes = torch.empty(x.shape, dtype=torch.uint8, device=DEV)
    scale = torch.empty((rows,), dtype=torch.float32, device=DEV)
    dsa.dsa_quantize_fp8(x, codes, scale, mode)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scale.cpu().numpy()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("cols", [1, 3, 100, 128, 1023, 1024, 3000, 8192])
def test_quantize_matches_oracle(cols, mode):
    dsa = lib()
    x = edge_rows(cols, seed=cols + 7 * mode)
    g = np.random.default_rng(cols)
    x = np.concatenate([x, (g.standard_normal((37, cols)) * 10 ** g.uniform(-2, 2, (37, 1))).astype(np.float32)])
    c, s = run(dsa, torch.from_numpy(x).to(DEV), mode)
    c_ref, s_ref = oracle.quantize_fp8(x, mode)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(c, c_ref)


@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_misaligned_rows(mode):
    """Rows that start off a 16-byte boundary (x) or a 4-byte boundary (codes) take the scalar path."""
    dsa = lib()
    rows, cols = 9, 257
    x = np.concatenate([edge_rows(cols, 3), edge_rows(cols, 4)])[:rows]
    base = torch.zeros(rows * cols + 1, dtype=torch.float32, device=DEV)
    xd = base[1:].view(rows, cols)
    xd.copy_(torch.from_numpy(x))
    cbase = torch.zeros(rows * cols + 1, dtype=torch.uint8, device=DEV)
    codes = cbase[1:].view(rows, cols)
    scale = torch.empty((rows,), dtype=torch.float32, device=DEV)
    dsa.dsa_quantize_fp8(xd, codes, scale, mode)
    torch.cuda.synchronize()
    c_ref, s_ref = oracle.quantize_fp8(x, mode)
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert int(cbase[0]) == 0  # nothing written before the first row


def test_quantize_full_size_indexer_queries():
    """L=32768 query rows (64 heads x 128): the kernel equals the input fixture bit for bit
    (amax/448 mode), and sampled rows equal the oracle in both modes."""
    dsa = lib()
    cfg = W.CONFIGS["prefill_32k"]
    x = W.randn((cfg.L, cfg.HI, cfg.dI), DEV, cfg.seed, 10)
    q8_fix, qs_fix = W.quantize_fp8_per_token(x)
    codes = torch.empty(x.shape, dtype=torch.uint8, device=DEV)
    scale = torch.empty((cfg.L,), dtype=torch.float32, device=DEV)
    dsa.dsa_quantize_fp8(x, codes, scale, 0)
    torch.cuda.synchronize()
    assert torch.equal(scale, qs_fix)
    assert torch.equal(codes, q8_fix)
    rows = np.array([0, 1, 4095, 4096, 20000, cfg.L - 1])
    xs = x[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    for mode in (0, 1):
        dsa.dsa_quantize_fp8(x, codes, scale, mode)
        torch.cuda.synchronize()
        c_ref, s_ref = oracle.quantize_fp8(xs, mode)
        r = torch.as_tensor(rows, device=DEV)
        assert np.array_equal(scale[r].cpu().numpy(), s_ref)
        assert np.array_equal(codes[r].cpu().numpy(), c_ref)
