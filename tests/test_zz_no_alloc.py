"""GPU test of dsa_sparse_mla_decode_paged_noalloc, the decode attention entry
point for callers that cannot allocate device memory (for example a plugin
whose host program owns every device allocation, or a service held to a fixed
device-memory budget): it takes no workspace and uses a static device buffer
built into the library instead.

Each case runs two calls in a row on different inputs through the C ABI and
checks every call's output and LSE against dsa_sparse_mla_decode_paged (the
allocating entry point, workspace from PyTorch) within the attention
tolerance the other GPU tests use.  The small batch cuts its rows into pieces,
so the static buffer carries the partial results; the second call shows that
what the first left in the buffer does not leak into it.  The file is named
to be collected last."""
import numpy as np
import pytest
import torch

import dsa_workloads as W
from tests.gpu_util import check_attention, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _decode_case(B, k, seed):
    cfg = W.CONFIGS["decode_paged"]
    g = np.random.default_rng(seed)
    ctx = g.integers(1, 3 * k, size=B)
    ctx[0] = 1
    d = W.decode_inputs(cfg, DEV, ctx=ctx.tolist(), seed=seed)
    idx = np.full((B, k), -1, np.int32)
    for b in range(B):
        c = int(ctx[b])
        m = min(k, c + 2)
        idx[b, :m] = g.choice(np.arange(-1, c + 1), size=m, replace=False)
    return cfg, d, torch.from_numpy(idx).to(DEV)


@pytest.mark.parametrize("B,k", [(8, 2048), (64, 2048)])
def test_noalloc_decode_matches_allocating_entry_point(B, k):
    dsa = lib()
    H = W.CONFIGS["decode_paged"].H
    need = dsa.dsa_sparse_mla_decode_workspace_size(B, H, k)
    if B == 8:
        assert need > 0  # rows are cut into pieces: the static buffer is in use
    for call in range(2):
        cfg, d, idx = _decode_case(B, k, seed=100 * B + call)
        args = (d["q"], d["kv_pool"], d["block_table"], d["ctx"], idx, cfg.sm_scale)
        out_ref = torch.empty((B, H, 512), dtype=torch.bfloat16, device=DEV)
        lse_ref = torch.empty((B, H), dtype=torch.float32, device=DEV)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=DEV)
        dsa.dsa_sparse_mla_decode_paged(*args, out_ref, lse_ref, workspace=ws)
        out = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
        dsa.dsa_sparse_mla_decode_paged_noalloc(*args, out, lse)
        torch.cuda.synchronize()
        assert dsa.dsa_get_device_status() == 0
        check_attention(out.cpu().double().numpy(), lse.cpu().double().numpy(),
                        out_ref.cpu().double().numpy(), lse_ref.cpu().double().numpy())
