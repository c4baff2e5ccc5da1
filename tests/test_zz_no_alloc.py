"""GPU test of dsa_sparse_mla_decode_paged_noalloc, the decode attention entry
point for callers that cannot allocate device memory (for example a plugin
whose host program owns every device allocation, or a service held to a fixed
device-memory budget): it takes no workspace and uses a static device buffer
built into the library instead.

Each case runs two calls in a row through the C ABI with different batch
shapes, so the second call's work split (which rows are cut into pieces, and
which workspace slots those pieces use) differs from the first's: a merge that
read a slot the current call did not write would find the previous call's data
and change the result.  Both entry points run the same plan and kernels, so
every call's output and LSE must be bit-identical to those of
dsa_sparse_mla_decode_paged (the allocating entry point, workspace from
PyTorch).  The file is named to be collected last."""
import numpy as np
import pytest
import torch

import dsa_workloads as W
from tests.gpu_util import lib

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


@pytest.mark.parametrize("calls", [[(8, 2048), (4, 512)], [(16, 1024), (3, 2048)], [(64, 2048), (8, 300)]])
def test_noalloc_decode_matches_allocating_entry_point(calls):
    dsa = lib()
    H = W.CONFIGS["decode_paged"].H
    for n, (B, k) in enumerate(calls):
        need = dsa.dsa_sparse_mla_decode_workspace_size(B, H, k)
        if B <= 16:
            assert need > 0  # rows are cut into pieces: the static buffer is in use
        cfg, d, idx = _decode_case(B, k, seed=100 * B + k + n)
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
        assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16)), f"call {n}: out differs"
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), f"call {n}: lse differs"
