"""Seeded synthetic inputs for the DSA hot path (shared by tests and bench).

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  The one preparation step it performs is the FP8 fixture
quantisation of the indexer inputs (per-token scale = amax / 448, codes rounded
to nearest-even and saturated to +-448), which sits upstream of the indexer: the
indexer's inputs are those codes plus their scales.

Shapes and distributions follow the workloads the pages describe for
DeepSeek-V3.2-Exp ("AMD Instinct MI355X GPUs Power DeepSeek-V3.2-Exp", section
"DeepSeek Sparse Attention (DSA)": FP8 indexer, top-2048 selection; release
summary "DeepSeek-V3.2-Exp: Boosting Long-Context Efficiency with DeepSeek
Sparse Attention", section "Method": MQA-mode MLA over a shared latent row):
  indexer: H_I heads of width d_I, q and k ~ N(0, 1), w ~ N(0, 1) * w_std;
  MLA: H query heads, latent width D = 576 (512 + 64 RoPE), V = first 512
  columns, Q and KV ~ N(0, 1) rounded to bf16; softmax scale 1/sqrt(576).

Every tensor is drawn in fixed row chunks, each from its own generator seeded
by (seed, tensor id, chunk), so a given seed gives the same bytes on every run
on the same device type.
"""
from __future__ import annotations

import dataclasses
import math

import torch

FP8_MAX = 448.0
D_LATENT = 576
D_V = 512
_CHUNK_ELEMS = 1 << 26  # elements drawn per generator call


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    L: int = 0              # prefill length (query rows = key rows = L)
    HI: int = 64            # indexer heads
    dI: int = 128           # indexer head width
    w_std: float = 0.125    # w ~ N(0,1) * w_std
    k: int = 2048           # selected tokens per query
    H: int = 128            # MLA query heads
    D: int = D_LATENT
    Dv: int = D_V
    chunk: int = 0          # chunked prefill: query rows per chunk (0 = unchunked)
    B: int = 0              # decode: sequences
    ctx_lo: int = 0         # decode: context length range, inclusive
    ctx_hi: int = 0
    page_size: int = 64
    seed: int = 0

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


CONFIGS = {
    "tiny": Config("tiny", L=256, HI=4, dI=32, w_std=0.5, k=64, H=16, seed=0),
    "prefill_4k": Config("prefill_4k", L=4096, seed=1),
    "prefill_32k": Config("prefill_32k", L=32768, seed=2),
    "decode_paged": Config("decode_paged", B=64, ctx_lo=8192, ctx_hi=65536, page_size=64, seed=3),
    "chunked_128k": Config("chunked_128k", L=131072, chunk=4096, seed=4),
}


def _gen(device, seed: int, tid: int, chunk: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tid * 10_007 + chunk * 101 + 17) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def randn(shape, device, seed: int, tid: int, std: float = 1.0, dtype=torch.float32) -> torch.Tensor:
    """N(0, std^2) samples in fixed row chunks, cast to ``dtype`` (round to nearest even)."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=dtype, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    row = flat.shape[1]
    rows_per = max(1, _CHUNK_ELEMS // max(row, 1))
    for c, r0 in enumerate(range(0, shape[0], rows_per)):
        r1 = min(shape[0], r0 + rows_per)
        x = torch.randn((r1 - r0, row), generator=_gen(device, seed, tid, c), device=device)
        if std != 1.0:
            x.mul_(std)
        flat[r0:r1].copy_(x.to(dtype))
    return out


def randn_rows(shape, rows, device, seed: int, tid: int, std: float = 1.0, dtype=torch.float32) -> torch.Tensor:
    """Rows ``rows`` (ascending) of ``randn(shape, ...)``, drawing only the chunks that hold them."""
    shape = tuple(int(s) for s in shape)
    rows = torch.as_tensor(rows, dtype=torch.int64)
    row = int(math.prod(shape[1:]))
    rows_per = max(1, _CHUNK_ELEMS // max(row, 1))
    out = torch.empty((len(rows), row), dtype=dtype, device=device)
    chunk_of = rows // rows_per
    for c in torch.unique(chunk_of).tolist():
        r0 = c * rows_per
        r1 = min(shape[0], r0 + rows_per)
        x = torch.randn((r1 - r0, row), generator=_gen(device, seed, tid, c), device=device)
        if std != 1.0:
            x.mul_(std)
        sel = (chunk_of == c).nonzero().flatten()
        out[sel.to(device)] = x[(rows[sel] - r0).to(device)].to(dtype)
    return out.view((len(rows),) + shape[1:])


def quantize_fp8_per_token(x: torch.Tensor):
    """Fixture quantiser: one scale per leading index over all trailing elements.

    scale = amax / 448 (1 when amax is 0); codes = RNE(x / scale) saturated to
    +-448, stored as E4M3.  Returns (codes as uint8, scale fp32).
    """
    n = x.shape[0]
    flat = x.reshape(n, -1).float()
    amax = flat.abs().amax(dim=1)
    # a tensor divisor: division by a Python scalar may run as a multiply by its
    # rounded reciprocal on CUDA, which is not the fp32 quotient
    scale = torch.where(amax > 0, amax / torch.full_like(amax, FP8_MAX), torch.ones_like(amax))
    codes = torch.empty(flat.shape, dtype=torch.uint8, device=x.device)
    step = max(1, _CHUNK_ELEMS // max(flat.shape[1], 1))
    for r0 in range(0, n, step):
        r1 = min(n, r0 + step)
        y = (flat[r0:r1] / scale[r0:r1, None]).clamp_(-FP8_MAX, FP8_MAX)
        codes[r0:r1] = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.view(x.shape), scale.contiguous()


def indexer_queries(cfg: Config, T: int, device, seed: int, tid0: int = 10):
    """q^I codes [T, HI, dI] + per-token scale [T] and head weights w [T, HI]."""
    qI = randn((T, cfg.HI, cfg.dI), device, seed, tid0)
    q8, qs = quantize_fp8_per_token(qI)
    del qI
    w = randn((T, cfg.HI), device, seed, tid0 + 1, std=cfg.w_std)
    return q8, qs, w


def indexer_keys(cfg: Config, S: int, device, seed: int, tid: int = 12):
    """k^I codes [S, dI] + per-token scale [S]."""
    kI = randn((S, cfg.dI), device, seed, tid)
    k8, ks = quantize_fp8_per_token(kI)
    return k8, ks


def prefill_inputs(cfg: Config, device, L: int | None = None, seed: int | None = None):
    """All inputs of a causal prefill over L tokens (queries at positions 0..L-1)."""
    L = cfg.L if L is None else L
    seed = cfg.seed if seed is None else seed
    q8, qs, w = indexer_queries(cfg, L, device, seed)
    k8, ks = indexer_keys(cfg, L, device, seed)
    q = randn((L, cfg.H, cfg.D), device, seed, 20, dtype=torch.bfloat16)
    kv = randn((L, cfg.D), device, seed, 21, dtype=torch.bfloat16)
    q_pos = torch.arange(L, dtype=torch.int32, device=device)
    return dict(q8=q8, qs=qs, w=w, k8=k8, ks=ks, q=q, kv=kv, q_pos=q_pos)


def prefill_rows(cfg: Config, device, rows, seed: int | None = None):
    """The query rows ``rows`` (ascending positions) of ``prefill_inputs(cfg)`` with all
    of the keys: the same bytes, without drawing the query chunks no row falls in."""
    seed = cfg.seed if seed is None else seed
    rows = torch.as_tensor(rows, dtype=torch.int64)
    L = cfg.L
    qI = randn_rows((L, cfg.HI, cfg.dI), rows, device, seed, 10)
    q8, qs = quantize_fp8_per_token(qI)
    del qI
    w = randn_rows((L, cfg.HI), rows, device, seed, 11, std=cfg.w_std)
    k8, ks = indexer_keys(cfg, L, device, seed)
    q = randn_rows((L, cfg.H, cfg.D), rows, device, seed, 20, dtype=torch.bfloat16)
    kv = randn((L, cfg.D), device, seed, 21, dtype=torch.bfloat16)
    q_pos = rows.to(torch.int32).to(device)
    return dict(q8=q8, qs=qs, w=w, k8=k8, ks=ks, q=q, kv=kv, q_pos=q_pos)


def decode_layout(cfg: Config, seed: int | None = None, B: int | None = None,
                  ctx_lo: int | None = None, ctx_hi: int | None = None, ctx=None):
    """Context lengths and a shuffled page pool (CPU tensors).

    Returns ctx [B] int32, block_table [B, max_pages] int32 (-1 past each
    sequence's pages) and the pool size.  Pages of all sequences are a random
    permutation of 0..num_pages-1.
    """
    seed = cfg.seed if seed is None else seed
    B = (cfg.B if B is None else B) if ctx is None else len(ctx)
    lo = cfg.ctx_lo if ctx_lo is None else ctx_lo
    hi = cfg.ctx_hi if ctx_hi is None else ctx_hi
    if ctx is None:
        g = _gen("cpu", seed, 30, 0)
        ctx = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    else:
        ctx = torch.as_tensor(ctx, dtype=torch.int32)
    ps = cfg.page_size
    npages = (ctx.to(torch.int64) + ps - 1) // ps
    num_pages = int(npages.sum())
    max_pages = int(npages.max())
    perm = torch.randperm(num_pages, generator=_gen("cpu", seed, 31, 0)).to(torch.int32)
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(npages[b])
        bt[b, :n] = perm[off:off + n]
        off += n
    return ctx, bt, num_pages


def decode_inputs(cfg: Config, device, seed: int | None = None, B: int | None = None,
                  ctx_lo: int | None = None, ctx_hi: int | None = None, poison: bool = True, ctx=None):
    """One decode step over a paged cache.

    Pools: FP8 key codes [P, page, dI] with scales [P, page]; bf16 latent KV
    [P, page, D].  Slots past each sequence's length in its last page are
    poisoned (NaN code 0x7F, NaN scale, NaN bf16) so any read of them shows.
    Queries: one token per sequence at position ctx-1.
    """
    seed = cfg.seed if seed is None else seed
    ctx, bt, P = decode_layout(cfg, seed, B, ctx_lo, ctx_hi, ctx)
    B = ctx.shape[0]
    ps = cfg.page_size
    kI = randn((P * ps, cfg.dI), device, seed, 12)
    k8, ks = quantize_fp8_per_token(kI)
    del kI
    k8 = k8.view(P, ps, cfg.dI)
    ks = ks.view(P, ps)
    kv = randn((P * ps, cfg.D), device, seed, 21, dtype=torch.bfloat16).view(P, ps, cfg.D)
    if poison:
        for b in range(B):
            c = int(ctx[b])
            tail = c % ps
            if tail:
                page = int(bt[b, (c - 1) // ps])
                k8[page, tail:] = 0x7F
                ks[page, tail:] = float("nan")
                kv[page, tail:] = float("nan")
    q8, qs, w = indexer_queries(cfg, B, device, seed)
    q = randn((B, cfg.H, cfg.D), device, seed, 20, dtype=torch.bfloat16)
    return dict(q8=q8, qs=qs, w=w, k8_pool=k8, ks_pool=ks, kv_pool=kv, q=q,
                ctx=ctx.to(device), q_pos=(ctx - 1).to(device), block_table=bt.to(device),
                num_pages=P)


def varlen_inputs(cfg: Config, device, seq_lens, queries_per_seq=None, seed: int | None = None):
    """Several sequences of different lengths over one shared, permuted page pool.

    Sequence b holds ``seq_lens[b]`` tokens; its query rows are the last
    ``queries_per_seq[b]`` positions (all of them when None: a ragged batched
    prefill; a few: a multi-token decode).  Every query row carries its own
    position, context length (position + 1) and copy of its sequence's block
    table, which is how the paged entry points see a row.  Also returns the
    same latent rows concatenated per sequence (``kv_concat`` with per-sequence
    start offsets) for the contiguous entry point.
    """
    seed = cfg.seed if seed is None else seed
    lens = torch.as_tensor(seq_lens, dtype=torch.int32)
    d = decode_inputs(cfg, device, seed=seed, ctx=lens)
    ps = cfg.page_size
    bt = d["block_table"].cpu()
    seq, pos = [], []
    for b, n in enumerate(lens.tolist()):
        m = n if queries_per_seq is None else int(queries_per_seq[b])
        for p in range(n - m, n):
            seq.append(b)
            pos.append(p)
    seq = torch.tensor(seq, dtype=torch.int64)
    pos = torch.tensor(pos, dtype=torch.int32)
    T = int(seq.numel())
    q8, qs, w = indexer_queries(cfg, T, device, seed, tid0=40)
    q = randn((T, cfg.H, cfg.D), device, seed, 42, dtype=torch.bfloat16)
    starts = torch.zeros(len(lens), dtype=torch.int64)
    starts[1:] = torch.cumsum(lens.to(torch.int64), 0)[:-1]
    rows = torch.cat([(bt[b, torch.arange(n) // ps].to(torch.int64) * ps + torch.arange(n) % ps)
                      for b, n in enumerate(lens.tolist())])
    kv_concat = d["kv_pool"].view(-1, cfg.D)[rows.to(device)].contiguous()
    return dict(q8=q8, qs=qs, w=w, q=q, k8_pool=d["k8_pool"], ks_pool=d["ks_pool"], kv_pool=d["kv_pool"],
                num_pages=d["num_pages"], seq=seq, q_pos=pos.to(device), ctx=(pos + 1).to(device),
                block_table=bt[seq].contiguous().to(device), seq_block_table=bt, seq_lens=lens,
                seq_starts=starts, kv_concat=kv_concat)
