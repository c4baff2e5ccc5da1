#!/usr/bin/env python3
"""Benchmark of the DSA hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over the L = 32768 causal prefill
workload: lightning indexer (FP8) -> top-k (k = 2048) -> sparse MQA-mode MLA
(128 heads, 576/512 bf16), all through libdsa's C ABI with inputs already in
HBM.  A paged decode step (64 sequences, contexts 8K..64K) is timed the same
way and reported under "decode".  L2 is flushed (256 MB write) before every
timed step, outside the timed events.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle on
a bounded row sample of the same workload instead (rank 0 only).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {dsa,reference}]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import dsa_workloads as W  # noqa: E402

METRIC = "DSA tokens/s at L=32K,k=2048 (prefill) and decode; % of FP8/BF16/HBM roofline"
WORKLOAD = "prefill_32k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s): the derived FP8 peak, a side column
OTHER_WORKLOADS = ("tiny", "prefill_4k", "chunked_128k")
NOMINAL = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0, "fp8_tflops": 4500.0}  # GB300 datasheet, dense
PROFILES = os.path.join(ROOT, "profiles")


# ------------------------------------------------------------------ helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def prefill_work(L: int, k: int, HI: int, dI: int, H: int, D: int = 576, Dv: int = 512):
    """Algorithmic work of one prefill pass (the method's own, not the dense work it avoids)."""
    t1 = np.arange(1, L + 1, dtype=np.float64)          # candidates per row (t + 1)
    sel = np.minimum(t1, k)                              # selected rows per query
    idx_flop = 2.0 * HI * dI * t1.sum()
    idx_bytes = L * HI * dI + L * (4 + 4 * HI) + L * dI + 4 * L + 4 * t1.sum()  # q8, scales+w, k8, ks, logits
    big = t1 > k
    topk_bytes = 4 * t1[big].sum() + 4 * L + 4 * L * k   # logits read (rows that need selection), valid_len, idx
    mla_flop = 2.0 * H * (D + Dv) * sel.sum()
    mla_bytes = 2 * L * H * D + 2 * L * D + 4 * L * k + 2 * L * H * Dv + 4 * L * H
    return dict(indexer_flop=idx_flop, indexer_bytes=idx_bytes, topk_bytes=topk_bytes, mla_flop=mla_flop,
                mla_bytes=mla_bytes, selected_pairs=sel.sum(), key_rows=t1.sum())


def workload_desc(cfg: W.Config) -> str:
    """One string per workload, the same in both arms of the bench."""
    if cfg.chunk:
        return (f"{cfg.name}: batch 1, L={cfg.L} causal in {cfg.L // cfg.chunk} chunks of {cfg.chunk} query rows, each "
                f"over its whole prefix, k={cfg.k}, indexer H_I={cfg.HI} d_I={cfg.dI} FP8 E4M3 per-token scales, "
                f"MLA H={cfg.H} D={cfg.D} Dv={cfg.Dv} bf16, inputs N(0,1)")
    return (f"{cfg.name}: batch 1, L={cfg.L} causal, k={cfg.k}, indexer H_I={cfg.HI} d_I={cfg.dI} FP8 E4M3 per-token "
            f"scales, MLA H={cfg.H} D={cfg.D} Dv={cfg.Dv} bf16, inputs N(0,1)")


def clock_adjusted(burst: float, clk: dict, what: str):
    """The peak a kernel timed inside this run can reach: the burst figure when the run's
    clock record shows the SM clock held at its maximum with no throttle reason, else
    the burst figure scaled by median / max SM clock.  Returns (peak, how)."""
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    reasons = [r for r in clk.get("reasons", []) if r != "nvidia-smi unavailable"]
    if sm and mx and sm >= 0.97 * mx and not reasons:
        return burst, f"{what} burst (SM clock median {sm:.0f} of max {mx:.0f} MHz, no throttle reason)"
    if sm and mx:
        return burst * sm / mx, (f"{what} burst x median/max SM clock ({sm:.0f}/{mx:.0f} MHz; "
                                 f"reasons {reasons or 'none'})")
    return burst, f"{what} burst (no clock record)"


def measure_matmul_peaks(dev, n: int = 8192, reps: int = 10):
    """Dense GEMM throughput on this GPU, best of `reps` single n^3 products (burst):
    bf16 through torch.matmul and FP8 E4M3 (fp32 accumulate, bf16 out) through
    torch._scaled_mm, the library routes to the tensor cores.  FP8 is None if the
    routine is unavailable here."""
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn((n, n), generator=g, device=dev).to(torch.bfloat16)
    b = torch.randn((n, n), generator=g, device=dev).to(torch.bfloat16)

    def best(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return 2.0 * n ** 3 / (min(ts) / 1e3) / 1e12

    out = {"n": n, "bf16_tflops": best(lambda: torch.matmul(a, b)), "fp8_tflops": None}
    try:
        a8, b8 = a.to(torch.float8_e4m3fn), b.to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=dev)
        out["fp8_tflops"] = best(lambda: torch._scaled_mm(a8, b8.t(), scale_a=one, scale_b=one,
                                                          out_dtype=torch.bfloat16))
    except Exception as e:  # noqa: BLE001
        out["fp8_error"] = f"{type(e).__name__}: {e}"[:200]
    out["how"] = (f"best of {reps} single {n}^3 products after 3 warm-ups, CUDA events: torch.matmul bf16, "
                  "torch._scaled_mm E4M3 x E4M3 (per-tensor scales, bf16 out)")
    return out


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.out = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            self.sel = None

    def start(self):
        try:
            import tempfile

            self.out = tempfile.TemporaryFile(mode="w+")
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.sel:
                cmd += ["-i", self.sel]
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_digest(*names):
    h = hashlib.sha1()
    for n in names:
        with open(os.path.join(ROOT, "sparse_attention_02_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str, sources):
    """DRAM bytes per launch from a committed ncu summary, if the kernel is unchanged since."""
    p = os.path.join(PROFILES, f"{name}.traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_digest") != source_digest(*sources):
        return None
    return d.get("dram_bytes_per_launch")


def aggregate_over_ranks(ms_local: float, tokens_local: int, dist=None, device=None):
    """Whole-job timing: the slowest rank's ms per step and all ranks' tokens per second."""
    ms = float(ms_local)
    world = 1
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_local / (ms / 1e3)


# ------------------------------------------------------------ CPU baseline

def oracle_sample(cfg: W.Config, rows: np.ndarray, x):
    """Time the fp64 oracle on `rows` of the prefill workload `x`; returns per-unit rates.

    The needed rows of the same inputs are copied to the host first (not timed).
    Units: indexer key-rows, top-k candidates, attention selected pairs.
    """
    import oracle

    n = int(rows.max()) + 1
    pos = x["q_pos"].cpu().numpy()  # positions of x's query rows (all L, or a subset)
    at = np.searchsorted(pos, rows)
    assert np.array_equal(pos[at], rows), "sampled rows missing from the inputs"
    r = torch.as_tensor(at, device=x["q"].device)
    h = {"q8": x["q8"][r].cpu(), "qs": x["qs"][r].cpu(), "w": x["w"][r].cpu(), "q": x["q"][r].cpu(),
         "k8": x["k8"][:n].cpu(), "ks": x["ks"][:n].cpu(), "kv": x["kv"][:n].cpu()}
    rows = np.asarray(rows)
    t0 = time.perf_counter()
    logits = oracle.indexer(h["q8"].numpy(), h["qs"].numpy(), h["w"].numpy(), rows,
                            h["k8"].numpy(), h["ks"].numpy(), ld=n, fill=-np.inf)
    t1 = time.perf_counter()
    idx = oracle.topk(logits, rows + 1, cfg.k)
    t2 = time.perf_counter()
    qb = h["q"].view(torch.int16).numpy().view(np.uint16)
    kvb = h["kv"].view(torch.int16).numpy().view(np.uint16)
    oracle.sparse_mla(qb, kvb, idx, cfg.sm_scale)
    t3 = time.perf_counter()
    key_rows = float((rows + 1).sum())
    pairs = float(np.minimum(rows + 1, cfg.k).sum())
    return dict(indexer_s_per_unit=(t1 - t0) / key_rows, topk_s_per_unit=(t2 - t1) / key_rows,
                mla_s_per_unit=(t3 - t2) / pairs, wall_s=t3 - t0, cores=oracle.num_threads(),
                rows=len(rows))


def oracle_full_estimate(rates, L, k):
    t1 = np.arange(1, L + 1, dtype=np.float64)
    return (rates["indexer_s_per_unit"] * t1.sum() + rates["topk_s_per_unit"] * t1.sum()
            + rates["mla_s_per_unit"] * np.minimum(t1, k).sum())


def cpu_baseline(cfg, x, rows=None):
    L = cfg.L
    if rows is None:
        # ~10-15 s of fp64 work on 16 cores: fixed rows around the k boundary and both
        # ends, plus rows drawn uniformly over the whole prefill
        rng = np.random.default_rng(7)
        fixed = [r for r in (0, 1, 255, 1023, 2047, 2048, 3071, 4095, L // 2 - 1, L - 1) if r < L]
        rows = np.unique(np.concatenate([fixed, rng.integers(0, L, 126)]))
    rates = oracle_sample(cfg, np.asarray(rows), x)
    est = oracle_full_estimate(rates, L, cfg.k)
    return {"value": L / est, "unit": "tokens/s", "cores": rates["cores"], "kind": "oracle",
            "sample": (f"{rates['rows']} query rows of the L={L} prefill (ten fixed positions, the rest uniform "
                       f"over [0, {L}); all of their keys and selections), {rates['wall_s']:.1f} s of CPU work; "
                       f"per-unit rates extrapolated to all {L} rows (indexer and top-k per key-row, attention "
                       f"per selected pair)"),
            "extrapolated_seconds_per_step": est}


def run_reference(args, rank, world):
    """--impl reference: the oracle on bounded row samples, rank 0 only."""
    if rank != 0:
        return
    cfg = W.CONFIGS[args.workload]
    L = cfg.L
    rng = np.random.default_rng(11)
    # a pool of query rows spread over the whole prefill: every row of eight of the
    # input generator's query chunks, evenly spaced (the keys are drawn in full)
    per = max(1, W._CHUNK_ELEMS // (cfg.H * cfg.D))
    nchunk = (L + per - 1) // per
    chunks = np.unique(np.linspace(0, nchunk - 1, min(8, nchunk)).round().astype(np.int64))
    pool = np.concatenate([np.arange(c * per, min(L, (c + 1) * per)) for c in chunks])
    x = W.prefill_rows(cfg, "cpu", pool)

    def step(i):
        rows = np.sort(rng.choice(pool, size=min(48, len(pool)), replace=False))
        return oracle_sample(cfg, rows, x)

    for i in range(args.warmup):
        step(i)
    ests, walls = [], []
    cores = None
    for i in range(args.steps):
        r = step(i)
        ests.append(oracle_full_estimate(r, L, cfg.k))
        walls.append(r["wall_s"])
        cores = r["cores"]
    est = statistics.median(ests)
    value = L / est
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": est * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_desc(cfg), "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: 48 distinct query rows drawn from {len(pool)} rows spread over all {L} "
                                       f"positions (all keys and selections), timed on the host cores; "
                                       f"per-unit rates extrapolated to the full {L}-row prefill (indexer and top-k "
                                       f"per key-row, attention per selected pair); median over {args.steps} steps "
                                       f"({statistics.mean(walls):.2f} s CPU wall per step). value and ms_per_step "
                                       f"are that extrapolation: a whole step is never run, so ms_per_step "
                                       f"({est:.0f} s) is far longer than this run's own wall time"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- GPU timing

def prefill_step(dsa, x, b, cfg):
    dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], b["logits"])
    dsa.dsa_topk(b["logits"], b["valid_len"], cfg.k, b["idx"])
    dsa.dsa_sparse_mla_prefill(x["q"], x["kv"], b["idx"], cfg.sm_scale, b["out"], b["lse"])


def time_prefill(dsa, x, b, cfg, steps, warmup, flush):
    """Whole steps (events only at step boundaries, so each kernel's launch can
    overlap the previous kernel's tail), then the same number of steps with an
    event between stages for the per-stage split.  Returns (step ms [steps],
    stage ms [steps, 3])."""
    for _ in range(warmup):
        prefill_step(dsa, x, b, cfg)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for s in range(steps):
        flush.zero_()
        ev[s][0].record()
        prefill_step(dsa, x, b, cfg)
        ev[s][1].record()
    torch.cuda.synchronize()
    step_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for s in range(steps):
        flush.zero_()
        e = ev[s]
        e[0].record()
        dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], b["logits"])
        e[1].record()
        dsa.dsa_topk(b["logits"], b["valid_len"], cfg.k, b["idx"])
        e[2].record()
        dsa.dsa_sparse_mla_prefill(x["q"], x["kv"], b["idx"], cfg.sm_scale, b["out"], b["lse"])
        e[3].record()
    torch.cuda.synchronize()
    st = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev])  # ms
    return step_ms, st


def stage_records(work, stage_ms, L, pk):
    """Per-stage ms, throughput and roofline fractions of one prefill pass.  `pk` holds the
    peaks this run's kernels are held to (see `run_peaks`)."""
    idx_tflops = work["indexer_flop"] / (stage_ms[0] / 1e3) / 1e12
    topk_gbs = work["topk_bytes"] / (stage_ms[1] / 1e3) / 1e9
    mla_tflops = work["mla_flop"] / (stage_ms[2] / 1e3) / 1e12
    return {
        "indexer": {"ms": float(stage_ms[0]), "tflops": idx_tflops, "bound": "tensor (fp8)",
                    "peak": pk["fp8"], "frac": idx_tflops / pk["fp8"], "peak_source": pk["fp8_how"],
                    "frac_derived_fp8": idx_tflops / pk["fp8_derived"],
                    "frac_nominal": idx_tflops / NOMINAL["fp8_tflops"],
                    "flop": work["indexer_flop"], "tokens_per_s": L / (stage_ms[0] / 1e3)},
        "topk": {"ms": float(stage_ms[1]), "gbs": topk_gbs, "bound": "hbm", "peak": pk["hbm"],
                 "frac": topk_gbs / pk["hbm"], "frac_nominal": topk_gbs / NOMINAL["hbm_gbs"],
                 "bytes": work["topk_bytes"], "tokens_per_s": L / (stage_ms[1] / 1e3)},
        "sparse_mla": {"ms": float(stage_ms[2]), "tflops": mla_tflops, "bound": "tensor (bf16)",
                       "peak": pk["bf16"], "frac": mla_tflops / pk["bf16"], "peak_source": pk["bf16_how"],
                       "frac_sustained": mla_tflops / pk["bf16_sustained"],
                       "frac_nominal": mla_tflops / NOMINAL["bf16_tflops"], "flop": work["mla_flop"],
                       "tokens_per_s": L / (stage_ms[2] / 1e3)},
    }


def run_peaks(peaks, peaks_src, clk, mm):
    """The denominators for one timed region: BF16 from the peaks file's burst figure and
    FP8 from this process's own measured burst figure (the derived 2 x BF16 when the
    measurement failed), each taken at the clock the region ran at (`clock_adjusted`)."""
    bf16, bf16_how = clock_adjusted(peaks["bf16_tflops"], clk, f"{peaks_src} bf16")
    fp8_derived = FP8_OVER_BF16 * bf16
    if mm and mm.get("fp8_tflops"):
        fp8, fp8_how = clock_adjusted(mm["fp8_tflops"], clk, "measured fp8 (torch._scaled_mm 8192^3 in this run)")
    else:
        fp8, fp8_how = fp8_derived, f"derived: {FP8_OVER_BF16} x ({bf16_how}); the FP8 measurement failed"
    return {"bf16": bf16, "bf16_how": bf16_how, "fp8": fp8, "fp8_how": fp8_how, "fp8_derived": fp8_derived,
            "bf16_sustained": peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]), "hbm": peaks["hbm_gbs"]}


def prefill_buffers(cfg, x, dev, rows=None):
    rows = cfg.L if rows is None else rows
    return {"logits": torch.empty((rows, cfg.L), dtype=torch.float32, device=dev),
            "valid_len": x["q_pos"] + 1,
            "idx": torch.empty((rows, cfg.k), dtype=torch.int32, device=dev),
            "out": torch.empty((cfg.L, cfg.H, cfg.Dv), dtype=torch.bfloat16, device=dev),
            "lse": torch.empty((cfg.L, cfg.H), dtype=torch.float32, device=dev)}


def chunked_stage_calls(dsa, x, b, cfg):
    """The three stages of each chunk of a chunked prefill, as (stage, thunk) pairs in
    launch order: chunk c holds query rows [C c, C (c + 1)) over keys [0, C (c + 1))."""
    C = cfg.chunk
    calls = []
    for c in range(cfg.L // C):
        r0, r1 = c * C, (c + 1) * C
        calls.append((0, lambda r0=r0, r1=r1: dsa.dsa_indexer_logits(
            x["q8"][r0:r1], x["qs"][r0:r1], x["w"][r0:r1], x["k8"][:r1], x["ks"][:r1], x["q_pos"][r0:r1],
            b["logits"])))
        calls.append((1, lambda r0=r0, r1=r1: dsa.dsa_topk(b["logits"], b["valid_len"][r0:r1], cfg.k, b["idx"])))
        calls.append((2, lambda r0=r0, r1=r1: dsa.dsa_sparse_mla_prefill(
            x["q"][r0:r1], x["kv"][:r1], b["idx"], cfg.sm_scale, b["out"][r0:r1], b["lse"][r0:r1])))
    return calls


def time_calls(calls, steps, warmup, flush):
    """Whole steps of `calls` (events only at step boundaries), then the same steps with an
    event around every call, summed per stage.  Returns (step ms [steps], stage ms [3])."""
    for _ in range(warmup):
        for _, f in calls:
            f()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in ev:
        flush.zero_()
        e[0].record()
        for _, f in calls:
            f()
        e[1].record()
    torch.cuda.synchronize()
    step_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])
    per = np.zeros((steps, 3))
    for s in range(steps):
        flush.zero_()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        es[0].record()
        for i, (_, f) in enumerate(calls):
            f()
            es[i + 1].record()
        torch.cuda.synchronize()
        for i, (st, _) in enumerate(calls):
            per[s, st] += es[i].elapsed_time(es[i + 1])
    return step_ms, per.mean(0)


def fused_bench(dsa, x, b, cfg, steps, warmup, flush, dev, two_call_stages, chunk_rows=None):
    """The same prefill with the indexer and top-k fused (dsa_indexer_topk: no index scores
    in memory) in place of the two calls; the attention stage is unchanged.  The indices of
    the last chunk (or the whole prefill) are compared byte for byte with the two-call path's."""
    L, C = cfg.L, chunk_rows or cfg.L
    ws = torch.empty(dsa.dsa_indexer_topk_workspace_size(C, L, cfg.HI, cfg.dI, cfg.k), dtype=torch.uint8, device=dev)
    idx_f = torch.empty_like(b["idx"])
    calls = []
    for c in range(L // C):
        r0, r1 = c * C, (c + 1) * C
        calls.append((0, lambda r0=r0, r1=r1: dsa.dsa_indexer_topk(
            x["q8"][r0:r1], x["qs"][r0:r1], x["w"][r0:r1], x["k8"][:r1], x["ks"][:r1], x["q_pos"][r0:r1], cfg.k,
            idx_f, workspace=ws)))
        calls.append((2, lambda r0=r0, r1=r1: dsa.dsa_sparse_mla_prefill(
            x["q"][r0:r1], x["kv"][:r1], idx_f, cfg.sm_scale, b["out"][r0:r1], b["lse"][r0:r1])))
    step_ms, stage_ms = time_calls(calls, steps, warmup, flush)
    # b["idx"] holds the two-call path's indices of the same (last) chunk
    same = bool(torch.equal(idx_f, b["idx"]))
    two = two_call_stages["indexer"]["ms"] + two_call_stages["topk"]["ms"]
    ms = float(step_ms.mean())
    del ws
    return {"ms_per_step": ms, "tokens_per_s": L / (ms / 1e3), "indexer_topk_ms": float(stage_ms[0]),
            "sparse_mla_ms": float(stage_ms[2]), "two_call_indexer_plus_topk_ms": two,
            "saved_ms": two - float(stage_ms[0]), "indices_match_two_call_path": same,
            "launches_per_step": 8 * (L // C),
            "what": "dsa_indexer_topk (sampled threshold, candidate-mode indexer, exact select; no scores "
                    "written) then sparse MLA, per chunk"}


def warmup_bench(dsa, steps, warmup, flush, peaks, peaks_src, mm, dev, name="prefill_4k"):
    """The indexer's warm-up step (dsa_indexer_warmup: target, loss, gradients) on the L = 4096
    prefill shapes.  Work counted once per step: the target's QK^T (one pass; the kernel takes
    two, one for the per-head LSE and one for the probabilities), the FP8 index scores, and the
    backward's three contractions (a, then dq and dk), 2 x H_I x d_I FLOP per (row, key) each; all
    of it on tensor cores (the backward in BF16: codes exact, coefficients as bf16 hi + lo pairs)."""
    cfg = W.CONFIGS[name]
    L = cfg.L
    x = W.prefill_inputs(cfg, dev)
    loss = torch.empty((L,), device=dev)
    dw = torch.empty((L, cfg.HI), device=dev)
    dq = torch.empty((L, cfg.HI, cfg.dI), device=dev)
    dk = torch.empty((L, cfg.dI), device=dev)
    ws = torch.empty(dsa.dsa_indexer_warmup_workspace_size(L, L, cfg.HI, cfg.dI), dtype=torch.uint8, device=dev)

    def call():
        dsa.dsa_indexer_warmup(x["q"], x["kv"], cfg.sm_scale, x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"],
                               loss, dw, dq, dk, workspace=ws)

    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    step_ms, _ = time_calls([(0, call)], steps, warmup, flush)
    clk = clocks.stop()
    pk = run_peaks(peaks, peaks_src, clk, mm)
    pairs = L * (L + 1) / 2
    f_target = 2.0 * cfg.H * cfg.D * pairs
    f_index = 2.0 * cfg.HI * cfg.dI * pairs
    f_bwd = 3 * 2.0 * cfg.HI * cfg.dI * pairs
    ms = float(step_ms.mean())
    total = f_target + f_index + f_bwd
    lower_ms = (f_target / (pk["bf16"] * 1e12) + f_index / (pk["fp8"] * 1e12) + f_bwd / (pk["bf16"] * 1e12)) * 1e3
    finite = bool(torch.isfinite(loss).all() and torch.isfinite(dq).all() and torch.isfinite(dk).all())
    del ws, x
    torch.cuda.empty_cache()
    return {"workload": f"{name}: L={L} causal, H={cfg.H} D={cfg.D} bf16 target, indexer H_I={cfg.HI} d_I={cfg.dI} FP8",
            "ms_per_step": ms, "tokens_per_s": L / (ms / 1e3), "steps": steps,
            "flop": {"target_qk": f_target, "indexer": f_index, "backward": f_bwd},
            "achieved_tflops": total / (ms / 1e3) / 1e12,
            "roofline_ms": lower_ms, "frac": lower_ms / ms,
            "bound": "target and backward on BF16 tensor cores, index scores on FP8",
            "peak_source": {"bf16": pk["bf16_how"], "fp8": pk["fp8_how"]},
            "outputs_finite": finite, "clocks": clk}


def workload_bench(dsa, name, steps, warmup, flush, peaks, peaks_src, mm, dev):
    """One more configured prefill workload (tiny, L = 4096, or the chunked L = 131072):
    per-stage ms, tokens/s and roofline fractions, clocks sampled over its own timed region."""
    cfg = W.CONFIGS[name]
    L = cfg.L
    x = W.prefill_inputs(cfg, dev)
    b = prefill_buffers(cfg, x, dev, rows=cfg.chunk or None)
    if cfg.chunk:
        calls = chunked_stage_calls(dsa, x, b, cfg)
    else:
        calls = [(0, lambda: dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"],
                                                    b["logits"])),
                 (1, lambda: dsa.dsa_topk(b["logits"], b["valid_len"], cfg.k, b["idx"])),
                 (2, lambda: dsa.dsa_sparse_mla_prefill(x["q"], x["kv"], b["idx"], cfg.sm_scale, b["out"],
                                                        b["lse"]))]
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    step_ms, stage_ms = time_calls(calls, steps, warmup, flush)
    clk = clocks.stop()
    pk = run_peaks(peaks, peaks_src, clk, mm)
    work = prefill_work(L, cfg.k, cfg.HI, cfg.dI, cfg.H)
    ms = float(step_ms.mean())
    rec = {"workload": workload_desc(cfg), "ms_per_step": ms, "tokens_per_s": L / (ms / 1e3),
           "steps": steps, "warmup": warmup, "launches_per_step": len(calls),
           "stages": stage_records(work, stage_ms, L, pk), "clocks": clk,
           "l2": "flushed before every timed step (256 MB write, outside the timed events)"}
    if cfg.chunk:
        # the logits each chunk's indexer writes and its top-k reads back (causal part only)
        rec["logits_bytes_write_read"] = 8.0 * work["key_rows"]
        rec["logits_hbm_ms_at_peak"] = rec["logits_bytes_write_read"] / (pk["hbm"] * 1e9) * 1e3
        rec["fused"] = fused_bench(dsa, x, b, cfg, steps, warmup, flush, dev, rec["stages"], chunk_rows=cfg.chunk)
    del x, b, calls
    torch.cuda.empty_cache()
    return rec


def quantize_bench(dsa, cfg, steps, warmup, flush, hbm, dev):
    """Per-token FP8 quantisation of the indexer inputs (q^I [L, H_I, d_I], k^I [L, d_I] fp32), timed on
    its own: the headline step starts from FP8 codes, as the workload defines it."""
    L = cfg.L
    xq = W.randn((L, cfg.HI, cfg.dI), dev, cfg.seed, 10)
    xk = W.randn((L, cfg.dI), dev, cfg.seed, 12)
    cq = torch.empty(xq.shape, dtype=torch.uint8, device=dev)
    ck = torch.empty(xk.shape, dtype=torch.uint8, device=dev)
    sq = torch.empty((L,), dtype=torch.float32, device=dev)
    sk = torch.empty((L,), dtype=torch.float32, device=dev)
    for _ in range(warmup):
        dsa.dsa_quantize_fp8(xq, cq, sq)
        dsa.dsa_quantize_fp8(xk, ck, sk)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in ev:
        flush.zero_()
        e[0].record()
        dsa.dsa_quantize_fp8(xq, cq, sq)
        dsa.dsa_quantize_fp8(xk, ck, sk)
        e[1].record()
    torch.cuda.synchronize()
    ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    nbytes = 5.0 * (xq.numel() + xk.numel()) + 8.0 * L
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"ms": ms, "gbs": gbs, "bound": "hbm", "peak": hbm, "frac": gbs / hbm,
            "frac_nominal": gbs / NOMINAL["hbm_gbs"], "bytes": nbytes,
            "in_step": False, "mode": "amax/448",
            "what": f"q^I [{L},{cfg.HI},{cfg.dI}] and k^I [{L},{cfg.dI}] fp32 -> E4M3 codes + per-token scales"}


def decode_bench(dsa, steps, warmup, flush, peaks, dev):
    cfg = W.CONFIGS["decode_paged"]
    d = W.decode_inputs(cfg, dev)
    B = int(d["ctx"].shape[0])
    ctx = d["ctx"].cpu().numpy().astype(np.int64)
    ld = int(ctx.max())
    logits = torch.empty((B, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((B, cfg.k), dtype=torch.int32, device=dev)
    out = torch.empty((B, cfg.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, cfg.H), dtype=torch.float32, device=dev)
    ws_n = dsa.dsa_sparse_mla_decode_workspace_size(B, cfg.H, cfg.k)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev) if ws_n else None

    def step():
        dsa.dsa_indexer_logits(d["q8"], d["qs"], d["w"], d["k8_pool"], d["ks_pool"], d["q_pos"], logits,
                               block_table=d["block_table"])
        dsa.dsa_topk(logits, d["ctx"], cfg.k, idx)
        dsa.dsa_sparse_mla_decode_paged(d["q"], d["kv_pool"], d["block_table"], d["ctx"], idx, cfg.sm_scale,
                                        out, lse, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in evs:
        flush.zero_()
        e[0].record()
        step()
        e[1].record()
    torch.cuda.synchronize()
    step_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for s in range(steps):
        flush.zero_()
        e = ev[s]
        e[0].record()
        dsa.dsa_indexer_logits(d["q8"], d["qs"], d["w"], d["k8_pool"], d["ks_pool"], d["q_pos"], logits,
                               block_table=d["block_table"])
        e[1].record()
        dsa.dsa_topk(logits, d["ctx"], cfg.k, idx)
        e[2].record()
        dsa.dsa_sparse_mla_decode_paged(d["q"], d["kv_pool"], d["block_table"], d["ctx"], idx, cfg.sm_scale,
                                        out, lse, workspace=ws)
        e[3].record()
    torch.cuda.synchronize()
    st = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev]).mean(0)
    sel = np.minimum(ctx, cfg.k).sum()
    key_bytes = ctx.sum() * (cfg.dI + 4)                         # FP8 key codes + per-key scale
    logit_bytes = ctx.sum() * 4 * 2                               # written by the indexer, read by top-k
    attn_bytes = sel * 1152 + B * cfg.H * (576 + 512) * 2 + B * cfg.k * 4 * 2
    q_bytes = B * (cfg.HI * cfg.dI + cfg.HI * 4 + 8)
    total = key_bytes + logit_bytes + attn_bytes + q_bytes
    ms = step_ms
    hbm = peaks["hbm_gbs"]
    return {"workload": f"decode_paged: B={B}, ctx U[{cfg.ctx_lo},{cfg.ctx_hi}] (sum {int(ctx.sum())}), page 64, "
                        f"k={cfg.k}, H_I={cfg.HI}, H={cfg.H}",
            "tokens_per_s": B / (ms / 1e3), "ms_per_step": ms,
            "stage_ms": {"indexer": float(st[0]), "topk": float(st[1]), "sparse_mla": float(st[2])},
            "stage_ms_note": "second pass with an event between stages (no launch overlap); ms_per_step is "
                             "timed over whole steps",
            "algorithmic_bytes": float(total),
            "hbm": {"achieved_gbs": total / (ms / 1e3) / 1e9, "peak_gbs": hbm,
                    "frac": total / (ms / 1e3) / 1e9 / hbm,
                    "frac_nominal": total / (ms / 1e3) / 1e9 / NOMINAL["hbm_gbs"]},
            "stage_hbm_frac": {"indexer": (key_bytes + ctx.sum() * 4 + q_bytes) / (st[0] / 1e3) / 1e9 / hbm,
                               "topk": (ctx.sum() * 4 + B * cfg.k * 4) / (st[1] / 1e3) / 1e9 / hbm,
                               "sparse_mla": attn_bytes / (st[2] / 1e3) / 1e9 / hbm}}


def e2e_timeline(dsa, step, steps, max_chunks_per_call=64):
    """After the timed steps, the same number of steps again with dsa_prefill_host's per-chunk
    timeline on (outside the timed region): per call, its span from the first input copy to the
    last output copy, the time its three streams were busy, and how long the stages' stream sat
    waiting between chunks (for copies).  A slow step shows up on the stream whose time grew."""
    cap = steps * max_chunks_per_call
    dsa.dsa_prefill_host_trace(cap)
    try:
        for _ in range(steps):
            step()
        torch.cuda.synchronize()
        t, call, rows = dsa.dsa_prefill_host_trace_read(cap)
    finally:
        dsa.dsa_prefill_host_trace(0)
    out = {"span_ms": [], "h2d_busy_ms": [], "stages_busy_ms": [], "stages_wait_ms": [], "d2h_busy_ms": [],
           "chunks_per_call": 0}
    for c in range(steps):
        m = t[call == c].astype(np.float64)
        if not len(m):
            continue
        out["chunks_per_call"] = int(len(m))
        busy = lambda a, b: float(np.sum(m[:, b] - m[:, a]))
        stages = busy(2, 3)
        out["span_ms"].append(round(float(m[:, 5].max() - m[:, 0].min()), 3))
        out["h2d_busy_ms"].append(round(busy(0, 1), 3))
        out["stages_busy_ms"].append(round(stages, 3))
        out["stages_wait_ms"].append(round(float(m[:, 3].max() - m[:, 2].min()) - stages, 3))
        out["d2h_busy_ms"].append(round(busy(4, 5), 3))
    return out


def e2e_bench(dsa, x, b, cfg, steps, dev, chunk_rows=2048):
    """The same step through the public C ABI on pinned HOST buffers: dsa_prefill_host copies the
    inputs in, runs the three stages chunk by chunk (copies of one chunk overlap the kernels of
    the next) and copies out and lse back; every copy is inside the timed region.  The value is
    the mean over the steps; each step's time and the median are reported beside it (a single
    step of a run has been seen to take several times the others)."""
    names = ["q8", "qs", "w", "q_pos", "q", "k8", "ks", "kv"]
    host = {n: torch.empty(x[n].shape, dtype=x[n].dtype, pin_memory=True) for n in names}
    for n in names:
        host[n].copy_(x[n])
    out_h = torch.empty(b["out"].shape, dtype=b["out"].dtype, pin_memory=True)
    lse_h = torch.empty(b["lse"].shape, dtype=b["lse"].dtype, pin_memory=True)
    L = cfg.L
    need = dsa.dsa_prefill_host_workspace_size(L, L, cfg.HI, cfg.dI, cfg.H, cfg.k, chunk_rows)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

    def step():
        dsa.dsa_prefill_host(host["q8"], host["qs"], host["w"], host["q_pos"], host["k8"], host["ks"], host["q"],
                             host["kv"], cfg.sm_scale, cfg.k, out_h, lse_h, chunk_rows=chunk_rows, workspace=ws)

    step()
    torch.cuda.synchronize()
    # back to back, with an event between steps (each call already waits for the
    # previous one on the stream, so the events add no serialisation)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        step()
        ev[i + 1].record()
    torch.cuda.synchronize()
    each = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    ms = ev[0].elapsed_time(ev[steps]) / steps
    trace = e2e_timeline(dsa, step, steps)
    # the host outputs are the device path's outputs (same kernels, same rows)
    same = bool(torch.equal(out_h.view(torch.int16), b["out"].cpu().view(torch.int16)))
    del ws, host
    return {"value": cfg.L / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms, "ms_each_step": [round(x, 3) for x in each],
            "median_ms_per_step": float(np.median(each)),
            "timeline": trace,
            "api": "dsa_prefill_host",
            "chunk_rows": chunk_rows, "matches_device_path": same}


def case_setup(dsa, name, dev):
    """One entry point on a small input, for narrow profiler captures of its kernels: returns
    (description, call).  Inputs are built once; the call does only the entry point's work."""
    if name in ("indexer_4k", "topk_4k", "mla_4k", "warmup_4k"):
        cfg = W.CONFIGS["prefill_4k"]
        L = cfg.L
        x = W.prefill_inputs(cfg, dev)
        logits = torch.empty((L, L), dtype=torch.float32, device=dev)
        vlen = x["q_pos"] + 1
        idx = torch.empty((L, cfg.k), dtype=torch.int32, device=dev)
        if name == "indexer_4k":
            return (f"dsa_indexer_logits, L={L} causal, H_I={cfg.HI}, d_I={cfg.dI}",
                    lambda: dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], logits))
        dsa.dsa_indexer_logits(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], logits)
        if name == "topk_4k":
            return f"dsa_topk, {L} rows of the causal L={L} scores, k={cfg.k}", lambda: dsa.dsa_topk(logits, vlen, cfg.k, idx)
        if name == "mla_4k":
            dsa.dsa_topk(logits, vlen, cfg.k, idx)
            out = torch.empty((L, cfg.H, cfg.Dv), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((L, cfg.H), dtype=torch.float32, device=dev)
            return (f"dsa_sparse_mla_prefill, L={L}, k={cfg.k}, H={cfg.H}",
                    lambda: dsa.dsa_sparse_mla_prefill(x["q"], x["kv"], idx, cfg.sm_scale, out, lse))
        del logits
        loss = torch.empty((L,), device=dev)
        dw = torch.empty((L, cfg.HI), device=dev)
        dq = torch.empty((L, cfg.HI, cfg.dI), device=dev)
        dk = torch.empty((L, cfg.dI), device=dev)
        ws = torch.empty(dsa.dsa_indexer_warmup_workspace_size(L, L, cfg.HI, cfg.dI), dtype=torch.uint8, device=dev)
        return (f"dsa_indexer_warmup, L={L} causal, H={cfg.H}, H_I={cfg.HI}",
                lambda: dsa.dsa_indexer_warmup(x["q"], x["kv"], cfg.sm_scale, x["q8"], x["qs"], x["w"], x["k8"],
                                               x["ks"], x["q_pos"], loss, dw, dq, dk, workspace=ws))
    if name == "fused_rows_32k":
        cfg = W.CONFIGS["prefill_32k"]
        rows = np.arange(cfg.L - 2048, cfg.L)
        x = W.prefill_rows(cfg, dev, rows)
        idx = torch.empty((len(rows), cfg.k), dtype=torch.int32, device=dev)
        ws = torch.empty(dsa.dsa_indexer_topk_workspace_size(len(rows), cfg.L, cfg.HI, cfg.dI, cfg.k),
                         dtype=torch.uint8, device=dev)
        return (f"dsa_indexer_topk, query rows [{cfg.L - 2048}, {cfg.L}) over {cfg.L} keys, k={cfg.k}",
                lambda: dsa.dsa_indexer_topk(x["q8"], x["qs"], x["w"], x["k8"], x["ks"], x["q_pos"], cfg.k, idx,
                                             workspace=ws))
    if name == "decode":
        cfg = W.CONFIGS["decode_paged"]
        d = W.decode_inputs(cfg, dev)
        B = int(d["ctx"].shape[0])
        logits = torch.empty((B, int(d["ctx"].max())), dtype=torch.float32, device=dev)
        idx = torch.empty((B, cfg.k), dtype=torch.int32, device=dev)
        out = torch.empty((B, cfg.H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, cfg.H), dtype=torch.float32, device=dev)
        ws_n = dsa.dsa_sparse_mla_decode_workspace_size(B, cfg.H, cfg.k)
        ws = torch.empty(ws_n, dtype=torch.uint8, device=dev) if ws_n else None

        def step():
            dsa.dsa_indexer_logits(d["q8"], d["qs"], d["w"], d["k8_pool"], d["ks_pool"], d["q_pos"], logits,
                                   block_table=d["block_table"])
            dsa.dsa_topk(logits, d["ctx"], cfg.k, idx)
            dsa.dsa_sparse_mla_decode_paged(d["q"], d["kv_pool"], d["block_table"], d["ctx"], idx, cfg.sm_scale,
                                            out, lse, workspace=ws)
        return (f"decode step: B={B}, ctx U[{cfg.ctx_lo},{cfg.ctx_hi}], page {cfg.page_size}, k={cfg.k}", step)
    raise ValueError(name)


PROFILE_CASES = ("indexer_4k", "topk_4k", "mla_4k", "warmup_4k", "fused_rows_32k", "decode")


def run_case(dsa, name, steps, warmup, dev):
    """--case: `warmup` calls, then `steps` calls of one entry point between two events.  The
    line is for locating launches in a profiler capture, not a measurement of the method."""
    what, call = case_setup(dsa, name, dev)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"case": name, "what": what, "warmup_calls": warmup, "calls": steps,
                      "ms_per_call": e0.elapsed_time(e1) / max(steps, 1),
                      "device_status": dsa.dsa_get_device_status()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="dsa", choices=["dsa", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=["prefill_32k", "prefill_4k"])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip tiny, L=4096 and the chunked L=131072")
    ap.add_argument("--case", choices=PROFILE_CASES,
                    help="only run one entry point on a small input (--warmup then --steps calls), for profiling")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.case:
        import sparse_attention_02_gb300 as dsa

        dsa.load_library()
        run_case(dsa, args.case, args.steps, args.warmup, torch.device("cuda", 0))
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import sparse_attention_02_gb300 as dsa

    dsa.load_library()  # fails loudly when the CUDA library is missing
    peaks, peaks_src = load_peaks()
    mm = measure_matmul_peaks(dev)
    torch.cuda.empty_cache()
    cfg = W.CONFIGS[args.workload]
    L = cfg.L
    x = W.prefill_inputs(cfg, dev)
    b = prefill_buffers(cfg, x, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t_wall0 = time.perf_counter()
    step_ms, st = time_prefill(dsa, x, b, cfg, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t_wall1 = time.perf_counter()
    clk = clocks.stop()
    status = dsa.dsa_get_device_status()

    stage_ms = st.mean(0)
    ms, value = aggregate_over_ranks(float(step_ms.mean()), L, dist, dev)
    work = prefill_work(L, cfg.k, cfg.HI, cfg.dI, cfg.H)
    pk = run_peaks(peaks, peaks_src, clk, mm)
    stages = stage_records(work, stage_ms, L, pk)
    mla = stages["sparse_mla"]
    traffic = recorded_traffic(f"sparse_mla_{args.workload}", ["sparse_mla.cu", "common.cuh"])

    out_hash = None
    if rank == 0:
        hsh = hashlib.sha1()
        hsh.update(b["idx"].cpu().numpy().tobytes())
        hsh.update(b["lse"].cpu().numpy().tobytes())
        out_hash = hsh.hexdigest()[:16]

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8e4m3+bf16 (fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": workload_desc(cfg),
                   "l2": "flushed before every timed step (256 MB write, outside the timed events)",
                   "timing": "ms_per_step: CUDA events at step boundaries only (kernels launched with programmatic "
                             "dependent launch overlap their launch with the previous kernel's tail); stage ms: "
                             "a second pass of the same steps with an event between stages",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "sparse_mla_prefill", "achieved": mla["tflops"],
                     "peak": pk["bf16"], "unit": "TFLOP/s", "frac": mla["frac"],
                     "frac_sustained": mla["frac_sustained"], "frac_nominal": mla["frac_nominal"],
                     "traffic": traffic, "peak_source": pk["bf16_how"],
                     "algorithmic_flop_per_launch": work["mla_flop"]},
        "stages": stages,
        "matmul_peaks": mm,
        "clocks": clk,
        "gpu_launches": 3 * args.steps,
        "device_status": status,
        "output_hash": out_hash,
        "timed_wall_s": t_wall1 - t_wall0,
    }
    line["fused"] = fused_bench(dsa, x, b, cfg, max(3, min(args.steps, 10)), args.warmup, flush, dev, stages)
    if not args.no_e2e:
        line["e2e"] = e2e_bench(dsa, x, b, cfg, max(2, min(args.steps, 16)), dev)
        line["e2e"]["value"] *= world
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, x)
    del b, x
    torch.cuda.empty_cache()
    if not args.no_decode:
        line["stages"]["quantize"] = quantize_bench(dsa, cfg, args.steps, args.warmup, flush, pk["hbm"], dev)
        torch.cuda.empty_cache()
        line["decode"] = decode_bench(dsa, args.steps, args.warmup, flush, peaks, dev)
    if not args.no_workloads:
        line["workloads"] = {}
        for name in OTHER_WORKLOADS:
            if name == args.workload:
                continue
            n_steps = 3 if W.CONFIGS[name].chunk else max(3, min(args.steps, 10))
            line["workloads"][name] = workload_bench(dsa, name, n_steps, args.warmup, flush, peaks, peaks_src, mm,
                                                     dev)
        line["workloads"]["warmup_4k"] = warmup_bench(dsa, 5, args.warmup, flush, peaks, peaks_src, mm, dev)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
