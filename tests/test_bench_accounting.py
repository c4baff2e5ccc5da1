"""The bench's algorithmic work counts (the numerators of every roofline fraction) against
closed forms and a brute-force count, and the oracle-time extrapolation (CPU)."""
import numpy as np

import bench


def _closed_forms(L, k, HI, dI, H, D=576, Dv=512):
    rows = L * (L + 1) // 2                                   # sum over t of (t + 1) candidates
    sel = k * (k + 1) // 2 + (L - k) * k if L >= k else rows  # sum over t of min(t + 1, k)
    need = rows - k * (k + 1) // 2 if L > k else 0            # candidates of rows with t + 1 > k
    return dict(indexer_flop=2 * HI * dI * rows, mla_flop=2 * H * (D + Dv) * sel,
                topk_bytes=4 * need + 4 * L + 4 * L * k, selected_pairs=sel, key_rows=rows)


def test_prefill_work_matches_closed_forms():
    for L, k, HI, dI, H in [(32768, 2048, 64, 128, 128), (4096, 2048, 64, 128, 128), (256, 64, 4, 32, 16),
                            (100, 2048, 4, 32, 16), (2049, 2048, 64, 128, 128)]:
        got = bench.prefill_work(L, k, HI, dI, H)
        want = _closed_forms(L, k, HI, dI, H)
        for key, v in want.items():
            assert got[key] == v, (L, k, key, got[key], v)


def test_prefill_work_headline_figures():
    w = bench.prefill_work(32768, 2048, 64, 128, 128)
    assert round(w["indexer_flop"] / 1e12, 2) == 8.80   # FP8 indexer at L = 32K
    assert round(w["mla_flop"] / 1e12, 1) == 18.1       # BF16 sparse attention at L = 32K
    assert round(w["topk_bytes"] / 1e9, 2) == 2.41      # top-k logits read + indices
    w4 = bench.prefill_work(4096, 2048, 64, 128, 128)
    assert round(w4["indexer_flop"] / 1e12, 3) == 0.137
    assert round(w4["mla_flop"] / 1e12, 2) == 1.75


def test_selected_pairs_brute_force():
    L, k = 37, 5
    pairs = 0
    for t in range(L):  # row t keeps k of its t + 1 candidates, or all of them
        for s in range(t + 1):
            pairs += 1 if s < k else 0
    assert bench.prefill_work(L, k, 1, 1, 1)["selected_pairs"] == pairs


def test_oracle_extrapolation_is_the_per_unit_sum():
    rates = dict(indexer_s_per_unit=3e-9, topk_s_per_unit=1e-9, mla_s_per_unit=7e-8)
    L, k = 1000, 64
    est = bench.oracle_full_estimate(rates, L, k)
    rows = L * (L + 1) / 2
    sel = k * (k + 1) / 2 + (L - k) * k
    assert np.isclose(est, 3e-9 * rows + 1e-9 * rows + 7e-8 * sel, rtol=1e-12)
