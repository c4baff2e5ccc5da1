"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, a wrong index, a transposed operand, a wrong bound),
builds it, and checks that at least one pin from test_oracle_pins fails on
it.  CPU only; the real oracle is restored afterwards.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_training as tpins

SRC = os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")

MUTANTS = {
    "relu_dropped": ("score += (double)wt[j] * (dot > 0.0 ? dot : 0.0);", "score += (double)wt[j] * dot;"),
    "relu_sign": ("(dot > 0.0 ? dot : 0.0)", "(dot < 0.0 ? dot : 0.0)"),
    "key_scale_dropped": ("(dsa_oracle_e4m3(k8s[d]) * ks)", "(dsa_oracle_e4m3(k8s[d]))"),
    "query_transposed": ("q8t[(int64_t)j * dI + d]", "q8t[(int64_t)d * HI + j]"),
    "causal_exclusive": ("for (int s = 0; s <= last; ++s)", "for (int s = 0; s < last; ++s)"),
    "head_weight_index": ("score += (double)wt[j]", "score += (double)wt[0]"),
    "e4m3_bias": ("ldexp(1.0 + (double)man / 8.0, ex - 7)", "ldexp(1.0 + (double)man / 8.0, ex - 8)"),
    "e4m3_subnormal": ("ldexp((double)man / 8.0, 1 - 7)", "ldexp((double)man / 8.0, -7)"),
    "tie_break_reversed": ("return (x->s > y->s) - (x->s < y->s);", "return (x->s < y->s) - (x->s > y->s);"),
    "topk_order_unsorted": ("qsort(o, (size_t)m, sizeof(int32_t), cmp_int32);", ""),
    "topk_rank_ascending": ("if (x->v > y->v) return -1;\n    if (x->v < y->v) return 1;",
                            "if (x->v < y->v) return -1;\n    if (x->v > y->v) return 1;"),
    "v_columns_shifted": ("o[v] += p * dsa_oracle_bf16(c[v]);", "o[v] += p * dsa_oracle_bf16(c[v + 64]);"),
    "lse_max_dropped": ("*lse = m + log(z);", "*lse = log(z);"),
    "softmax_unnormalised": ("o[v] /= z;", "o[v] /= 1.0;"),
    "sm_scale_dropped": ("score[i] = sm_scale * dot;", "score[i] = dot;"),
    "paged_slot": ("rows_sel[i] = (int64_t)page * page_size + s % page_size;",
                   "rows_sel[i] = (int64_t)page * page_size + s / page_size;"),
    "paged_index_slot": ("int64_t slot = (int64_t)page * page_size + s % page_size;",
                         "int64_t slot = (int64_t)page * page_size;"),
    "prefill_bound": ("rows_sel[i] = (s >= 0 && s < S) ? (int64_t)s : -1;", "rows_sel[i] = (int64_t)s;"),
    "query_scale_dropped": ("(dsa_oracle_e4m3(q8t[(int64_t)j * dI + d]) * qs)",
                            "(dsa_oracle_e4m3(q8t[(int64_t)j * dI + d]))"),
    "paged_table_row": ("block_table[(int64_t)r * max_pages + s / page_size]", "block_table[s / page_size]"),
    "rope_dropped": ("for (int d = 0; d < D; ++d)\n            dot += dsa_oracle_bf16(q_rh[d])",
                     "for (int d = 0; d < 512; ++d)\n            dot += dsa_oracle_bf16(q_rh[d])"),
    "topk_pad_zero": ("            o[i] = -1;", "            o[i] = 0;"),
    "topk_k_off_by_one": ("int m = n < k ? n : k;", "int m = n < k ? n : k - 1;"),
    "lse_log2": ("*lse = m + log(z);", "*lse = m + log2(z);"),
    "paged_ctx_bound": ("if (s < 0 || s >= ctx_len[r] || s / page_size >= max_pages)",
                        "if (s < 0 || s / page_size >= max_pages)"),
    "e4m3_ties_up": ("code = (lo % 2 == 0) ? lo : hi;", "code = hi;"),
    "e4m3_saturates_to_nan": ("return (uint8_t)(sign | 0x7E);", "return (uint8_t)(sign | 0x7F);"),
    "quant_scale_constant": ("const float ratio = amax / 448.f;", "const float ratio = amax / 447.f;"),
    "quant_amax_signed": ("const float m = fabsf(xr[c]);", "const float m = xr[c];"),
    "quant_zero_row_scale": ("        float s = 1.f;\n", "        float s = 0.5f;\n"),
    "ue8m0_rounds_down": ("ldexp(1.0, e)", "ldexp(1.0, e - 1)"),
    # indexer warm-up (training path)
    "kl_grad_sign": ("g[s] = exp(g[s] - lse) - ps;", "g[s] = ps - exp(g[s] - lse);"),
    "kl_lse_dropped": ("L += ps * (log(ps) - (g[s] - lse));", "L += ps * (log(ps) - g[s]);"),
    "kl_grad_relu_mask_dropped": ("        return a > 0.0;\n", "        return 1;\n"),
    "kl_dk_relu_mask_dropped": ("sabs))\n                    for", "sabs) || 1)\n                    for"),
    "kl_relu_fp64_sign_at_zero": ("    return acc > 0;\n", "    return a > 0.0;\n"),
    "kl_dw_relu_dropped": ("dw[(int64_t)r * HI + j] += g[s] * a;", "dw[(int64_t)r * HI + j] += g[s];"),
    "kl_dk_weight_dropped": ("dk[(int64_t)s * dI + d] += gs * w[(int64_t)r * HI + j] * qr[(int64_t)j * dI + d];",
                             "dk[(int64_t)s * dI + d] += gs * qr[(int64_t)j * dI + d];"),
    "target_not_head_mean": ("acc[s] += exp(sc[s] - m) / z / H;", "acc[s] += exp(sc[s] - m) / z;"),
    "target_causal_exclusive": ("const int cnt = last + 1;\n        double *sc", "const int cnt = last;\n        double *sc"),
    "target_scale_dropped": ("sc[s] = sm_scale * dot;", "sc[s] = dot;"),
}

PINS = [
    lambda: pins.test_e4m3_decoder_matches_torch_all_codes(),
    lambda: pins.test_indexer_hand_example(False),
    lambda: pins.test_indexer_hand_example(True),
    lambda: pins.test_topk_hand_example(),
    lambda: pins.test_indexer_single_head_is_relu_of_matmul(),
    lambda: pins.test_indexer_head_weights_are_linear_and_heads_commute(),
    lambda: pins.test_indexer_relu_sign(),
    lambda: pins.test_indexer_paged_equals_contiguous(),
    lambda: pins.test_topk_worked_tie_row(),
    lambda: pins.test_topk_matches_brute_force(False),
    lambda: pins.test_topk_matches_brute_force(True),
    lambda: pins.test_mla_equals_dense_causal_when_everything_is_selected(),
    lambda: pins.test_mla_permutation_invariance_and_padding(),
    lambda: pins.test_mla_closed_forms(),
    lambda: pins.test_mla_split_and_combine(),
    lambda: pins.test_mla_paged_equals_contiguous(),
    lambda: pins.test_quantize_hand_example(),
    lambda: pins.test_e4m3_encoder_inverts_the_decoder(),
    lambda: pins.test_e4m3_encoder_ties_to_even_and_saturates(),
    lambda: pins.test_e4m3_encoder_matches_torch_cast(),
    lambda: pins.test_quantize_matches_torch_per_row_and_scale_modes(),
    lambda: tpins.test_gradients_match_central_differences(),
    lambda: tpins.test_minimum_at_the_indexers_own_distribution(),
    lambda: tpins.test_uniform_indexer_closed_form(),
    lambda: tpins.test_target_one_head_is_the_library_softmax(),
    lambda: tpins.test_target_is_the_head_mean_and_sums_to_one(),
    lambda: tpins.test_relu_decision_is_exact_at_cancellation(),
]


def _build_mutant(src_text: str, d: str) -> str:
    c = os.path.join(d, "mutant.c")
    so = os.path.join(d, "libmutant.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", c, "-o", so, "-lm"])
    return so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_planted_mistake_fails_a_pin(name, monkeypatch):
    before, after = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(before) >= 1, f"mutation site for {name} not found"
    mutated = text.replace(before, after)
    with tempfile.TemporaryDirectory() as d:
        so = _build_mutant(mutated, d)
        monkeypatch.setattr(oracle, "_LIB_PATH", so)
        monkeypatch.setattr(oracle, "_SRC", os.path.join(d, "mutant.c"))
        monkeypatch.setattr(oracle, "_lib", None)
        failed = []
        for i, pin in enumerate(PINS):
            try:
                pin()
            except AssertionError:
                failed.append(i)
        monkeypatch.setattr(oracle, "_lib", None)
    assert failed, f"mutant {name} passed every pin"
