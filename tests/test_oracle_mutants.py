"""The oracle's pins have teeth: plausible mistakes planted in a copy of the
oracle (compiled on the CPU into a temporary library) must each fail at least
one pin from test_oracle_pins.py.  Nothing here touches a GPU."""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_append as app
import test_oracle_hier as hier
import test_oracle_pins as pins

SRC = open(oracle._SRC).read()

MUTANTS = {
    "drop_head_weight": ("total += (double)C->w[(size_t)t * D->H_I + j] * relu;", "total += relu;"),
    "relu_wrong_side": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot < 0.0 ? -dot : 0.0;"),
    "no_relu": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "ties_to_higher": ("return (x->pos > y->pos) - (x->pos < y->pos);", "return (x->pos < y->pos) - (x->pos > y->pos);"),
    "ignore_block_table": ("return (int64_t)blk * D->block_size + s % D->block_size;",
                           "return (int64_t)b * D->max_blocks * D->block_size + s;"),
    "transposed_query": ("dot += q[(size_t)j * D->d_I + e] * k[e];", "dot += q[(size_t)e * D->H_I + j] * k[e];"),
    "e4m3_bias_8": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);", "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_no_subnormal": ("if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = ldexp(1.0 + (double)m / 8.0, -7);"),
    "no_block_scale": ("double scale = (OMODE(D) == 2) ? (double)C->k_I_scale[blk] : 1.0;", "double scale = 1.0;"),
    "not_causal_inclusive": ("if (s1 > pos + 1) s1 = pos + 1;", "if (s1 > pos) s1 = pos;"),
    "drop_sm_scale": ("z[i] = C->sm_scale * dot;", "z[i] = dot;"),
    "value_width_d_v": ("o[c] += p * rows[(size_t)i * D->d + c];", "o[c] += p * rows[(size_t)i * D->d_v + c];"),
    "no_max_shift": ("for (int i = 0; i < n; ++i) { z[i] = exp(z[i] - m); l += z[i]; }",
                     "for (int i = 0; i < n; ++i) { z[i] = exp(z[i]); l += z[i]; }"),
    "kth_off_by_one": ("C->kth[2 * t + 0] = (K - 1 < n) ? a[K - 1].s : NAN;", "C->kth[2 * t + 0] = (K < n) ? a[K].s : NAN;"),
    "e4m3_encode_truncates": ("double m = rint((ldexp(a, -E) - 1.0) * 8.0); /* 0..8 */",
                              "double m = floor((ldexp(a, -E) - 1.0) * 8.0); /* 0..8 */"),
    "e4m3_encode_no_subnormal": ("const double m = rint(ldexp(a, 9));", "const double m = 0.0;"),
    "append_ignores_earlier_tokens": ("if (u < 0 && i >= n_old) continue;\n            for (int d = 0; d < D->d_I; ++d) {\n                float x;\n                if (u >= 0) x = (float)oracle_bf16_to_f64(knew[(int64_t)u * D->d_I + d]);\n                else x = (float)oracle_e4m3_to_f64(codes[((int64_t)blk * bs + i) * D->d_I + d]) * old_scale;\n                const float ax",
                                      "if (u < 0) continue;\n            for (int d = 0; d < D->d_I; ++d) {\n                float x;\n                if (u >= 0) x = (float)oracle_bf16_to_f64(knew[(int64_t)u * D->d_I + d]);\n                else x = (float)oracle_e4m3_to_f64(codes[((int64_t)blk * bs + i) * D->d_I + d]) * old_scale;\n                const float ax"),
    "summary_divides_by_block_size": ("f32_to_bf16_rne(acc / (float)cnt);", "f32_to_bf16_rne(acc / (float)bs);"),
    "summary_skips_last_token": ("for (int i = 0; i < cnt; ++i) {\n                    const size_t e = ((size_t)blk * bs + i) * D->d_I + d;",
                                 "for (int i = 0; i + 1 < cnt; ++i) {\n                    const size_t e = ((size_t)blk * bs + i) * D->d_I + d;"),
    "append_keeps_old_scale": ("const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;", "const float scale = old_scale;"),
    "append_wrong_slot": ("const int64_t row = (int64_t)block_table[(int64_t)b * D->max_blocks + pos / bs] * bs + pos % bs;",
                          "const int64_t row = (int64_t)block_table[(int64_t)b * D->max_blocks + pos / bs] * bs + (pos + 1) % bs;"),
    "mx_query_not_quantised": ("    if (OMODE(D) == 3)  /* the MXFP8 query", "    if (0)  /* the MXFP8 query"),
    "mx_scale_bias_126": ("e / 32] - 127);\n            k[e]", "e / 32] - 126);\n            k[e]"),
    "mx_first_group_scale_only": ("[(size_t)row * (D->d_I / 32) + e / 32] - 127);", "[(size_t)row * (D->d_I / 32)] - 127);"),
    "mx_exponent_is_ceil": ("X = (e - 1) - 8;", "X = e - 8;"),
    "mx_summary_first_group_scale": ("* (D->d_I / 32) + d / 32] - 127);", "* (D->d_I / 32)] - 127);"),
    "mx_append_quantises_group_0_everywhere": ("[(int64_t)t * D->d_I + 32 * g + i]);", "[(int64_t)t * D->d_I + i]);"),
    "kv_fp8_tile_of_64": ("memcpy(&scale, rec + D->d + 4 * (e / 128), sizeof scale);",
                          "memcpy(&scale, rec + D->d + 4 * ((e / 64) % ((D->d + 127) / 128)), sizeof scale);"),
    "kv_fp8_ignores_scale": ("return oracle_e4m3_to_f64(rec[e]) * (double)scale;", "return oracle_e4m3_to_f64(rec[e]);"),
    "kv_fp8_append_first_tile_amax": ("for (int e = e0; e < e1; ++e) {\n                    const float v = fabsf(",
                                      "for (int e = 0; e < (D->d < 128 ? D->d : 128); ++e) {\n                    const float v = fabsf("),
    "kv_fp8_append_scale_slot": ("memcpy(rec + D->d + 4 * j, &tile_scale, sizeof tile_scale);",
                                 "memcpy(rec + D->d, &tile_scale, sizeof tile_scale);"),
    "mx_append_wrong_scale_row": ("((uint8_t*)k_scale)[row * (D->d_I / 32) + g] = (uint8_t)(X + 127);",
                                  "((uint8_t*)k_scale)[(row ^ 1) * (D->d_I / 32) + g] = (uint8_t)(X + 127);"),
}

PIN_TESTS = [
    pins.test_e4m3_decoder_all_codes_vs_torch,
    pins.test_hand_example_indexer,
    pins.test_hand_example_attention,
    lambda: [pins.test_topk_matches_brute_force(*p) for p in pins.TINY],
    pins.test_prefill_rows_are_causal,
    pins.test_exact_ties_go_to_lower_position,
    lambda: [pins.test_attention_full_selection_equals_dense_sdpa(m) for m in ("f32", "bf16")],
    pins.test_attention_zero_query_is_mean_of_values,
    app.test_e4m3_encoder_matches_torch_cast,
    app.test_append_copies_rows_in_f32_and_bf16,
    app.test_append_whole_new_block_matches_the_generators_quantisation,
    app.test_append_requantises_the_earlier_tokens_of_the_block,
    app.test_append_keeps_codes_when_the_block_scale_does_not_grow,
    lambda: [hier.test_summaries_match_sequential_numpy_mean(m) for m in ("f32", "bf16", "bf16_kfp8", "mxfp8")],
    lambda: pins.test_topk_matches_brute_force(*pins.TINY[-1]),
    pins.test_mx_quantiser_matches_numpy_torch_recipe,
    pins.test_mx_scores_equal_bf16_scores_of_the_decoded_values,
    app.test_append_mx_quantises_each_new_key_on_its_own,
    hier.test_planted_block_is_chosen,
    pins.test_kv_fp8_attention_matches_brute_force,
    pins.test_kv_fp8_single_row_is_its_decoded_values,
    pins.test_kv_fp8_power_of_two_tile_scales_change_nothing,
    app.test_append_fp8_latent_rows_match_the_generators_quantisation,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(SRC.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o",
                           lib_path, str(src), "-lm"])
    saved = oracle._lib
    oracle._lib = oracle._bind(ctypes.CDLL(lib_path))
    caught = []
    try:
        for fn in PIN_TESTS:
            try:
                fn()
            except (AssertionError, RuntimeError, ValueError):
                caught.append(getattr(fn, "__name__", "lambda"))
    finally:
        oracle._lib = saved
    assert caught, f"no pin caught mutant {name}"


# The coarse -> fine composition of hierarchical selection is Python (oracle.summary_case and
# oracle.hierarchical_topk over the C indexer); its mutants are planted in a copy of one
# function's source, which replaces that function in the module.
PY_MUTANTS = {
    "hier_no_causal_cut": ("hierarchical_topk", "min((b + 1) * bs, n)", "(b + 1) * bs"),
    "hier_fine_ties_to_higher": ("hierarchical_topk", "order = np.lexsort((pos, -sc))[: s.K]",
                                 "order = np.lexsort((-pos, -sc))[: s.K]"),
    "hier_first_blocks_not_best": ("hierarchical_topk", "bl = np.sort(bidx[r][bidx[r] >= 0])",
                                   "bl = np.arange(min(n_sel, (n + bs - 1) // bs))"),
    "hier_positions_in_score_order": ("hierarchical_topk", "chosen = np.sort(pos[order])", "chosen = pos[order]"),
    "hier_coarse_sees_next_block": ("summary_case", "q_pos=(case.q_pos // bs).astype(np.int32)",
                                    "q_pos=(case.q_pos // bs + 1).astype(np.int32)"),
    "hier_coarse_block_rounded_up": ("summary_case", "q_pos=(case.q_pos // bs).astype(np.int32)",
                                     "q_pos=np.minimum((case.q_pos + bs - 1) // bs, lens[case.q_seq] - 1).astype(np.int32)"),
}

HIER_PINS = [
    lambda: [hier.test_hierarchical_matches_brute_force(m) for m in ("bf16", "bf16_kfp8", "mxfp8")],
    hier.test_all_blocks_kept_reproduces_the_exact_topk,
    hier.test_planted_block_is_chosen,
    hier.test_equal_keys_take_the_lowest_blocks_and_positions,
    hier.test_block_past_the_row_is_never_chosen,
]


def _patched(monkeypatch, fn_name: str, old: str = "", new: str = ""):
    """Replaces oracle.<fn_name> with a copy of its source (with old -> new), compiled against the
    module's globals, so the module's other functions call the copy."""
    import inspect
    src = inspect.getsource(getattr(oracle, fn_name))
    if old:
        assert src.count(old) == 1, f"mutation anchor {old!r} not found exactly once"
    ns = dict(vars(oracle))
    exec(src.replace(old, new) if old else src, ns)
    monkeypatch.setattr(oracle, fn_name, ns[fn_name])


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_python_mutant_is_caught(name, monkeypatch):
    _patched(monkeypatch, *PY_MUTANTS[name])
    caught = []
    for fn in HIER_PINS:
        try:
            fn()
        except (AssertionError, IndexError, RuntimeError, ValueError):
            caught.append(getattr(fn, "__name__", "lambda"))
    assert caught, f"no pin caught mutant {name}"


@pytest.mark.parametrize("fn_name", ["hierarchical_topk", "summary_case"])
def test_python_mutant_harness_control(fn_name, monkeypatch):
    """An unmodified copy of the function, made the same way, passes every pin (so a caught
    mutant is caught by its mutation, not by the copying)."""
    _patched(monkeypatch, fn_name)
    for fn in HIER_PINS:
        fn()
