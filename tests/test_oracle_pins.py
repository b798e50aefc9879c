"""Pins for the fp64 oracle against things other than itself (CPU only).

* decoders: every bf16 pattern against NumPy's bit widening, every e4m3 code
  against torch's float8_e4m3fn cast and the OCP spec values in
  tests/golden/e4m3_spec_values.json;
* indexer + Top-K: a hand-worked example (tests/golden/indexer_hand.json),
  NumPy brute force (full score matrix + lexsort) on tiny inputs in all four
  storage modes, exact ties on integer data, the single-column special case
  (a plain sort), power-of-two FP8 scale changes and planted index sets;
* attention: the hand-worked example, K >= L equals dense attention (torch
  CPU float64 SDPA), softmax weights sum to one, q = 0 gives the mean of the
  selected value rows, a dominant logit gives that row, one row gives that
  row, no row gives zeros and lse = -inf;
* paging: a different physical block permutation changes nothing;
* MXFP8: the oracle's group quantiser against the generator's NumPy/torch
  recipe and closed forms, and MXFP8 scores equal to bf16 scores of the
  decoded values (the bf16 path being pinned above).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from cases import (act, brute_attn_row, brute_scores_row, brute_topk_row, logical_keys, logical_kv, mx_roundtrip,
                   np_bf16, np_e4m3, np_mx, sdpa_f64, small_spec)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# decoders
# ----------------------------------------------------------------------------

def test_bf16_decoder_all_patterns():
    lib = oracle._load()
    bits = np.arange(1 << 16, dtype=np.uint32)
    ref = np_bf16(bits)
    got = np.array([lib.oracle_bf16_to_f64(int(b)) for b in bits[::37]])
    r = ref[::37]
    both_nan = np.isnan(got) & np.isnan(r)
    assert np.all(both_nan | (got == r))
    # signed zeros and infinities keep their sign
    assert math.copysign(1.0, oracle.bf16_to_f64(0x8000)) == -1.0
    assert oracle.bf16_to_f64(0x7F80) == math.inf
    assert oracle.bf16_to_f64(0x3F80) == 1.0


def test_e4m3_decoder_all_codes_vs_torch():
    ref = np_e4m3(np.arange(256, dtype=np.uint8))
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_decoder_spec_values():
    spec = json.load(open(os.path.join(GOLDEN, "e4m3_spec_values.json")))
    for row in spec["values"]:
        v = oracle.e4m3_to_f64(int(row["code"], 16))
        if row["value"] == "nan":
            assert math.isnan(v), row
        else:
            assert v == row["value"], row
            assert math.copysign(1.0, v) == math.copysign(1.0, row["value"]), row


# ----------------------------------------------------------------------------
# hand-worked example
# ----------------------------------------------------------------------------

def _hand_case():
    g = json.load(open(os.path.join(GOLDEN, "indexer_hand.json")))
    dm = g["dims"]
    spec = W.Spec("hand", "f32", [dm["seq_len"]], [1], H_I=dm["H_I"], d_I=dm["d_I"], H=dm["H"], d=dm["d"],
                  d_v=dm["d_v"], K=dm["K"], spare_blocks=0)
    L = dm["seq_len"]
    k_I = np.full((1, 64, dm["d_I"]), 99.0, np.float32)
    k_I[0, :L] = np.asarray(g["k_I"], np.float32)
    kv = np.full((1, 64, dm["d"]), 99.0, np.float32)
    kv[0, :L] = np.asarray(g["kv"], np.float32)
    case = W.Case(spec, 0, np.zeros((1, 1), np.int32), np.array([L], np.int32), np.array([0], np.int32),
                  np.array([L - 1], np.int32), np.asarray(g["q_I"], np.float32)[None], np.asarray(g["w"], np.float32)[None],
                  k_I, None, np.asarray(g["q"], np.float32)[None], kv)
    return g, case


def test_hand_example_indexer():
    g, case = _hand_case()
    S = oracle.index_scores(case)[0]
    assert np.array_equal(S, np.asarray(g["expected_scores"]))
    idx, kth = oracle.indexer_topk(case)
    assert idx[0].tolist() == g["expected_idx"]
    assert kth[0].tolist() == g["expected_kth"]


def test_hand_example_attention():
    g, case = _hand_case()
    idx = np.asarray(g["expected_idx"], np.int32)[None]
    out, lse, psum = oracle.sparse_attn(case, idx)
    np.testing.assert_allclose(out[0], np.asarray(g["expected_out"]), rtol=0, atol=1e-6)
    np.testing.assert_allclose(lse[0], np.asarray(g["expected_lse"]), rtol=0, atol=1e-6)
    np.testing.assert_allclose(psum[0], 1.0, atol=1e-15)


# ----------------------------------------------------------------------------
# brute force on tiny inputs
# ----------------------------------------------------------------------------

TINY = [
    ("f32", [0, 1, 63, 64, 65, 200], 8),
    ("f32", [130, 7], 256),          # K > L
    ("bf16", [1, 64, 65, 129], 16),
    ("bf16_kfp8", [63, 64, 65, 300], 32),
    ("mxfp8", [63, 64, 65, 300], 32),
]


@pytest.mark.parametrize("mode,lens,K", TINY)
def test_topk_matches_brute_force(mode, lens, K):
    kw = {} if mode == "f32" else dict(H_I=8, d_I=64 if mode == "mxfp8" else 32, H=4, d=64, d_v=48)
    spec = small_spec(mode, lens, K, **kw)
    case = W.generate(spec, seed=11 + len(lens))
    S_or = oracle.index_scores(case)
    idx, kth = oracle.indexer_topk(case)
    for t in range(spec.T):
        S = brute_scores_row(case, t)
        n = len(S)
        np.testing.assert_allclose(S_or[t, :n], S, rtol=1e-12, atol=1e-12)
        assert np.all(np.isnan(S_or[t, n:]))
        assert idx[t].tolist() == brute_topk_row(S, K).tolist()
        srt = np.sort(S)[::-1]
        want = [srt[K - 1] if K - 1 < n else np.nan, srt[K] if K < n else np.nan]
        np.testing.assert_allclose(kth[t], want, rtol=1e-12, atol=1e-12, equal_nan=True)


def test_prefill_rows_are_causal():
    spec = small_spec("f32", [300, 150], 32, new_tokens=[40, 7])
    case = W.generate(spec, seed=5)
    S = oracle.index_scores(case)
    idx, _ = oracle.indexer_topk(case)
    for t in range(spec.T):
        n = int(case.q_pos[t]) + 1
        ref = brute_scores_row(case, t)
        np.testing.assert_allclose(S[t, :n], ref, rtol=1e-12, atol=1e-12)
        assert idx[t].max() <= case.q_pos[t]
        assert idx[t].tolist() == brute_topk_row(ref, 32).tolist()


def test_exact_ties_go_to_lower_position():
    """Integer-valued inputs make every score exact, so duplicated keys tie exactly."""
    rng = np.random.default_rng(3)
    spec = small_spec("bf16", [150], 20, H_I=4, d_I=8)
    case = W.generate(spec, seed=3)
    q = rng.integers(-3, 4, size=case.q_I.shape).astype(np.float32)
    case.q_I = W.to_bf16_bits(q)
    case.w = rng.integers(0, 4, size=case.w.shape).astype(np.float32) / 4
    base = rng.integers(-4, 5, size=(10, spec.d_I)).astype(np.float32)
    keys = base[rng.integers(0, 10, size=150)]       # only 10 distinct keys -> many exact ties
    bs = spec.block_size
    for s in range(150):
        case.k_I[case.block_table[0, s // bs], s % bs] = W.to_bf16_bits(keys[s])
    S = brute_scores_row(case, 0)
    idx, _ = oracle.indexer_topk(case)
    assert idx[0].tolist() == brute_topk_row(S, 20).tolist()
    # among equal scores, the lower position comes first and is the one kept
    sel = idx[0]
    for a, b in zip(sel[:-1], sel[1:]):
        assert S[a] > S[b] or (S[a] == S[b] and a < b)
    cut = S[sel[-1]]
    dropped_equal = [s for s in range(150) if S[s] == cut and s not in sel]
    assert all(s > sel[-1] for s in dropped_equal)


def test_single_column_special_case_is_a_sort():
    """H_I = 1, w = 1, q_I = e_c: S[s] = max(0, k[s, c]) -> Top-K is a sort of one key column."""
    spec = small_spec("f32", [500], 64, H_I=1, d_I=16)
    case = W.generate(spec, seed=8)
    c = 5
    case.q_I[:] = 0
    case.q_I[0, 0, c] = 1.0
    case.w[:] = 1.0
    col = logical_keys(case, 0)[:, c]
    relu = np.maximum(col, 0.0)
    idx, _ = oracle.indexer_topk(case)
    expect = sorted(range(500), key=lambda s: (-relu[s], s))[:64]
    assert idx[0].tolist() == expect


def test_fp8_power_of_two_scale_scales_scores_exactly():
    spec = small_spec("bf16_kfp8", [400], 50, H_I=4, d_I=16)
    case = W.generate(spec, seed=9)
    S0 = oracle.index_scores(case)[0]
    idx0, _ = oracle.indexer_topk(case)
    case.k_I_scale = case.k_I_scale * np.float32(8.0)
    S1 = oracle.index_scores(case)[0]
    idx1, _ = oracle.indexer_topk(case)
    assert np.array_equal(S1, 8.0 * S0)
    assert np.array_equal(idx0, idx1)
    # a single block scaled up changes the ranking towards that block
    case.k_I_scale = case.k_I_scale / np.float32(8.0)
    b0 = case.block_table[0, 2]
    case.k_I_scale[b0] *= np.float32(1024.0)
    idx2, _ = oracle.indexer_topk(case)
    in_blk = [s for s in idx2[0] if 128 <= s < 192]
    S2 = brute_scores_row(case, 0)
    assert len(in_blk) == sum(1 for s in range(128, 192) if s in set(brute_topk_row(S2, 50).tolist()))


def test_planted_set_is_recovered():
    """Keys pushed along the row's weighted query direction dominate -> idx is exactly the planted set."""
    spec = small_spec("bf16", [1000], 40, H_I=8, d_I=32)
    case = W.generate(spec, seed=21)
    rng = np.random.default_rng(4)
    P = np.sort(rng.choice(1000, size=40, replace=False))
    u = (case.w[0][:, None].astype(np.float64) * np_bf16(case.q_I[0])).sum(0)
    u /= np.linalg.norm(u)
    bs = spec.block_size
    for s in P:
        blk, off = case.block_table[0, s // bs], s % bs
        k = np_bf16(case.k_I[blk, off]) + 12.0 * u
        case.k_I[blk, off] = W.to_bf16_bits(k.astype(np.float32))
    S = oracle.index_scores(case)[0]
    assert S[P].min() > 1.01 * np.delete(S, P).max()
    idx, _ = oracle.indexer_topk(case)
    assert sorted(idx[0].tolist()) == P.tolist()


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["f32", "bf16"])
def test_attention_full_selection_equals_dense_sdpa(mode):
    kw = dict(H_I=4, d_I=16, H=6, d=40, d_v=24)
    spec = small_spec(mode, [90, 33], 128, **kw)   # K >= L: every causal position is selected
    case = W.generate(spec, seed=31)
    idx, _ = oracle.indexer_topk(case)
    out, lse, psum = oracle.sparse_attn(case, idx)
    for t in range(spec.T):
        b = int(case.q_seq[t])
        rows = logical_kv(case, b)
        q = act(case, case.q[t])
        ref = sdpa_f64(q, rows, rows[:, : spec.d_v], spec.sm_scale)
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-12)
        z = (q @ rows.T) * spec.sm_scale
        np.testing.assert_allclose(lse[t], np.log(np.exp(z).sum(axis=1)), rtol=1e-12)
        np.testing.assert_allclose(psum[t], 1.0, atol=1e-12)


def test_attention_matches_brute_force_on_subset():
    spec = small_spec("bf16", [300], 64, H_I=4, d_I=16, H=4, d=64, d_v=32)
    case = W.generate(spec, seed=32)
    idx, _ = oracle.indexer_topk(case)
    out, lse, _ = oracle.sparse_attn(case, idx)
    ref, ref_lse = brute_attn_row(case, 0, idx[0])
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-12)


def test_attention_zero_query_is_mean_of_values():
    spec = small_spec("f32", [200], 32)
    case = W.generate(spec, seed=33)
    case.q[:] = 0.0
    idx, _ = oracle.indexer_topk(case)
    out, lse, _ = oracle.sparse_attn(case, idx)
    rows = logical_kv(case, 0)[idx[0]]
    np.testing.assert_allclose(out[0], np.broadcast_to(rows[:, : spec.d_v].mean(0), out[0].shape), atol=1e-13)
    np.testing.assert_allclose(lse[0], math.log(32), atol=1e-13)


def test_attention_dominant_logit_selects_that_row():
    spec = small_spec("f32", [100], 16, H=2, d=8, d_v=8)
    case = W.generate(spec, seed=34)
    idx, _ = oracle.indexer_topk(case)
    target = int(idx[0][3])
    rows = logical_kv(case, 0)
    case.q[0, 0] = (rows[target] * 1e3).astype(np.float32)   # logit of target >> others
    out, _, _ = oracle.sparse_attn(case, idx)
    np.testing.assert_allclose(out[0, 0], rows[target, : spec.d_v], atol=1e-9)


def test_attention_single_row_and_empty():
    spec = small_spec("f32", [1, 0], 8)
    case = W.generate(spec, seed=35)
    idx, _ = oracle.indexer_topk(case)
    assert idx[0].tolist() == [0] + [-1] * 7
    assert idx[1].tolist() == [-1] * 8
    out, lse, psum = oracle.sparse_attn(case, idx)
    v0 = logical_kv(case, 0)[0, : spec.d_v]
    np.testing.assert_allclose(out[0], np.broadcast_to(v0, out[0].shape), atol=0)
    q = act(case, case.q[0])
    np.testing.assert_allclose(lse[0], spec.sm_scale * (q @ logical_kv(case, 0)[0]), rtol=1e-13)
    assert np.all(out[1] == 0.0) and np.all(np.isneginf(lse[1])) and np.all(psum[1] == 0.0)


def test_attention_rejects_out_of_range_index():
    spec = small_spec("f32", [50], 8)
    case = W.generate(spec, seed=36)
    bad = np.array([[0, 1, 50, -1, -1, -1, -1, -1]], np.int32)
    with pytest.raises(RuntimeError):
        oracle.sparse_attn(case, bad)


# ----------------------------------------------------------------------------
# paging
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["f32", "bf16_kfp8"])
def test_repaging_changes_nothing(mode):
    kw = {} if mode == "f32" else dict(H_I=4, d_I=16, H=4, d=32, d_v=16)
    spec = small_spec(mode, [333, 64, 129], 48, **kw)
    case = W.generate(spec, seed=41)
    other = W.repage(case, seed=42)
    assert not np.array_equal(case.block_table, other.block_table)
    a, ka = oracle.indexer_topk(case)
    b, kb = oracle.indexer_topk(other)
    assert np.array_equal(a, b) and np.array_equal(ka, kb, equal_nan=True)
    oa = oracle.sparse_attn(case, a)[0]
    ob = oracle.sparse_attn(other, b)[0]
    assert np.array_equal(oa, ob)


def test_poisoned_slots_are_never_read():
    """Tail slots hold a huge poison value; if the oracle read them the scores would explode."""
    spec = small_spec("f32", [70], 8)
    case = W.generate(spec, seed=43)
    S = oracle.index_scores(case)[0]
    assert np.nanmax(np.abs(S)) < 1e3
    tail = case.k_I[case.block_table[0, 1], 70 % 64:]
    assert np.all(tail == W.POISON)


# ----------------------------------------------------------------------------
# MXFP8 (OCP Microscaling, E4M3 elements, one E8M0 scale per 32)
# ----------------------------------------------------------------------------

def _mx_groups():
    rng = np.random.default_rng(77)
    out = []
    for e in (-140, -126, -100, -20, -8, -1, 0, 1, 7, 8, 9, 60, 120, 126):  # scales across the range
        out.append(rng.standard_normal(32).astype(np.float32) * np.float32(2.0 ** e))
    out.append(np.zeros(32, np.float32))
    p = np.zeros(32, np.float32)
    p[3] = 2.0 ** 5                                                # amax exactly a power of two
    p[4] = -(2.0 ** -20)                                           # underflows to a zero code
    out.append(p)
    for m in (1.75, 1.8125, 1.875, 1.9375, 1.96875, 1.99):         # scaled amax near / above 448
        g = rng.uniform(-1, 1, 32).astype(np.float32)
        g[0] = np.float32(m * 4.0)
        out.append(g)
    reps = np.array([oracle.e4m3_to_f64(c) for c in range(0x7F)], np.float64)
    mids = ((reps[1:] + reps[:-1]) / 2)                            # ties at the element rounding
    for k in range(0, len(mids), 31):
        g = np.zeros(32, np.float32)
        g[:len(mids[k:k + 31])] = mids[k:k + 31] / 256.0
        g[31] = 1.0                                                # X = -8: element = x * 256
        out.append(g)
    return out


def test_mx_quantiser_matches_numpy_torch_recipe():
    for g in _mx_groups():
        X, codes = oracle.mx_quantize32(g)
        ref_codes, ref_byte = W.to_mx_e4m3(g)
        assert X == int(ref_byte[0]) - 127, g
        same = (codes == ref_codes) | (((codes & 0x7F) == 0) & ((ref_codes & 0x7F) == 0))
        assert same.all(), (g, codes, ref_codes)


def test_mx_closed_forms():
    X, c = oracle.mx_quantize32(np.full(32, 3.0, np.float32))      # floor(log2 3) = 1 -> X = -7, 3*2^7 = 384
    assert X == -7 and (c == 0x7C).all()
    X, c = oracle.mx_quantize32(np.zeros(32, np.float32))
    assert X == -127 and (c == 0).all()
    g = np.zeros(32, np.float32)
    g[0], g[1], g[2] = 1.0, -0.5, 2.0 ** -20                       # X = -8: 256, -128, below the smallest code
    X, c = oracle.mx_quantize32(g)
    assert X == -8 and c[0] == 0x78 and c[1] == 0xF0 and (c[2] & 0x7F) == 0
    g = np.full(32, 1.99, np.float32)                              # 1.99 * 256 = 509 saturates to 448
    X, c = oracle.mx_quantize32(g)
    assert X == -8 and (c == 0x7E).all()


def test_mx_scores_equal_bf16_scores_of_the_decoded_values():
    spec = small_spec("mxfp8", [200, 64, 1], 24, H_I=8, d_I=64)
    mx = W.generate(spec, seed=61)
    bf = W.generate(small_spec("bf16", [200, 64, 1], 24, H_I=8, d_I=64), seed=61)
    bf.block_table = mx.block_table.copy()
    keys = np_mx(mx.k_I, mx.k_I_scale).astype(np.float32)
    bf.k_I = W.to_bf16_bits(keys)
    assert np.array_equal(np_bf16(bf.k_I), keys.astype(np.float64))   # exactly representable
    qd = mx_roundtrip(np_bf16(mx.q_I)).astype(np.float32)
    bf.q_I = W.to_bf16_bits(qd)
    assert np.array_equal(np_bf16(bf.q_I), qd.astype(np.float64))
    bf.w = mx.w.copy()
    S_mx, S_bf = oracle.index_scores(mx), oracle.index_scores(bf)
    assert np.array_equal(S_mx, S_bf, equal_nan=True)
    assert np.array_equal(oracle.indexer_topk(mx)[0], oracle.indexer_topk(bf)[0])
    # and the query really was quantised: scores with the unquantised query differ
    bf.q_I = mx.q_I.copy()
    assert not np.array_equal(oracle.index_scores(bf), S_mx, equal_nan=True)


# ------------------------------------------------------------------ FP8 latent cache (attention stage)
# "FP8 block quantization in the attention stage" (Ascend CANN page §3): per token and head,
# independent blocks of 128 elements. A latent row is one record: d e4m3 codes, one fp32 scale per
# 128-element tile (the last tile holds the remaining d mod 128 elements), zero padding to 16 bytes.

def _kv_fp8_case(lens, K, seed, d=192, d_v=160, H=4):
    spec = small_spec("bf16", lens, K, H_I=4, d_I=16, H=H, d=d, d_v=d_v, kv="fp8")
    return W.generate(spec, seed=seed)


def test_kv_fp8_record_layout():
    """The generator's records decode to the bf16 draw within e4m3 rounding, and each tile's largest
    magnitude is stored as code 448 (scale = amax / 448)."""
    case = _kv_fp8_case([130], 32, seed=60)
    d = case.spec.d
    assert case.kv.shape[-1] == W.kv_record_bytes(d) == 208   # 192 codes + 2 scales + 8 zero bytes
    rec = case.kv[case.block_table[0, 0], 5]
    assert np.all(rec[d + 8:] == 0)
    vals = logical_kv(case, 0)[5]
    for j, (e0, e1) in enumerate(((0, 128), (128, 192))):
        assert np.max(np.abs(np_e4m3(rec[e0:e1]))) == 448.0
        sc = float(rec[d + 4 * j: d + 4 * j + 4].view(np.float32)[0])
        np.testing.assert_allclose(vals[e0:e1], np_e4m3(rec[e0:e1]) * sc, rtol=0, atol=0)


def test_kv_fp8_attention_matches_brute_force():
    """Oracle attention over FP8 records against NumPy on rows decoded with torch's e4m3 cast and the
    tile scales (a second tile of 64 elements exercises the partial last tile)."""
    case = _kv_fp8_case([5, 200, 700], 64, seed=61)
    idx, _ = oracle.indexer_topk(case)
    out, lse, psum = oracle.sparse_attn(case, idx)
    for t in range(case.spec.T):
        ref, ref_lse = brute_attn_row(case, t, idx[t])
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[t], ref_lse, rtol=1e-12)
    np.testing.assert_allclose(psum, 1.0, atol=1e-12)


def test_kv_fp8_single_row_is_its_decoded_values():
    case = _kv_fp8_case([90], 16, seed=62)
    idx = np.full((1, 16), -1, np.int32)
    idx[0, 0] = 37
    out, _, _ = oracle.sparse_attn(case, idx)
    row = logical_kv(case, 0)[37, : case.spec.d_v]
    assert np.array_equal(out[0], np.broadcast_to(row, out[0].shape))


def test_kv_fp8_power_of_two_tile_scales_change_nothing():
    """Halving every code of a tile and doubling its scale leaves every element's value, hence the
    attention, bit-identical (codes whose halving is not exact are zeroed in both copies first);
    doubling one tile's scale alone changes the output."""
    case = _kv_fp8_case([300], 64, seed=63)
    d, nt = case.spec.d, 2
    codes = case.kv[..., :d].copy()
    v = np_e4m3(codes)
    exact_half = (np.abs(v) >= 2.0 ** -5) | (v == 0)              # exponent field >= 2: halving is exact
    codes[~exact_half] = 0
    a = case.kv.copy()
    a[..., :d] = codes
    b = a.copy()
    b[..., :d] = W.to_e4m3_codes((np_e4m3(codes) / 2).astype(np.float32))
    sc = np.ascontiguousarray(a[..., d: d + 4 * nt]).view(np.float32) * np.float32(2.0)
    b[..., d: d + 4 * nt] = sc.view(np.uint8).reshape(b[..., d: d + 4 * nt].shape)
    assert np.array_equal(np_e4m3(b[..., :d]) * 2, np_e4m3(a[..., :d]))
    idx, _ = oracle.indexer_topk(case)
    case.kv = a
    out_a, lse_a, _ = oracle.sparse_attn(case, idx)
    case.kv = b
    out_b, lse_b, _ = oracle.sparse_attn(case, idx)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)
    c = a.copy()
    sc1 = np.ascontiguousarray(c[..., d + 4: d + 8]).view(np.float32) * np.float32(2.0)
    c[..., d + 4: d + 8] = sc1.view(np.uint8).reshape(c[..., d + 4: d + 8].shape)   # tile 1 only
    case.kv = c
    out_c, _, _ = oracle.sparse_attn(case, idx)
    assert not np.array_equal(out_c, out_a)
