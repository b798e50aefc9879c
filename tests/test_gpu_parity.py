"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on seeded inputs.

Index sets follow the rule: exact where the oracle's K-th and (K+1)-th scores differ by more
than 1e-3 (relative), else the 1e-3 band rule; attention is compared with the oracle evaluated on
the GPU's own index sets, max-abs 2e-2 for bf16 outputs and 1e-4 for fp32.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from cases import brute_scores_row, np_bf16, small_spec
from gpu_helpers import Dev, assert_attn_parity, assert_index_parity

pytestmark = pytest.mark.gpu


def _full_check(case, explicit_rows=True, attn_rows=None):
    dev = Dev(case)
    idx = dev.indexer(explicit_rows=explicit_rows)
    assert dev.faults() == 0
    exact = assert_index_parity(case, idx)
    out, lse = dev.attn(idx)
    assert dev.faults() == 0
    assert_attn_parity(case, idx, out, lse, rows=attn_rows)
    return dev, idx, out, lse, exact


# ------------------------------------------------------------------ fp32 (CUDA-core kernels)

def test_tiny_decode_f32_workload():
    spec, seed = W.named(1)
    case = W.generate(spec, seed)
    dev, idx, out, lse, _ = _full_check(case)
    didx, dout, dlse = dev.decode()
    assert np.array_equal(didx, idx)
    assert np.array_equal(dout, out)


def test_f32_ragged_lengths():
    spec = small_spec("f32", [0, 1, 63, 64, 65, 127, 128, 129, 300, 2500], 256)
    case = W.generate(spec, seed=101)
    _full_check(case)


def test_f32_prefill_rows():
    spec = small_spec("f32", [700, 260], 64, new_tokens=[33, 9])
    case = W.generate(spec, seed=102)
    _full_check(case)


# ------------------------------------------------------------------ small shapes, bf16 / FP8 keys

@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8"])
def test_small_heads_bf16_modes(mode):
    spec = small_spec(mode, [5, 64, 200, 1000], 96, H_I=8, d_I=32, H=4, d=64, d_v=48)
    case = W.generate(spec, seed=103)
    _full_check(case)


# ------------------------------------------------------------------ full head shapes, tensor cores

def test_tc_ragged_lengths_k2048():
    spec = small_spec("bf16", [1, 64, 129, 2047, 2048, 2049, 5000], 2048)
    case = W.generate(spec, seed=104)
    dev, idx, out, lse, _ = _full_check(case)
    didx, dout, dlse = dev.decode()
    assert np.array_equal(didx, idx)
    assert np.array_equal(dout, out)


def test_tc_k256_several_tiles():
    spec = small_spec("bf16", [300, 1000, 4097], 256)
    case = W.generate(spec, seed=105)
    _full_check(case)


def test_tc_prefill_rows():
    spec = small_spec("bf16", [3000, 1500], 512, new_tokens=[24, 9])
    case = W.generate(spec, seed=106)
    _full_check(case)


def test_tc_negative_head_weights():
    spec = small_spec("bf16", [3000, 700], 256)
    case = W.generate(spec, seed=107)
    case.w = (case.w - 0.5).astype(np.float32)
    _full_check(case)


def test_fp8_keys_full_heads():
    spec = small_spec("bf16_kfp8", [100, 3000], 512)
    case = W.generate(spec, seed=108)
    _full_check(case)


def test_planted_sets_are_exact():
    """Planted data makes the K-th gap large, so the exact branch of the index rule must hold."""
    spec = small_spec("bf16", [6000, 4500, 3000], 512)
    case = W.generate(spec, seed=109)
    rng = np.random.default_rng(7)
    bs = spec.block_size
    planted = []
    for t in range(spec.T):
        L = int(case.seq_lens[t])
        P = np.sort(rng.choice(L, size=spec.K, replace=False))
        u = (case.w[t][:, None].astype(np.float64) * np_bf16(case.q_I[t])).sum(0)
        u /= np.linalg.norm(u)
        for s in P:
            blk, off = case.block_table[t, s // bs], s % bs
            k = np_bf16(case.k_I[blk, off]) + 30.0 * u
            case.k_I[blk, off] = W.to_bf16_bits(k.astype(np.float32))
        planted.append(P)
    dev = Dev(case)
    idx = dev.indexer()
    exact = assert_index_parity(case, idx)
    assert exact == spec.T
    for t in range(spec.T):
        assert idx[t].tolist() == planted[t].tolist()


def test_duplicated_keys_break_ties_to_lower_position():
    spec = small_spec("bf16", [1500], 256)
    case = W.generate(spec, seed=110)
    rng = np.random.default_rng(8)
    bs = spec.block_size
    # one strong key copied to 400 random positions: exact ties, Top-K = its 256 lowest positions
    u = (case.w[0][:, None].astype(np.float64) * np_bf16(case.q_I[0])).sum(0)
    strong = W.to_bf16_bits((40.0 * u / np.linalg.norm(u)).astype(np.float32))
    P = np.sort(rng.choice(1500, size=400, replace=False))
    for s in P:
        case.k_I[case.block_table[0, s // bs], s % bs] = strong
    S = brute_scores_row(case, 0)
    assert np.all(S[P] == S[P[0]]) and S[P[0]] > np.delete(S, P).max()
    dev = Dev(case)
    idx = dev.indexer()
    assert idx[0].tolist() == P[:256].tolist()


def test_repaging_is_bit_identical():
    spec = small_spec("bf16", [2500, 900, 4100], 512)
    case = W.generate(spec, seed=111)
    other = W.repage(case, seed=112)
    a = Dev(case)
    b = Dev(other)
    ia, ib = a.indexer(), b.indexer()
    assert np.array_equal(ia, ib)
    oa, la = a.attn(ia)
    ob, lb = b.attn(ib)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_split_count_does_not_change_results():
    """Row 0 alone (many splits + combine) vs. inside a batch of 80 rows (one split per row)."""
    spec1 = small_spec("bf16", [3000], 2048)
    case1 = W.generate(spec1, seed=113)
    d1 = Dev(case1)
    idx1 = d1.indexer()
    out1, lse1 = d1.attn(idx1)
    specn = small_spec("bf16", [3000] * 80, 2048)
    casen = W.generate(specn, seed=113)
    casen.block_table[:] = case1.block_table[0]
    casen.k_I[: case1.num_blocks], casen.kv[: case1.num_blocks] = case1.k_I, case1.kv
    casen.q_I[:], casen.q[:], casen.w[:] = case1.q_I[0], case1.q[0], case1.w[0]
    dn = Dev(casen)
    idxn = np.repeat(idx1, 80, axis=0)
    outn, lsen = dn.attn(idxn)
    assert np.abs(outn[0] - out1[0]).max() <= 2e-2
    assert np.abs(lsen[0] - lse1[0]).max() <= 1e-3
    assert_attn_parity(case1, idx1, out1, lse1)


def test_long_rows_merge_through_the_group_tree():
    """A row whose tiles span ~130 indexer CTAs (17 merge groups, merged by the row's last group),
    one spanning ~18 (3 groups) and a short one (1 group)."""
    spec = small_spec("bf16", [150000, 3000, 20000], 2048)
    case = W.generate(spec, seed=116)
    _full_check(case, attn_rows=np.arange(3))


def test_long_row_fp8_keys_k512():
    spec = small_spec("bf16_kfp8", [90000, 400], 512)
    case = W.generate(spec, seed=117)
    _full_check(case)


def test_prefill_groups_on_the_score_gemm():
    """Rows 0-7 and 8-11 form groups of four rows of one sequence (score GEMM + per-row Top-K,
    rows longer than the 8192-key candidate buffer: sampled admission threshold); row 12 is left
    over for the decode kernels."""
    spec = small_spec("bf16", [12000, 9000], 2048, new_tokens=[8, 5])
    case = W.generate(spec, seed=118)
    _full_check(case, attn_rows=np.array([0, 7, 8, 12]))


def test_prefill_gemm_fp8_keys_and_mixed_groups():
    """FP8 keys; decode rows first, so the first groups mix sequences (decode path) and the
    chunk's groups run on the score GEMM."""
    spec = small_spec("bf16_kfp8", [700, 5000, 20000, 10000], 1024, new_tokens=[1, 1, 1, 14])
    case = W.generate(spec, seed=119)
    _full_check(case, attn_rows=np.array([0, 2, 3, 16]))


def test_prefill_gemm_equal_scores_take_the_lowest_positions():
    """Zero queries give every key the score 0: the admission threshold admits the whole row,
    which overflows the candidate buffer, and the exact streaming selection must return the K
    lowest positions (ties go to the lower position)."""
    spec = small_spec("bf16", [20000], 2048, new_tokens=[4])
    case = W.generate(spec, seed=120)
    case.q_I[:] = W.to_bf16_bits(np.zeros(case.q_I.shape, np.float32))
    dev = Dev(case)
    idx = dev.indexer()
    assert dev.faults() == 0
    for t in range(spec.T):
        assert idx[t].tolist() == list(range(2048))


# ------------------------------------------------------------------ the named workloads at full size

def test_decode_bf16_b32_full_size():
    spec, seed = W.named(2)
    case = W.generate(spec, seed)
    dev, idx, out, lse, _ = _full_check(case, explicit_rows=False)  # every row: indices and attention
    didx, dout, dlse = dev.decode()
    assert np.array_equal(didx, idx)
    assert np.array_equal(dout, out)


# ------------------------------------------------------------------ device-side guards

def test_bad_block_table_entry_is_reported_not_faulted():
    spec = small_spec("bf16", [700, 900], 256)
    case = W.generate(spec, seed=114)
    case.block_table[1, 3] = case.num_blocks + 5
    dev = Dev(case)
    idx = dev.indexer()
    assert dev.faults() & 0x1
    assert np.all(idx[0] >= -1)


def test_bad_index_is_reported_not_faulted():
    spec = small_spec("bf16", [700], 256)
    case = W.generate(spec, seed=115)
    dev = Dev(case)
    idx = dev.indexer()
    idx[0, 5] = 10_000
    out, lse = dev.attn(idx)
    assert dev.faults() & 0x2
    assert np.all(np.isfinite(out))
