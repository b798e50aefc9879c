"""Pins for the oracle's hierarchical (coarse -> fine) selection: block summaries against a
sequential NumPy fp32 sum and torch's bf16 cast; the whole method against a NumPy brute force;
the invariant that keeping every block reproduces the exact Top-K; a planted case."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from cases import brute_scores_row, logical_rows, np_bf16, np_e4m3, np_mx, small_spec


def np_summaries(case):
    s = case.spec
    out = np.zeros((s.B, case.max_blocks, s.d_I), np.uint16)
    for b in range(s.B):
        L = int(case.seq_lens[b])
        for lb in range((L + 63) // 64):
            blk = int(case.block_table[b, lb])
            cnt = min(64, L - lb * 64)
            if s.mode == "f32":
                x = case.k_I[blk, :cnt].astype(np.float32)
            elif s.mode == "bf16":
                x = np_bf16(case.k_I[blk, :cnt]).astype(np.float32)
            elif s.mode == "mxfp8":
                x = np_mx(case.k_I[blk, :cnt], case.k_I_scale[blk, :cnt]).astype(np.float32)
            else:
                x = (np_e4m3(case.k_I[blk, :cnt]).astype(np.float32) * np.float32(case.k_I_scale[blk])).astype(np.float32)
            acc = np.zeros(s.d_I, np.float32)
            for i in range(cnt):
                acc = (acc + x[i]).astype(np.float32)
            mean = (acc / np.float32(cnt)).astype(np.float32)
            out[b, lb] = torch.from_numpy(mean).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out


@pytest.mark.parametrize("mode", ["f32", "bf16", "bf16_kfp8", "mxfp8"])
def test_summaries_match_sequential_numpy_mean(mode):
    spec = small_spec(mode, [1, 63, 64, 65, 300], 64, H_I=4, d_I=64) if mode != "f32" else small_spec(mode, [1, 63, 64, 65, 300], 64)
    case = W.generate(spec, seed=401)
    assert np.array_equal(oracle.block_summaries(case), np_summaries(case))


def _brute_hier(case, t, n_sel):
    s = case.spec
    b, n = int(case.q_seq[t]), int(case.q_pos[t]) + 1
    summ = np_bf16(np_summaries(case)[b, : (n + 63) // 64])            # [nb, d_I]
    q = np_bf16(case.q_I[t]) if s.mode != "f32" else case.q_I[t].astype(np.float64)
    w = case.w[t].astype(np.float64)
    bsc = w @ np.maximum(q @ summ.T, 0.0)
    border = np.lexsort((np.arange(len(bsc)), -bsc))[:n_sel]
    blocks = np.sort(border)
    S = brute_scores_row(case, t)
    pos = np.concatenate([np.arange(bb * 64, min(bb * 64 + 64, n)) for bb in blocks])
    order = np.lexsort((pos, -S[pos]))[: s.K]
    return np.sort(pos[order]), blocks


@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8", "mxfp8"])
def test_hierarchical_matches_brute_force(mode):
    spec = small_spec(mode, [700, 2000, 130], 96, H_I=4, d_I=32, new_tokens=[1, 3, 1])
    case = W.generate(spec, seed=402)
    idx, blocks = oracle.hierarchical_topk(case, n_sel=5)
    for t in range(spec.T):
        bi, bb = _brute_hier(case, t, 5)
        assert idx[t][idx[t] >= 0].tolist() == bi.tolist()
        assert blocks[t][blocks[t] >= 0].tolist() == bb.tolist()


def test_all_blocks_kept_reproduces_the_exact_topk():
    spec = small_spec("bf16", [3000, 777, 64], 256, H_I=8, d_I=32, new_tokens=[2, 1, 1])
    case = W.generate(spec, seed=403)
    idx, _ = oracle.hierarchical_topk(case, n_sel=64)
    exact, _ = oracle.indexer_topk(case)
    for t in range(spec.T):
        assert idx[t].tolist() == sorted(exact[t][exact[t] >= 0].tolist()) + [-1] * int((exact[t] < 0).sum())


def test_planted_block_is_chosen():
    """Block 7 of the sequence gets keys aligned with the query: n_sel = 1 keeps it alone."""
    spec = small_spec("bf16", [2000], 32, H_I=4, d_I=32)
    case = W.generate(spec, seed=404)
    u = (case.w[0][:, None].astype(np.float64) * np_bf16(case.q_I[0])).sum(0)
    u /= np.linalg.norm(u)
    blk = int(case.block_table[0, 7])
    case.k_I[blk] = W.to_bf16_bits((np_bf16(case.k_I[blk]) + 20.0 * u).astype(np.float32))
    idx, blocks = oracle.hierarchical_topk(case, n_sel=1)
    assert blocks[0].tolist() == [7]
    assert np.all((idx[0] >= 7 * 64) & (idx[0] < 8 * 64))


def test_equal_keys_take_the_lowest_blocks_and_positions():
    """Every key equal: all summaries score alike and so do all tokens, so the coarse stage keeps
    the lowest blocks and the fine stage the lowest positions, never past the row's own position
    (the 70-token sequence's rows have fewer causal tokens than K)."""
    spec = small_spec("bf16", [300, 200, 70], 100, new_tokens=[3, 2, 3], H_I=4, d_I=32)
    case = W.generate(spec, seed=405)
    case.k_I[...] = 0x3F80  # bf16 1.0
    n_sel = 2
    idx, blocks = oracle.hierarchical_topk(case, n_sel=n_sel)
    short_rows = 0
    for t in range(spec.T):
        n = int(case.q_pos[t]) + 1
        nb = min(n_sel, (n + 63) // 64)
        assert blocks[t].tolist() == list(range(nb)) + [-1] * (n_sel - nb)
        m = min(spec.K, nb * 64, n)
        short_rows += m < spec.K
        assert idx[t].tolist() == list(range(m)) + [-1] * (spec.K - m)
    assert short_rows == 3


def test_block_past_the_row_is_never_chosen():
    """Every row has the same query and block 4 (positions 256..299) is given keys aligned with it:
    with n_sel = 1 the rows at positions 256.. choose block 4, and the rows before it, for which
    that block lies past their causal limit, choose another."""
    spec = small_spec("bf16", [300], 16, new_tokens=[100], H_I=4, d_I=32)
    case = W.generate(spec, seed=406)
    case.q_I[:] = case.q_I[0]
    case.w[:] = case.w[0]
    u = (case.w[0][:, None].astype(np.float64) * np_bf16(case.q_I[0])).sum(0)
    u /= np.linalg.norm(u)
    blk = int(case.block_table[0, 4])
    case.k_I[blk] = W.to_bf16_bits((np_bf16(case.k_I[blk]) + 20.0 * u).astype(np.float32))
    idx, blocks = oracle.hierarchical_topk(case, n_sel=1)
    pos = case.q_pos.astype(int)
    assert np.all(blocks[pos >= 256, 0] == 4)
    assert np.all(blocks[pos < 256, 0] <= pos[pos < 256] // 64)
    assert np.all(idx[pos < 256] < 256)
    assert (pos < 256).sum() == 56 and (pos >= 256).sum() == 44
