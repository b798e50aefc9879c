"""Parity of hierarchical (coarse -> fine) selection through the C ABI with the oracle:
block summaries bit for bit; the coarse block choice under the index rule of the indexer
(the summaries are identical, so the coarse problem is the same); the fine choice against the
oracle inside the chosen blocks wherever the two block sets agree; the all-blocks case equals
the exact indexer; a planted block is found."""
import numpy as np
import pytest
import torch

import indexer_top_sparse_paged_gb300 as dsa
import oracle
import workloads as W
from cases import REL_GAP, np_bf16, small_spec
from gpu_helpers import Dev, assert_index_parity

pytestmark = pytest.mark.gpu


def _gpu_summaries(dev, case):
    summ = dsa.summaries_buffer(dev.dims)
    dsa.block_summaries(dev.dims, dev.k_I, dev.k_I_scale, dev.block_table, dev.seq_lens, summ, ws=dev.ws)
    torch.cuda.synchronize()
    assert dsa.read_error(dev.ws) == 0
    return summ


def _gpu_hier(dev, case, summ, n_sel, explicit_rows=True):
    ws = dsa.hier_workspace(dev.dims, case.spec.T, n_sel)
    kw = dict(q_seq=dev.q_seq, q_pos=dev.q_pos) if explicit_rows else {}
    idx, blocks = dsa.indexer_topk_hier(dev.dims, dev.q_I, dev.w, dev.k_I, dev.k_I_scale, dev.block_table,
                                        dev.seq_lens, summ, n_sel, ws=ws, **kw)
    torch.cuda.synchronize()
    assert dsa.read_error(ws) == 0
    return idx.cpu().numpy(), blocks.cpu().numpy()


@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8", "mxfp8"])
def test_block_summaries_bit_exact(mode):
    spec = small_spec(mode, [1, 63, 64, 65, 700, 5000], 64)
    case = W.generate(spec, seed=501)
    dev = Dev(case)
    summ = _gpu_summaries(dev, case).view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.block_summaries(case)
    assert np.array_equal(summ[:, : case.max_blocks], ref)


def _check_fine(case, t, gpu_row, oracle_blocks, S_row, K):
    """The GPU's fine set against the oracle's scores inside the chosen blocks (index rule)."""
    n = int(case.q_pos[t]) + 1
    pos = np.concatenate([np.arange(b * 64, min(b * 64 + 64, n)) for b in oracle_blocks])
    g = gpu_row[gpu_row >= 0]
    assert np.all(np.diff(g) > 0) and np.all(gpu_row[len(g):] == -1)
    assert set(g.tolist()) <= set(pos.tolist()), "position outside the chosen blocks"
    if len(pos) <= K:
        assert set(g.tolist()) == set(pos.tolist())
        return True
    sc = S_row[pos]
    srt = np.sort(sc)[::-1]
    sk, sk1 = srt[K - 1], srt[K]
    tau = REL_GAP * (abs(sk) if sk != 0 else 1.0)
    assert len(g) == K
    must = pos[sc > sk + tau]
    assert set(must.tolist()) <= set(g.tolist())
    assert np.all(S_row[g] >= sk - tau)
    return (sk - sk1) / (abs(sk) if sk else 1.0) > REL_GAP


@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8", "mxfp8"])
def test_hierarchical_decode_and_prefill_rows(mode):
    spec = small_spec(mode, [20000, 9000, 3000, 700, 16384], 512, new_tokens=[1, 1, 6, 1, 9])
    case = W.generate(spec, seed=502 if mode == "bf16" else 503)
    n_sel = 24
    dev = Dev(case)
    summ = _gpu_summaries(dev, case)
    idx, blocks = _gpu_hier(dev, case, summ, n_sel)
    # coarse: the summary problem is identical on both sides (bit-exact summaries)
    c2 = oracle.summary_case(case, oracle.block_summaries(case), n_sel)
    assert_index_parity(c2, blocks)
    o_idx, o_blocks = oracle.hierarchical_topk(case, n_sel)
    S = oracle.index_scores(case)
    same = 0
    for t in range(spec.T):
        gb = blocks[t][blocks[t] >= 0]
        ob = o_blocks[t][o_blocks[t] >= 0]
        if gb.tolist() != ob.tolist():
            continue  # a near tie in the coarse stage (allowed by the index rule above)
        same += 1
        _check_fine(case, t, idx[t], ob, S[t], spec.K)
    assert same >= spec.T - 2


def test_all_blocks_kept_equals_the_exact_indexer():
    spec = small_spec("bf16", [3000, 5000, 65], 512)
    case = W.generate(spec, seed=504)
    dev = Dev(case)
    summ = _gpu_summaries(dev, case)
    idx, blocks = _gpu_hier(dev, case, summ, n_sel=100, explicit_rows=False)
    exact = dev.indexer(explicit_rows=False)
    assert np.array_equal(idx, exact)
    for t in range(spec.T):
        nb = (int(case.seq_lens[t]) + 63) // 64
        assert blocks[t][:nb].tolist() == list(range(nb)) and np.all(blocks[t][nb:] == -1)


def test_planted_block_is_found():
    spec = small_spec("bf16", [8000], 256)
    case = W.generate(spec, seed=505)
    u = (case.w[0][:, None].astype(np.float64) * np_bf16(case.q_I[0])).sum(0)
    u /= np.linalg.norm(u)
    blk = int(case.block_table[0, 40])
    case.k_I[blk] = W.to_bf16_bits((np_bf16(case.k_I[blk]) + 20.0 * u).astype(np.float32))
    dev = Dev(case)
    summ = _gpu_summaries(dev, case)
    idx, blocks = _gpu_hier(dev, case, summ, n_sel=1, explicit_rows=False)
    assert blocks[0].tolist() == [40]
    assert idx[0][:64].tolist() == list(range(40 * 64, 41 * 64)) and np.all(idx[0][64:] == -1)


@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8", "mxfp8"])
def test_summaries_follow_the_cache_append(mode):
    """Append new tokens (a decode token, a chunk crossing blocks), update only the touched
    blocks' summaries, and compare with the oracle's summaries of the oracle's appended cache."""
    spec = small_spec(mode, [700, 3000, 129], 256, new_tokens=[1, 150, 2])
    case = W.generate(spec, seed=506)
    dev = Dev(case)
    summ = _gpu_summaries(dev, case)
    rng = np.random.default_rng(507)
    k_new = W.to_bf16_bits(rng.standard_normal((spec.T, spec.d_I), dtype=np.float32) * 2.0)
    kv_new = W.to_bf16_bits(rng.standard_normal((spec.T, spec.d), dtype=np.float32))
    t_k = torch.from_numpy(k_new.view(np.int16)).cuda()
    t_kv = torch.from_numpy(kv_new.view(np.int16)).cuda()
    dsa.cache_append(dev.dims, t_k, t_kv, dev.block_table, dev.seq_lens, dev.k_I, dev.k_I_scale, dev.kv,
                     q_seq=dev.q_seq, q_pos=dev.q_pos, ws=dev.ws)
    dsa.block_summaries_append(dev.dims, dev.k_I, dev.k_I_scale, dev.block_table, dev.seq_lens, spec.T, summ,
                               q_seq=dev.q_seq, q_pos=dev.q_pos, ws=dev.ws)
    torch.cuda.synchronize()
    assert dsa.read_error(dev.ws) == 0
    k2, s2, kv2 = oracle.cache_append(case, k_new, kv_new)
    case.k_I, case.k_I_scale, case.kv = k2, s2, kv2
    got = summ.view(torch.int16).cpu().numpy().view(np.uint16)[:, : case.max_blocks]
    assert np.array_equal(got, oracle.block_summaries(case))
