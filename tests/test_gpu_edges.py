"""Edge cases of the tensor-core paths: a Top-K that is not a multiple of 64, prefill rows whose
causal prefix is shorter than K (all of it, then -1), a prefill group whose rows end inside the
same key tile, and a single-row call."""
import numpy as np
import pytest

import workloads as W
from cases import small_spec
from gpu_helpers import Dev, assert_attn_parity, assert_index_parity

pytestmark = pytest.mark.gpu


def _check(case, explicit_rows=True):
    dev = Dev(case)
    idx = dev.indexer(explicit_rows=explicit_rows)
    assert dev.faults() == 0
    assert_index_parity(case, idx)
    out, lse = dev.attn(idx)
    assert dev.faults() == 0
    assert_attn_parity(case, idx, out, lse)
    return idx


def test_decode_k_not_a_multiple_of_64():
    spec = small_spec("bf16", [50, 100, 101, 3000, 9000], 100)
    case = W.generate(spec, seed=601)
    _check(case, explicit_rows=False)


def test_prefill_k_100_and_short_prefixes():
    """A chunk starting at position 0: its first rows see fewer than K positions."""
    spec = small_spec("bf16", [160, 5000], 100, new_tokens=[160, 8])
    case = W.generate(spec, seed=602)
    idx = _check(case)
    assert idx[0].tolist() == [0] + [-1] * 99          # row at position 0: only itself
    assert idx[99].tolist() == list(range(100))         # 100 positions for K = 100


def test_prefill_group_ending_inside_one_tile():
    spec = small_spec("bf16_kfp8", [130, 70], 256, new_tokens=[4, 4])
    case = W.generate(spec, seed=603)
    _check(case)


def test_single_row_call():
    spec = small_spec("bf16", [4097], 2048)
    case = W.generate(spec, seed=604)
    _check(case, explicit_rows=False)


@pytest.mark.parametrize("mode,small", [("bf16", False), ("bf16_kfp8", False), ("mxfp8", False), ("bf16", True)])
def test_relu_zero_ties_at_the_boundary(mode, small):
    """Most keys score exactly 0 (every head's dot product is negative) and only 700 per sequence
    are positive, so the K-th key lies inside a tie of thousands of zero scores. The streaming
    selection has to resolve that tie exactly (ties to the lower position) instead of keeping the
    whole boundary bucket; the index sets must equal the oracle's."""
    kw = dict(H_I=8, d_I=32, H=4, d=64, d_v=48) if small else {}
    spec = small_spec(mode, [20000, 9000, 3000], 2048, **kw)
    case = W.generate(spec, seed=131)
    rng = np.random.default_rng(132)
    q = np.zeros((spec.T, spec.H_I, spec.d_I), np.float32)
    q[:, :, 0] = 1.0  # every head looks at key component 0
    case.q_I = W.to_bf16_bits(q)
    case.w[:] = 1.0
    pos_mask = np.zeros(case.k_I.shape[:2], bool)
    for b, L in enumerate(spec.seq_lens):
        for s in rng.choice(L, size=700, replace=False):
            pos_mask[case.block_table[b, s // 64], s % 64] = True
    if mode == "bf16":
        x = W.bf16_bits_to_f32(case.k_I)
        x[..., 0] = np.where(pos_mask, np.abs(x[..., 0]) + 0.25, -np.abs(x[..., 0]))
        case.k_I = W.to_bf16_bits(x)
    else:  # e4m3 codes: the sign bit of component 0
        c = case.k_I[..., 0]
        case.k_I[..., 0] = np.where(pos_mask, (c & 0x3F) | 0x08, c | 0x80)  # positive, finite, non-zero
    dev = Dev(case)
    idx = dev.indexer()
    assert dev.faults() == 0
    import oracle
    o_idx, _ = oracle.indexer_topk(case)
    for t in range(spec.T):
        assert idx[t].tolist() == sorted(int(v) for v in o_idx[t] if v >= 0) + [-1] * int((o_idx[t] < 0).sum())
