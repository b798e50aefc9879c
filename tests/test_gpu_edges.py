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
