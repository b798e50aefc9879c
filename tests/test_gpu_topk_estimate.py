"""The decode indexer's sample estimates (each long segment of a row raises its admission
threshold to an estimate of the row's K-th key taken from its first tiles) and their check: when
a segment's sample is not representative of the row, the merge finds fewer than K candidates at or
above the estimates and recomputes the row exactly. Both outcomes must match the fp64 oracle.

The planted rows put keys with very large scores in the first two tiles of a 200,000-key row, so
the first segment's estimate (the r-th largest of its first four tiles, r far below the 256
planted keys) lies far above the row's K-th key and that segment turns away the ordinary keys
that belong to the row's Top-K."""
import numpy as np
import pytest

import indexer_top_sparse_paged_gb300 as dsa
import workloads as W
from cases import np_bf16, small_spec
from gpu_helpers import Dev, assert_index_parity

pytestmark = pytest.mark.gpu


def _planted_front(case, n_front: int = 256, alpha: float = 30.0):
    bs = case.spec.block_size
    for t in range(case.spec.T):
        u = (case.w[t][:, None].astype(np.float64) * np_bf16(case.q_I[t])).sum(0)
        u /= np.linalg.norm(u)
        for s in range(n_front):
            blk, off = case.block_table[t, s // bs], s % bs
            k = np_bf16(case.k_I[blk, off]) + alpha * u
            case.k_I[blk, off] = W.to_bf16_bits(k.astype(np.float32))
    return case


@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8", "mxfp8"])
def test_unrepresentative_sample_is_recomputed_exactly(mode):
    case = _planted_front(W.generate(small_spec("bf16", [200000], 2048), seed=130))
    if mode != "bf16":
        case = W.with_key_format(case, mode)
    dev = Dev(case)
    idx = dev.indexer(explicit_rows=False)
    assert dev.faults() == 0
    assert_index_parity(case, idx)
    assert np.all(idx[0, :256] == np.arange(256))  # the planted keys are all in the Top-K


def test_estimates_on_rows_of_many_lengths():
    """Rows of 3K to 120K keys (estimates with small and large margins, one to ~7 segments, rows
    too short to be sampled) next to each other in one call."""
    lens = [3000, 7000, 12000, 25000, 40000, 64000, 120000, 2100, 9000]
    case = W.generate(small_spec("bf16", lens, 2048), seed=131)
    dev = Dev(case)
    idx = dev.indexer(explicit_rows=False)
    assert dev.faults() == 0
    assert_index_parity(case, idx)


def _planted_segment_start(case, n_front: int = 256, alpha: float = 30.0):
    """Plant keys with very large scores in the first two tiles of a segment that starts inside a row
    (the indexer CTAs split all rows' 128-key tiles evenly, CTA c owning tiles [c*total/G,
    (c+1)*total/G)), in a row whose lists one merge group takes (at most 8 CTAs)."""
    import torch
    G = torch.cuda.get_device_properties(0).multi_processor_count
    n = case.q_pos.astype(np.int64) + 1
    tiles = (n + 127) // 128
    prefix = np.concatenate([[0], np.cumsum(tiles)])
    total = int(prefix[-1])
    tb = lambda c: c * total // G
    for c in range(1, G):
        x = tb(c)
        t = int(np.searchsorted(prefix, x, side="right") - 1)
        p0, p1 = int(prefix[t]), int(prefix[t + 1])
        owners = ((p1 - 1 + 1) * G - 1) // total - ((p0 + 1) * G - 1) // total + 1
        if x > p0 and min(tb(c + 1), p1) - x >= 16 and owners <= 8:  # a segment long enough to be sampled
            s0 = (x - p0) * 128
            bs = case.spec.block_size
            u = (case.w[t][:, None].astype(np.float64) * np_bf16(case.q_I[t])).sum(0)
            u /= np.linalg.norm(u)
            for s in range(s0, s0 + n_front):
                blk, off = case.block_table[t, s // bs], s % bs
                k = np_bf16(case.k_I[blk, off]) + alpha * u
                case.k_I[blk, off] = W.to_bf16_bits(k.astype(np.float32))
            return t
    raise AssertionError("no segment to plant in")


def test_segment_with_an_unrepresentative_sample_inside_a_batch():
    """A batch of decode rows like the batch-32 workload; one row's segment (not the row's first)
    starts with planted keys, the row's estimate check fails in the merge and the row is rescored;
    every row matches the oracle."""
    rng = np.random.default_rng(132)
    lens = [int(x) for x in rng.integers(16384, 32768, size=32)]
    case = W.generate(small_spec("bf16", lens, 2048), seed=132)
    t = _planted_segment_start(case)
    dev = Dev(case)
    idx = dev.indexer(explicit_rows=False)
    assert dev.faults() == 0
    assert_index_parity(case, idx)
    idx2 = dev.indexer(explicit_rows=False)  # the next call on the same workspace is the same
    assert np.array_equal(idx, idx2)


def test_one_workspace_for_calls_of_different_row_counts():
    """Calls with 4, 32 and 4 rows (and a prefill-shaped call) sharing one workspace all match the
    oracle: nothing a call leaves in the workspace changes the next one's result."""
    rng = np.random.default_rng(133)
    big = W.generate(small_spec("bf16", [int(x) for x in rng.integers(3000, 20000, size=32)], 1024), seed=133)
    small = W.generate(small_spec("bf16", [9000, 12000, 700, 30000], 1024), seed=134)
    pre = W.generate(small_spec("bf16", [9000, 5000], 1024, new_tokens=[12, 5]), seed=135)
    devs = {id(c): Dev(c) for c in (small, big, pre)}
    ws = max((d.ws for d in devs.values()), key=lambda w: w.numel())  # the largest, shared by all calls
    for case in (small, big, pre, small, big):
        dev = devs[id(case)]
        assert dsa.workspace_size(dev.dims, case.spec.T) <= ws.numel()
        dev.ws = ws
        idx = dev.indexer(explicit_rows=case is pre)
        assert dev.faults() == 0
        assert_index_parity(case, idx)
