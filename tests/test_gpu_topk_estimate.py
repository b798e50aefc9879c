"""The decode indexer's sample estimates (each long segment of a row raises its admission
threshold to an estimate of the row's K-th key taken from its first tiles) and their check: when
a segment's sample is not representative of the row, the merge finds fewer than K candidates at or
above the estimates and recomputes the row exactly. Both outcomes must match the fp64 oracle.

The planted rows put keys with very large scores in the first two tiles of a 200,000-key row, so
the first segment's estimate lies far above the row's K-th key and that segment turns away the
ordinary keys that belong to the row's Top-K."""
import numpy as np
import pytest

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
