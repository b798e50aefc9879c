"""Parity at the full sizes of the long-context, prefill and mixed workloads (through the C ABI).

The GPU computes every row; the fp64 oracle checks a sample of rows (it scores one row of a
1M-token context in seconds, so all decode rows and a spread of prefill rows are checked):

* 1M-token decode with FP8 e4m3 indexer keys (one fp32 scale per 64-token block);
* chunked prefill, 2 x 4096 new tokens on a 61,440-token cached prefix (64K in total);
* a mixed serving batch: 64 decode rows (contexts log-uniform in [1K, 256K]) plus one
  2048-token prefill chunk at 128K, FP8 keys;
* the chunked prefill with an MXFP8 indexer (MX keys, MX-quantised queries).

Index sets follow the same rule as the other parity tests (exact where the oracle's K-th gap
exceeds 1e-3 relative, else the 1e-3 band); attention is compared with the oracle evaluated on
the GPU's own index sets, max-abs 2e-2 (bf16 outputs).
"""
import dataclasses

import numpy as np
import pytest

import workloads as W
from gpu_helpers import Dev, assert_attn_parity, assert_index_parity

pytestmark = pytest.mark.gpu


def _check_rows(case, rows, decode_shaped=False):
    dev = Dev(case)
    idx = dev.indexer(explicit_rows=not decode_shaped)
    assert dev.faults() == 0
    assert np.all(idx >= -1)
    assert_index_parity(case, idx, rows=rows)
    out, lse = dev.attn(idx)
    assert dev.faults() == 0
    assert np.all(np.isfinite(out))
    assert_attn_parity(case, idx, out, lse, rows=rows)
    return dev, idx, out, lse


def test_decode_1m_fp8_keys_full_size():
    spec, seed = W.named(3)
    case = W.generate(spec, seed)
    dev, idx, out, lse = _check_rows(case, [0], decode_shaped=True)
    didx, dout, _ = dev.decode()
    assert np.array_equal(didx, idx)
    assert np.array_equal(dout, out)


def _spread_rows(lo: int, hi: int, n: int) -> np.ndarray:
    """n rows spread over [lo, hi): both ends, and every position inside a group of four rows
    (the prefill path scores rows 4g..4g+3 together) in turn."""
    base = np.linspace(lo, hi - 4, n).astype(np.int64) // 4 * 4
    rows = base + np.arange(n) % 4
    return np.unique(np.concatenate([[lo, lo + 1, hi - 2, hi - 1], rows]))


def test_chunked_prefill_2x4096_full_size():
    spec, seed = W.named(4)
    case = W.generate(spec, seed)
    T = spec.T
    # 2 x 68 rows: both ends of each chunk and every position inside a group of four
    rows = np.concatenate([_spread_rows(0, T // 2, 64), _spread_rows(T // 2, T, 64)])
    assert len(rows) >= 128 and set((rows % 4).tolist()) == {0, 1, 2, 3}
    _check_rows(case, rows)


def test_mixed_serving_batch_full_size():
    spec, seed = W.named(5)
    case = W.generate(spec, seed)
    n_dec = 64
    # every decode row and 68 rows of the 2048-row chunk (both ends, every group position)
    chunk = _spread_rows(n_dec, spec.T, 64)
    assert len(chunk) >= 64
    _check_rows(case, np.concatenate([np.arange(n_dec), chunk]))


@pytest.mark.parametrize("mode", ["bf16", "mxfp8"])
def test_chunked_prefill_shrunk_every_row(mode):
    """The chunked prefill shape shrunk to 2 x 256 new tokens on a 1024-token cached prefix (1280
    in total): every row's index set and attention against the oracle."""
    spec = W.prefill_chunk(B=2, new=256, total=1280, mode=mode)
    case = W.generate(spec, seed=40)
    _check_rows(case, np.arange(spec.T))


def test_chunked_prefill_2x4096_mxfp8_full_size():
    spec, seed = W.named(4)
    case = W.generate(dataclasses.replace(spec, mode="mxfp8"), seed)
    T = spec.T
    rows = np.concatenate([_spread_rows(0, T // 2, 16), _spread_rows(T // 2, T, 16)])
    _check_rows(case, rows)
