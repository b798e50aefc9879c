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


def test_chunked_prefill_2x4096_full_size():
    spec, seed = W.named(4)
    case = W.generate(spec, seed)
    T = spec.T
    # first, last and interior rows of both chunks (every row of the sample has > K positions)
    rows = np.unique(np.concatenate([np.linspace(0, T // 2 - 1, 7), np.linspace(T // 2, T - 1, 7)]).astype(np.int64))
    _check_rows(case, rows)


def test_mixed_serving_batch_full_size():
    spec, seed = W.named(5)
    case = W.generate(spec, seed)
    n_dec = 64
    rows = np.concatenate([np.arange(n_dec), n_dec + np.linspace(0, spec.T - n_dec - 1, 8).astype(np.int64)])
    _check_rows(case, rows)


def test_chunked_prefill_2x4096_mxfp8_full_size():
    spec, seed = W.named(4)
    case = W.generate(dataclasses.replace(spec, mode="mxfp8"), seed)
    T = spec.T
    rows = np.array([0, 1, 2047, T // 2 - 1, T // 2, T // 2 + 3001, T - 1])
    _check_rows(case, rows)
