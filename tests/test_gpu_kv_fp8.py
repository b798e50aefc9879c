"""Sparse attention over an FP8 latent cache (DSA_KV_FP8: per token, e4m3 codes with one fp32 scale
per 128-element tile; "Day0 Inference Support ... on Huawei Ascend CANN Architecture" §3, FP8 block
quantisation in the attention stage), through the C ABI, against the fp64 oracle evaluated on the
GPU's own index sets: max-abs 2e-2 on the bf16 outputs, as for bf16 latent rows. The GPU widens
code * scale to bf16 before its tensor-core products; the oracle decodes exactly."""
import numpy as np
import pytest

import workloads as W
from cases import small_spec
from gpu_helpers import Dev, assert_attn_parity, assert_index_parity

pytestmark = pytest.mark.gpu


def _check(case, rows=None, decode_shaped=False):
    dev = Dev(case)
    idx = dev.indexer(explicit_rows=not decode_shaped)
    assert dev.faults() == 0
    assert_index_parity(case, idx, rows=rows)
    out, lse = dev.attn(idx)
    assert dev.faults() == 0
    assert np.all(np.isfinite(out))
    assert_attn_parity(case, idx, out, lse, rows=rows)
    return dev, idx, out, lse


@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8", "mxfp8"])
def test_tensor_core_shapes_ragged(mode):
    """128 heads over 576-wide records (four full tiles and one of 64), rows shorter and longer
    than K, one split and several."""
    spec = small_spec(mode, [1, 64, 700, 2049, 5000], 2048, kv="fp8")
    dev, idx, out, lse = _check(W.generate(spec, seed=220), decode_shaped=True)
    didx, dout, dlse = dev.decode()
    assert np.array_equal(didx, idx)
    assert np.array_equal(dout, out)


def test_tensor_core_single_row_many_splits():
    spec = small_spec("bf16", [3000], 2048, kv="fp8")
    _check(W.generate(spec, seed=221), decode_shaped=True)


def test_prefill_rows():
    spec = small_spec("bf16", [3000, 1500], 512, new_tokens=[24, 9], kv="fp8")
    _check(W.generate(spec, seed=222))


def test_prefill_rows_one_split_per_row():
    """Enough rows (T = 100) that every row gets one split of 16 tiles: the path without L2
    prefetches, where the producers copy every tile's codes between their sends."""
    spec = small_spec("bf16", [6000, 4500], 1024, new_tokens=[60, 40], kv="fp8")
    _check(W.generate(spec, seed=225), rows=list(range(0, 100, 7)))


def test_cuda_core_shapes():
    """Small head shapes run on the CUDA cores: a row of 80 elements is one partial tile, a row of
    272 two full tiles and one of 16."""
    spec = small_spec("bf16", [5, 64, 200, 1000], 96, H_I=8, d_I=32, H=4, d=80, d_v=48, kv="fp8")
    _check(W.generate(spec, seed=223))
    spec = small_spec("bf16", [300, 900], 64, H_I=8, d_I=32, H=4, d=272, d_v=200, kv="fp8")
    _check(W.generate(spec, seed=224))


def test_decode_bf16_b32_fp8_latent_full_size():
    """The batch-32 decode workload with its latent rows stored as FP8 records: every row."""
    spec, seed = W.named(2)
    case = W.with_kv_format(W.generate(spec, seed), "fp8")
    dev, idx, out, lse = _check(case, decode_shaped=True)
    didx, dout, _ = dev.decode()
    assert np.array_equal(didx, idx)
    assert np.array_equal(dout, out)
