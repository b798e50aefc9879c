"""MXFP8 indexer (OCP Microscaling, E4M3 elements, one E8M0 scale per 32) through the C ABI
against the fp64 oracle: the query quantisation kernel, the decode tensor-core indexer, the
CUDA-core indexer for small heads, the merge tree on a long row and the prefill score GEMM, with
per-group scales spread over a wide range; attention on the selected rows stays bf16."""
import numpy as np
import pytest

import workloads as W
from cases import small_spec
from gpu_helpers import Dev, assert_attn_parity, assert_index_parity

pytestmark = pytest.mark.gpu


def _full_check(case, attn_rows=None):
    dev = Dev(case)
    idx = dev.indexer()
    assert dev.faults() == 0
    assert_index_parity(case, idx)
    rows = np.arange(case.spec.T) if attn_rows is None else attn_rows
    out, lse = dev.attn(idx)
    assert dev.faults() == 0
    assert_attn_parity(case, idx, out, lse, rows=rows)
    return dev, idx


def _spread_scales(case, seed):
    """Key groups rescaled by 2^-6..2^6 (their E8M0 bytes), query groups by 2^-20..2^20, one
    query group per row set to zero: every group quantises with its own exponent."""
    rng = np.random.default_rng(seed)
    sc = case.k_I_scale.astype(np.int32) + rng.integers(-6, 7, size=case.k_I_scale.shape)
    case.k_I_scale = np.clip(sc, 1, 254).astype(np.uint8)
    q = W.bf16_bits_to_f32(case.q_I).reshape(case.spec.T, case.spec.H_I, -1, 32)
    q = q * np.exp2(rng.integers(-20, 21, size=q.shape[:3] + (1,))).astype(np.float32)
    q[:, 0, 0] = 0.0
    case.q_I = W.to_bf16_bits(q.reshape(case.q_I.shape))
    return case


def test_small_heads_simt():
    spec = small_spec("mxfp8", [5, 64, 200, 1000], 96, H_I=8, d_I=64, H=4, d=64, d_v=48)
    _full_check(W.generate(spec, seed=501))


def test_tc_decode_ragged_k512():
    spec = small_spec("mxfp8", [1, 64, 129, 2049, 5000], 512)
    dev, idx = _full_check(W.generate(spec, seed=502))
    didx, dout, dlse = dev.decode()
    assert np.array_equal(didx, idx)


def test_tc_decode_group_scales_spread():
    spec = small_spec("mxfp8", [3000, 700, 4500], 256)
    _full_check(_spread_scales(W.generate(spec, seed=503), 504))


def test_simt_group_scales_spread():
    spec = small_spec("mxfp8", [900, 2000], 128, H_I=16, d_I=96, H=4, d=64, d_v=48)
    _full_check(_spread_scales(W.generate(spec, seed=505), 506))


def test_long_row_k2048_merge_tree():
    spec = small_spec("mxfp8", [90000, 400], 2048)
    _full_check(W.generate(spec, seed=507), attn_rows=np.arange(2))


def test_prefill_gemm_and_mixed_groups():
    spec = small_spec("mxfp8", [700, 5000, 20000, 10000], 1024, new_tokens=[1, 1, 1, 14])
    _full_check(_spread_scales(W.generate(spec, seed=508), 509), attn_rows=np.array([0, 2, 3, 16]))


def test_misaligned_or_missing_scales_are_rejected():
    """The E8M0 scales are fetched with 16-byte bulk copies: a misaligned or missing scale pointer
    is an argument error (nothing is launched), not a fault."""
    import torch

    import indexer_top_sparse_paged_gb300 as dsa
    spec = small_spec("mxfp8", [300, 900], 256)
    dev = Dev(W.generate(spec, seed=510))
    shifted = torch.empty(dev.k_I_scale.numel() + 16, dtype=torch.uint8, device="cuda")[1:1 + dev.k_I_scale.numel()]
    shifted.copy_(dev.k_I_scale.reshape(-1))
    for bad in (shifted, None):
        with pytest.raises(dsa.DsaError) as e:
            dsa.indexer_topk(dev.dims, dev.q_I, dev.w, dev.k_I, bad, dev.block_table, dev.seq_lens, ws=dev.ws)
        assert e.value.status == 1
    assert dev.faults() == 0
