"""dsa_indexer_topk_noalloc: the indexer + Top-K with the library's static scratch gives the same
indices as dsa_indexer_topk with a caller workspace, call after call, and rejects calls that do
not fit the static buffer. Named to be collected last; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import indexer_top_sparse_paged_gb300 as dsa
import workloads as W
from cases import small_spec
from gpu_helpers import Dev, assert_index_parity

pytestmark = pytest.mark.gpu


def _noalloc(dev: Dev, fault_word=None):
    idx = dsa.indexer_topk_noalloc(dev.dims, dev.q_I, dev.w, dev.k_I, dev.k_I_scale, dev.block_table,
                                   dev.seq_lens, dev.q_seq, dev.q_pos, fault_word=fault_word)
    torch.cuda.synchronize()
    return idx.cpu().numpy()


@pytest.mark.parametrize("which", ["tc_ragged", "simt_fp8", "decode_b32", "tc_mxfp8"])
def test_noalloc_matches_workspace_call_twice(which):
    if which == "tc_ragged":
        case = W.generate(small_spec("bf16", [3000, 130, 2049, 64], 2048), seed=301)
    elif which == "tc_mxfp8":
        case = W.generate(small_spec("mxfp8", [1500, 700, 64], 512), seed=305)
    elif which == "simt_fp8":
        case = W.generate(small_spec("bf16_kfp8", [1500, 700], 512, H_I=64, d_I=128), seed=302)
    else:
        spec, seed = W.named(2)
        case = W.generate(spec, seed)
    dev = Dev(case)
    ref = dev.indexer()
    ref_launches = dsa.last_launch_count()
    assert dev.faults() == 0
    fw = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    first = _noalloc(dev, fw)
    assert int(fw.item()) == 0
    second = _noalloc(dev)
    # same kernels, same work plan: the index sets are identical, not just within tolerance
    assert np.array_equal(first, ref)
    assert np.array_equal(second, ref)
    assert dsa.last_launch_count() == ref_launches  # the same kernels as the workspace call


def test_noalloc_prefill_shaped_rows_match_the_oracle():
    """Several causal rows of one sequence (a chunk of new tokens): the workspace call scores them
    on the prefill path, the call without a workspace on the decode kernels; both must follow the
    oracle's index rule row by row."""
    case = W.generate(small_spec("bf16", [3000, 2000], 512, new_tokens=[16, 8]), seed=306)
    dev = Dev(case)
    fw = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    idx = _noalloc(dev, fw)
    assert int(fw.item()) == 0
    assert_index_parity(case, idx)
    assert_index_parity(case, dev.indexer())


def test_noalloc_reports_faults_in_the_callers_word():
    case = W.generate(small_spec("bf16", [700, 900], 256), seed=303)
    case.block_table[1, 3] = case.num_blocks + 5
    dev = Dev(case)
    fw = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = _noalloc(dev, fw)
    assert int(fw.item()) & 0x1
    assert np.all(idx[0] >= -1)
    # the next clean call starts from a cleared error word
    case2 = W.generate(small_spec("bf16", [700, 900], 256), seed=304)
    dev2 = Dev(case2)
    _noalloc(dev2, fw)
    assert int(fw.item()) == 0


def test_noalloc_rejects_calls_over_the_static_limit():
    # valid device buffers for a call that needs more scratch than the static buffer holds: the
    # call must return DSA_ERR_TOO_LARGE and leave idx untouched
    T, K = 1024, 2048
    dims = dsa.make_dims("bf16", T, 1, 1, 64, 128, 128, 576, 512, K)
    assert dsa.workspace_size(dims, T) > 16 << 20
    q_I = torch.zeros((T, 64, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((T, 64), dtype=torch.float32, device="cuda")
    k_I = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((T, 1), dtype=torch.int32, device="cuda")
    sl = torch.full((T,), 64, dtype=torch.int32, device="cuda")
    idx = torch.full((T, K), 7, dtype=torch.int32, device="cuda")
    with pytest.raises(dsa.DsaError) as e:
        dsa.indexer_topk_noalloc(dims, q_I, w, k_I, None, bt, sl, idx=idx)
    assert e.value.status == 7
    assert b"static" in dsa.lib().dsa_status_string(7)
    torch.cuda.synchronize()
    assert bool((idx == 7).all())
