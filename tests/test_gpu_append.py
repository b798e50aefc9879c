"""Parity of dsa_cache_append (through the C ABI) with the oracle's append, byte for byte:
indexer-key caches (fp32 / bf16 copies, or FP8 codes with their block scales after the block
requantisation) and latent rows, for decode appends (one token per sequence) and prefill chunks
that cross block boundaries."""
import numpy as np
import pytest
import torch

import indexer_top_sparse_paged_gb300 as dsa
import oracle
import workloads as W
from cases import np_bf16, np_e4m3, small_spec

pytestmark = pytest.mark.gpu


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def _new_tokens(case, seed):
    rng = np.random.default_rng(seed)
    s = case.spec
    k = rng.standard_normal((s.T, s.d_I), dtype=np.float32) * 3.0
    v = rng.standard_normal((s.T, s.d), dtype=np.float32)
    if s.mode == "f32":
        return k, v
    return W.to_bf16_bits(k), W.to_bf16_bits(v)


def _gpu_append(case, k_new, kv_new, explicit_rows=True):
    s = case.spec
    dims = dsa.make_dims(s.mode, s.B, case.max_blocks, case.num_blocks, s.H_I, s.d_I, s.H, s.d, s.d_v, s.K, kv=s.kv)
    k_I, kv = _t(case.k_I), _t(case.kv)
    scale = _t(case.k_I_scale) if case.k_I_scale is not None else None
    ws = dsa.workspace(dims, 1)
    dsa.cache_append(dims, _t(k_new), _t(kv_new), _t(case.block_table), _t(case.seq_lens), k_I, scale, kv,
                     q_seq=_t(case.q_seq) if explicit_rows else None, q_pos=_t(case.q_pos) if explicit_rows else None,
                     ws=ws)
    torch.cuda.synchronize()
    assert dsa.read_error(ws) == 0
    out_k = k_I.cpu().numpy().view(case.k_I.dtype)
    out_kv = kv.cpu().numpy().view(case.kv.dtype)
    out_s = scale.cpu().numpy() if scale is not None else None
    return out_k, out_s, out_kv


def _check(case, seed, explicit_rows=True):
    k_new, kv_new = _new_tokens(case, seed)
    gk, gs, gkv = _gpu_append(case, k_new, kv_new, explicit_rows)
    ok, osc, okv = oracle.cache_append(case, k_new, kv_new)
    assert np.array_equal(gkv, okv), "latent rows differ"
    if osc is not None:
        bad = np.nonzero(gs.view(np.uint32) != osc.view(np.uint32))[0]
        assert len(bad) == 0, f"block scales differ at {bad[:5]}"
    diff = np.nonzero((gk != ok).reshape(gk.shape[0], -1).any(axis=1))[0]
    assert len(diff) == 0, f"indexer-key blocks differ: {diff[:5]}"


@pytest.mark.parametrize("mode", ["f32", "bf16", "bf16_kfp8", "mxfp8"])
def test_decode_append_one_token_per_sequence(mode):
    kw = dict(H_I=8, d_I=32, H=4, d=64, d_v=48) if mode == "f32" else {}
    spec = small_spec(mode, [1, 63, 64, 65, 128, 500, 2049], 64, **kw)
    case = W.generate(spec, seed=201)
    _check(case, 202, explicit_rows=False)


@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8", "mxfp8"])
def test_prefill_append_crosses_blocks(mode):
    spec = small_spec(mode, [300, 1000, 77, 4096], 64, new_tokens=[150, 1, 13, 200])
    case = W.generate(spec, seed=203)
    _check(case, 204)


def test_append_decode_bf16_b32_full_size():
    spec, seed = W.named(2)
    case = W.generate(spec, seed)
    _check(case, 205, explicit_rows=False)


def test_append_fp8_mixed_chunk():
    """The mixed serving workload's shapes at reduced size: decode rows and a 2048-token chunk."""
    spec = small_spec("bf16_kfp8", [1024, 3000, 9000, 16384], 64, new_tokens=[1, 1, 1, 2048])
    case = W.generate(spec, seed=206)
    _check(case, 207)


@pytest.mark.parametrize("mode", ["bf16", "bf16_kfp8"])
def test_append_fp8_latent_records(mode):
    """FP8 latent cache: every new row becomes one record (each 128-element tile quantised on its
    own, the scales after the codes, zero padding), byte for byte as the oracle writes it; decode
    appends and a chunk that crosses blocks, at the tensor-core row width (576) and a small one."""
    spec = small_spec(mode, [300, 1000, 77, 4096], 64, new_tokens=[150, 1, 13, 200], kv="fp8")
    _check(W.generate(spec, seed=208), 209)
    spec = small_spec(mode, [1, 64, 65, 700], 64, H=4, d=80, d_v=48, kv="fp8")
    _check(W.generate(spec, seed=210), 211, explicit_rows=False)


@pytest.mark.parametrize("mode", ["mxfp8", "bf16_kfp8"])
def test_indexer_prolog_is_the_append_and_the_query_quantisation_in_one_launch(mode):
    """dsa_indexer_prolog: the caches byte for byte as the oracle's append, the MX query (MXFP8) bit
    for bit as the oracle's OCP MX quantisation, one launch; the indexer fed the prepared query
    (DSA_Q_MX_READY) gives the same indices with one launch fewer."""
    spec = small_spec(mode, [300, 1000, 77, 4096], 256, new_tokens=[1, 1, 1, 1])
    case = W.generate(spec, seed=212)
    k_new, kv_new = _new_tokens(case, 213)
    s = case.spec
    dims = dsa.make_dims(s.mode, s.B, case.max_blocks, case.num_blocks, s.H_I, s.d_I, s.H, s.d, s.d_v, s.K)
    k_I, kv = _t(case.k_I), _t(case.kv)
    scale = _t(case.k_I_scale)
    ws = dsa.workspace(dims, s.T)
    q_I = _t(case.q_I).view(torch.bfloat16)
    mx = mode == "mxfp8"
    q_out = dsa.indexer_prolog(dims, _t(k_new).view(torch.bfloat16), _t(kv_new).view(torch.bfloat16),
                               _t(case.block_table), _t(case.seq_lens), k_I, scale, kv, q_I=q_I if mx else None, ws=ws)
    torch.cuda.synchronize()
    assert dsa.read_error(ws) == 0
    assert dsa.last_launch_count() == 1
    ok, osc, okv = oracle.cache_append(case, k_new, kv_new)
    assert np.array_equal(kv.cpu().numpy().view(case.kv.dtype), okv)
    assert np.array_equal(k_I.cpu().numpy().view(case.k_I.dtype), ok)
    assert np.array_equal(scale.cpu().numpy().view(osc.dtype), osc)
    if not mx:
        return
    # the query: every group of 32 quantised by the oracle, decoded exactly, as bf16 bits
    qf = np_bf16(case.q_I).astype(np.float32).reshape(-1, 32)
    want = np.empty_like(qf)
    for g in range(qf.shape[0]):
        X, codes = oracle.mx_quantize32(qf[g])
        want[g] = np_e4m3(codes) * 2.0 ** X
    got = q_out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1, 32)
    assert np.array_equal(got, W.to_bf16_bits(want))
    # the indexer on the appended caches: the prepared query with DSA_Q_MX_READY, and the raw query
    bt, sl = _t(case.block_table), _t(case.seq_lens)
    w = _t(case.w)
    idx_raw = dsa.indexer_topk(dims, q_I, w, k_I, scale, bt, sl, ws=ws)
    n_raw = dsa.last_launch_count()
    ready = dsa.make_dims(s.mode, s.B, case.max_blocks, case.num_blocks, s.H_I, s.d_I, s.H, s.d, s.d_v, s.K,
                          q_ready=True)
    idx_ready = dsa.indexer_topk(ready, q_out, w, k_I, scale, bt, sl, ws=ws)
    assert dsa.last_launch_count() == n_raw - 1
    torch.cuda.synchronize()
    assert torch.equal(idx_raw, idx_ready)
