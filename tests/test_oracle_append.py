"""Pins for the oracle's cache append (the step before the path) and its e4m3 encoder.

The append writes each new token's latent row (and, in the fp32 / bf16 modes, its indexer key)
into its paged slot; with FP8 indexer keys every touched 64-token block is requantised with
scale = amax / 448 over the block's earlier tokens (code * old scale) and the new keys. The pins
check it against independent routines: torch's float8_e4m3fn cast, the synthetic generator's
own block quantisation (torch), and NumPy gathers through the block table.
"""
import numpy as np
import torch

import oracle
import workloads as W
from cases import np_bf16, np_e4m3, small_spec


def torch_e4m3(x: np.ndarray) -> np.ndarray:
    x = np.clip(np.asarray(x, np.float32), -448.0, 448.0)
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encoder_matches_torch_cast():
    rng = np.random.default_rng(0)
    mags = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), size=20000)).astype(np.float32)
    x = mags * rng.choice([-1.0, 1.0], size=mags.size).astype(np.float32)
    # every representable value, and the midpoints between neighbours (ties to even)
    reps = np.array([oracle.e4m3_to_f64(c) for c in range(0x7F)], np.float64)
    mids = ((reps[1:] + reps[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, reps.astype(np.float32), mids, -mids, np.float32([0.0, -0.0, 448.0, 449.0, 1e9])])
    ours = np.array([oracle.f32_to_e4m3(v) for v in x], np.uint8)
    ref = torch_e4m3(x)
    same = (ours == ref) | ((ours & 0x7F) == 0) & ((ref & 0x7F) == 0)  # +-0 both fine
    assert same.all(), x[~same][:10]


def _new_tokens(case, seed):
    rng = np.random.default_rng(seed)
    s = case.spec
    k = rng.standard_normal((s.T, s.d_I), dtype=np.float32)
    v = rng.standard_normal((s.T, s.d), dtype=np.float32)
    if s.mode == "f32":
        return k, v
    return W.to_bf16_bits(k), W.to_bf16_bits(v)


def _slot(case, t):
    b, p = int(case.q_seq[t]), int(case.q_pos[t])
    return int(case.block_table[b, p // 64]), p % 64


def test_append_copies_rows_in_f32_and_bf16():
    for mode in ("f32", "bf16"):
        spec = small_spec(mode, [70, 200, 64], 64, new_tokens=[3, 70, 1])
        case = W.generate(spec, seed=31)
        k_new, kv_new = _new_tokens(case, 32)
        k_I, _, kv = oracle.cache_append(case, k_new, kv_new)
        touched = set()
        for t in range(spec.T):
            blk, off = _slot(case, t)
            assert np.array_equal(kv[blk, off], kv_new[t])
            assert np.array_equal(k_I[blk, off], k_new[t])
            touched.add((blk, off))
        for blk in range(case.num_blocks):  # nothing else changed
            for off in range(64):
                if (blk, off) not in touched:
                    assert np.array_equal(kv[blk, off], case.kv[blk, off])
                    assert np.array_equal(k_I[blk, off], case.k_I[blk, off])


def test_append_whole_new_block_matches_the_generators_quantisation():
    """64 new tokens filling a block: scale = amax/448 and codes = RNE(x / scale), exactly the
    recipe the generator applies with torch."""
    spec = small_spec("bf16_kfp8", [128], 64, new_tokens=[64])
    case = W.generate(spec, seed=33)
    k_new, kv_new = _new_tokens(case, 34)
    k_I, scale, _ = oracle.cache_append(case, k_new, kv_new)
    blk = int(case.block_table[0, 1])
    x = np_bf16(k_new).astype(np.float32)
    s = np.float32(np.abs(x).max()) / np.float32(448.0)
    assert scale[blk] == s
    assert np.array_equal(k_I[blk], torch_e4m3(x / s))
    assert np.array_equal(scale[np.arange(case.num_blocks) != blk], case.k_I_scale[np.arange(case.num_blocks) != blk])


def test_append_requantises_the_earlier_tokens_of_the_block():
    spec = small_spec("bf16_kfp8", [100, 30], 64, new_tokens=[5, 1])
    case = W.generate(spec, seed=35)
    k_new, kv_new = _new_tokens(case, 36)
    k_new[0, 0] = W.to_bf16_bits(np.float32([60.0]))[0]  # raises the amax of sequence 0's block 1
    k_I, scale, _ = oracle.cache_append(case, k_new, kv_new)
    for b, first_row, n_new in ((0, 0, 5), (1, 5, 1)):
        p0 = int(case.q_pos[first_row])
        lb = p0 // 64
        blk = int(case.block_table[b, lb])
        n_old = p0 - lb * 64
        old = (np_e4m3(case.k_I[blk, :n_old]).astype(np.float32) * case.k_I_scale[blk]).astype(np.float32)
        new = np_bf16(k_new[first_row:first_row + n_new]).astype(np.float32)
        amax = max(np.abs(old).max() if n_old else 0.0, np.abs(new).max())
        s = np.float32(amax) / np.float32(448.0)
        assert scale[blk] == s
        assert np.array_equal(k_I[blk, :n_old], torch_e4m3(old / s))
        assert np.array_equal(k_I[blk, n_old:n_old + n_new], torch_e4m3(new / s))
    assert scale[int(case.block_table[0, 1])] == np.float32(60.0) / np.float32(448.0)


def test_append_keeps_codes_when_the_block_scale_does_not_grow():
    """Small new keys: an earlier token holding the code 448 fixes amax = 448 * old scale, so the
    scale is kept and every earlier code survives the requantisation unchanged."""
    spec = small_spec("bf16_kfp8", [90], 64, new_tokens=[1])
    case = W.generate(spec, seed=37)
    k_new, kv_new = _new_tokens(case, 38)
    k_new[:] = W.to_bf16_bits(np_bf16(k_new).astype(np.float32) * np.float32(1e-3))
    blk = int(case.block_table[0, 1])
    case.k_I[blk, 3, 7] = 0x7E
    old_codes = case.k_I[blk, :25].copy()
    k_I, scale, _ = oracle.cache_append(case, k_new, kv_new)
    assert scale[blk] == case.k_I_scale[blk]
    assert np.array_equal(k_I[blk, :25], old_codes)
    x = np_bf16(k_new[0]).astype(np.float32)
    assert np.array_equal(k_I[blk, 25], torch_e4m3(x / case.k_I_scale[blk]))


def test_append_mx_quantises_each_new_key_on_its_own():
    """MXFP8 keys: every new token's key gets its own codes and E8M0 bytes (the generator's
    NumPy/torch recipe applied to the bf16 key); no other key row and no other scale changes."""
    spec = small_spec("mxfp8", [130, 64, 7], 64, new_tokens=[70, 1, 7], H_I=4, d_I=64)
    case = W.generate(spec, seed=35)
    k_new, kv_new = _new_tokens(case, 36)
    k_I, scale, kv = oracle.cache_append(case, k_new, kv_new)
    codes, byts = W.to_mx_e4m3(np_bf16(k_new).astype(np.float32))
    touched = set()
    for t in range(spec.T):
        blk, off = _slot(case, t)
        assert np.array_equal(k_I[blk, off], codes[t])
        assert np.array_equal(scale[blk, off], byts[t])
        assert np.array_equal(kv[blk, off], kv_new[t])
        touched.add((blk, off))
    for blk in range(case.num_blocks):
        for off in range(64):
            if (blk, off) not in touched:
                assert np.array_equal(k_I[blk, off], case.k_I[blk, off])
                assert np.array_equal(scale[blk, off], case.k_I_scale[blk, off])


def test_append_fp8_latent_rows_match_the_generators_quantisation():
    """FP8 latent records: each new row's 128-element tiles quantised on their own (the generator's
    NumPy/torch recipe applied to the bf16 row), bit for bit; no other record changes."""
    spec = small_spec("bf16", [130, 64, 7], 64, new_tokens=[70, 1, 7], H_I=4, d_I=16, H=4, d=192, d_v=160,
                      kv="fp8")
    case = W.generate(spec, seed=37)
    k_new, kv_new = _new_tokens(case, 38)
    k_I, _, kv = oracle.cache_append(case, k_new, kv_new)
    recs = W.to_kv_fp8_records(np_bf16(kv_new).astype(np.float32))
    touched = set()
    for t in range(spec.T):
        blk, off = _slot(case, t)
        assert np.array_equal(kv[blk, off], recs[t])
        assert np.array_equal(k_I[blk, off], k_new[t])
        touched.add((blk, off))
    for blk in range(case.num_blocks):
        for off in range(64):
            if (blk, off) not in touched:
                assert np.array_equal(kv[blk, off], case.kv[blk, off])
