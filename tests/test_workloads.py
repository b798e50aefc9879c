"""The synthetic inputs: the key-format re-storing helper (used by the bench's FP8 / MXFP8 timings
and profiles) keeps every token's key within its format's rounding of the bf16 key, poisons the
slots that hold no token, and scales FP8 blocks by amax / 448 over the block's tokens."""
import numpy as np

import workloads as W
from cases import np_bf16, np_e4m3, np_mx, small_spec


def _valid_slots(case):
    valid = np.zeros(case.k_I.shape[:2], bool)
    for b, L in enumerate(case.seq_lens.tolist()):
        for s in range(L):
            valid[case.block_table[b, s // 64], s % 64] = True
    return valid


def test_with_key_format_mxfp8():
    case = W.generate(small_spec("bf16", [1, 63, 64, 65, 300], 64), seed=71)
    mx = W.with_key_format(case, "mxfp8")
    valid = _valid_slots(case)
    x = np_bf16(case.k_I)[valid]
    y = np_mx(mx.k_I, mx.k_I_scale)[valid]
    # MX E4M3: relative rounding 2^-4 of the group maximum scale at most, plus the clamp at 448
    g = np.abs(x).reshape(len(x), -1, 32).max(axis=2)
    assert np.all(np.abs(y - x).reshape(len(x), -1, 32) <= 0.126 * g[..., None] + 1e-30)
    assert np.array_equal(mx.k_I_scale, W.to_mx_e4m3(np.where(valid[..., None], np_bf16(case.k_I), 0.0).astype(np.float32))[1] * valid[..., None] + 127 * ~valid[..., None])
    assert np.all(mx.k_I[~valid] == W.POISON_E4M3)
    assert mx.spec.mode == "mxfp8" and mx.q_I is case.q_I and mx.kv is case.kv


def test_with_key_format_fp8_block_scale():
    case = W.generate(small_spec("bf16", [1, 63, 64, 65, 300], 64), seed=72)
    f8 = W.with_key_format(case, "bf16_kfp8")
    valid = _valid_slots(case)
    x = np_bf16(case.k_I)
    for blk in range(case.num_blocks):
        v = valid[blk]
        if not v.any():
            assert np.all(f8.k_I[blk] == W.POISON_E4M3)
            continue
        amax = np.float32(np.abs(x[blk][v]).max())
        assert f8.k_I_scale[blk] == np.float32(amax / np.float32(448.0))
        y = np_e4m3(f8.k_I[blk][v]) * np.float64(f8.k_I_scale[blk])
        assert np.all(np.abs(y - x[blk][v]) <= amax * 2.0 ** -4 + 1e-30)
        assert np.all(f8.k_I[blk][~v] == W.POISON_E4M3)
