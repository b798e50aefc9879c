"""A seeded sweep of small random shapes in every storage mode: the oracle's scores, Top-K and
attention against the NumPy brute force (full score rows sorted by (score desc, position asc);
softmax attention over the decoded rows). The fixed-shape pins cover chosen edge cases; this
covers head counts, widths, K and prefill-row layouts drawn at random."""
import numpy as np
import pytest

import oracle
import workloads as W
from cases import brute_attn_row, brute_scores_row, brute_topk_row, small_spec

MODES = ["f32", "bf16", "bf16_kfp8", "mxfp8"]


def _random_spec(mode: str, rng: np.random.Generator):
    B = int(rng.integers(1, 4))
    lens = [int(x) for x in rng.integers(0, 400, size=B)]
    new = [int(rng.integers(1, 4)) if n > 3 else 1 for n in lens]
    K = int(rng.integers(1, 300))
    H_I = int(rng.choice([1, 2, 4, 8]))
    d_I = int(rng.choice([32, 64])) if mode == "mxfp8" else int(rng.choice([8, 16, 32, 64]))
    H = int(rng.choice([1, 2, 4]))
    d = int(rng.choice([16, 32, 48, 64, 144]))
    d_v = int(rng.choice([x for x in (8, 16, 32, d) if x <= d]))
    kv = "fp8" if mode != "f32" and rng.random() < 0.3 else "act"
    return small_spec(mode, lens, K, new_tokens=new, H_I=H_I, d_I=d_I, H=H, d=d, d_v=d_v, kv=kv)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("draw", range(6))
def test_random_small_shapes_match_brute_force(mode, draw):
    rng = np.random.default_rng(1000 + 17 * draw + MODES.index(mode))
    spec = _random_spec(mode, rng)
    case = W.generate(spec, seed=int(rng.integers(1 << 30)))
    S_or = oracle.index_scores(case)
    idx, _ = oracle.indexer_topk(case)
    for t in range(spec.T):
        S = brute_scores_row(case, t)
        n = len(S)
        np.testing.assert_allclose(S_or[t, :n], S, rtol=1e-12, atol=1e-12)
        assert idx[t].tolist() == brute_topk_row(S, spec.K).tolist(), (spec, t)
    out, lse, psum = oracle.sparse_attn(case, idx)
    for t in range(spec.T):
        o_b, l_b = brute_attn_row(case, t, idx[t])
        np.testing.assert_allclose(out[t], o_b, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[t], l_b, rtol=1e-12, atol=1e-12)
        if np.any(idx[t] >= 0):
            np.testing.assert_allclose(psum[t], 1.0, rtol=0, atol=1e-12)
