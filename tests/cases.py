"""Test-side helpers: small workloads, an independent NumPy brute force and the parity rules.

The brute force here is a pin for the oracle, not a second oracle: it decodes
inputs with NumPy / torch casts (not the oracle's C decoders), builds the full
score matrix with matrix products and ranks it with ``np.lexsort``.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import workloads as W


def small_spec(mode: str, lens, K: int, new_tokens=None, H_I=None, d_I=None, H=None, d=None, d_v=None,
               kv: str = "act") -> W.Spec:
    """Small shapes per mode (f32: 4x64 indexer, 8 heads d=128; bf16 modes: the full head counts)."""
    if mode == "f32":
        dims = dict(H_I=4, d_I=64, H=8, d=128, d_v=128)
    else:
        dims = dict(H_I=64, d_I=128, H=128, d=576, d_v=512)
    for k, v in dict(H_I=H_I, d_I=d_I, H=H, d=d, d_v=d_v).items():
        if v is not None:
            dims[k] = v
    lens = [int(x) for x in lens]
    nt = [1] * len(lens) if new_tokens is None else [int(x) for x in new_tokens]
    return W.Spec(f"small_{mode}", mode, lens, nt, K=K, kv=kv, **dims)


# ----------------------------------------------------------------------------
# independent decoding (NumPy / torch casts)
# ----------------------------------------------------------------------------

def np_bf16(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def np_e4m3(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def act(case, a) -> np.ndarray:
    return np.asarray(a, np.float64) if case.spec.mode == "f32" else np_bf16(a)


def logical_rows(case, b: int, cache: np.ndarray, scale=None, n=None) -> np.ndarray:
    """Logical rows 0..n-1 of sequence b gathered through the block table (fancy indexing)."""
    bs = case.spec.block_size
    L = int(case.seq_lens[b]) if n is None else int(n)
    s = np.arange(L)
    blk = case.block_table[b, s // bs]
    rows = cache[blk, s % bs]
    if scale is not None:
        return rows, scale[blk]
    return rows


def np_mx(codes, scale_bytes) -> np.ndarray:
    """MXFP8 values: e4m3 code times 2^(byte - 127), one byte per 32 elements of the last axis."""
    x = np_e4m3(codes)
    return x * np.exp2(np.repeat(np.asarray(scale_bytes, np.float64) - 127.0, 32, axis=-1))


def mx_roundtrip(x) -> np.ndarray:
    """fp32 values -> their MXFP8 quantisation (the generator's NumPy/torch recipe), decoded."""
    return np_mx(*W.to_mx_e4m3(np.asarray(x, np.float32)))


def logical_keys(case, b: int, n=None) -> np.ndarray:
    if case.spec.mode == "bf16_kfp8":
        codes, sc = logical_rows(case, b, case.k_I, case.k_I_scale, n)
        return np_e4m3(codes) * sc.astype(np.float64)[:, None]
    if case.spec.mode == "mxfp8":
        bs = case.spec.block_size
        L = int(case.seq_lens[b]) if n is None else int(n)
        s = np.arange(L)
        blk = case.block_table[b, s // bs]
        return np_mx(case.k_I[blk, s % bs], case.k_I_scale[blk, s % bs])
    return act(case, logical_rows(case, b, case.k_I, None, n))


def kv_fp8_decode(recs, d: int) -> np.ndarray:
    """FP8 latent records -> row values in fp64: torch's e4m3 cast of the codes times the fp32 scale
    of each element's 128-wide tile (the scales follow the d codes)."""
    recs = np.ascontiguousarray(recs, dtype=np.uint8)
    nt = (d + 127) // 128
    sc = np.ascontiguousarray(recs[..., d: d + 4 * nt]).view(np.float32).astype(np.float64)
    return np_e4m3(recs[..., :d]) * np.repeat(sc, 128, axis=-1)[..., :d]


def logical_kv(case, b: int, n=None) -> np.ndarray:
    if getattr(case.spec, "kv", "act") == "fp8":
        return kv_fp8_decode(logical_rows(case, b, case.kv, None, n), case.spec.d)
    return act(case, logical_rows(case, b, case.kv, None, n))


# ----------------------------------------------------------------------------
# brute force
# ----------------------------------------------------------------------------

def brute_scores_row(case, t: int) -> np.ndarray:
    b = int(case.q_seq[t])
    n = int(case.q_pos[t]) + 1
    if n <= 0:
        return np.zeros(0)
    K = logical_keys(case, b, n)                      # [n, d_I]
    q = act(case, case.q_I[t])                        # [H_I, d_I]
    if case.spec.mode == "mxfp8":                     # the query is MX-quantised too
        q = mx_roundtrip(q)
    w = case.w[t].astype(np.float64)                  # [H_I]
    return w @ np.maximum(q @ K.T, 0.0)               # [n]


def brute_topk_row(S: np.ndarray, K: int) -> np.ndarray:
    order = np.lexsort((np.arange(len(S)), -S))       # score desc, position asc
    out = np.full(K, -1, np.int32)
    m = min(K, len(S))
    out[:m] = order[:m]
    return out


def brute_attn_row(case, t: int, idx_row, sm_scale=None):
    b = int(case.q_seq[t])
    sel = np.asarray([i for i in idx_row if i >= 0], np.int64)
    s = case.spec
    if len(sel) == 0:
        return np.zeros((s.H, s.d_v)), np.full(s.H, -np.inf)
    rows = logical_kv(case, b)[sel]                   # [n, d]
    q = act(case, case.q[t])                          # [H, d]
    z = (q @ rows.T) * (s.sm_scale if sm_scale is None else sm_scale)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    l = e.sum(axis=1, keepdims=True)
    return (e / l) @ rows[:, : s.d_v], (m + np.log(l))[:, 0]


# ----------------------------------------------------------------------------
# parity rules for Top-K index sets
# ----------------------------------------------------------------------------

REL_GAP = 1e-3


def check_index_row(gpu_row, oracle_row, S_row, K: int, kth=None) -> str | None:
    """Compare one query row's index set with the oracle's.

    * fewer than K causal positions: the set must be exactly all of them;
    * K-th and (K+1)-th oracle scores more than 1e-3 apart (relative): the
      sets must be equal, bit for bit;
    * otherwise (near tie at the boundary, band tau = 1e-3*|S_(K)|): K
      distinct in-range entries, every s with S_s > S_(K)+tau present and no s
      with S_s < S_(K)-tau present.
    Returns None when the row passes, else a message.
    """
    g = np.asarray(gpu_row, np.int64)
    o = np.asarray(oracle_row, np.int64)
    n = len(S_row)
    gv = g[g >= 0]
    if len(np.unique(gv)) != len(gv):
        return "duplicate indices"
    if np.any(gv >= n):
        return "index beyond the causal prefix"
    if np.any((g < 0) & (g != -1)):
        return "negative index other than -1"
    if n <= K:
        if len(gv) != n or set(gv.tolist()) != set(range(n)):
            return f"short row: expected all {n} positions, got {len(gv)}"
        return None
    if len(gv) != K:
        return f"expected {K} entries, got {len(gv)}"
    if kth is None:
        srt = np.sort(S_row)[::-1]
        sk, sk1 = srt[K - 1], srt[K]
    else:
        sk, sk1 = kth
    denom = abs(sk) if sk != 0 else 1.0
    gap = (sk - sk1) / denom
    if sk == 0:
        gap = sk - sk1  # absolute 1e-3 when S_(K) is zero
    if gap > REL_GAP:
        if set(gv.tolist()) != set(o[o >= 0].tolist()):
            return f"set differs although gap {gap:.3g} > 1e-3"
        return None
    tau = REL_GAP * (abs(sk) if sk != 0 else 1.0)
    must = np.nonzero(S_row > sk + tau)[0]
    if not set(must.tolist()) <= set(gv.tolist()):
        return "missing an index above the band"
    if np.any(S_row[gv] < sk - tau):
        return "contains an index below the band"
    return None


def ulp_tol_bf16(x: np.ndarray) -> np.ndarray:
    return np.abs(x) * 2.0 ** -8


def sdpa_f64(q, k, v, scale):
    """torch CPU float64 scaled-dot-product attention (an independent library routine)."""
    qt = torch.from_numpy(q)[None]          # [1, H, d]
    kt = torch.from_numpy(k)[None, None].expand(1, q.shape[0], *k.shape)  # [1,H,n,d]
    vt = torch.from_numpy(v)[None, None].expand(1, q.shape[0], *v.shape)
    out = torch.nn.functional.scaled_dot_product_attention(qt[:, :, None, :], kt, vt, scale=scale)
    return out[0, :, 0, :].numpy()


def log_uniform_lens(rng, n, lo, hi):
    return [int(round(math.exp(x))) for x in rng.uniform(math.log(lo), math.log(hi), size=n)]
