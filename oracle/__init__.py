"""fp64 CPU oracle (test infrastructure) for index-selection sparse attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference legs of ``bench.py`` may import this package.  It wraps the plain C
library ``oracle.c`` (compiled here with gcc, ``-ffp-contract=off``) through
ctypes and shares no code with the CUDA path.

Functions take a :class:`workloads.Case`-like object (or explicit arrays) and
return NumPy arrays:

* :func:`index_scores` -- ``S[t, s]`` for every causal ``s <= q_pos[t]`` (NaN
  beyond), the indexer score of the lightweight indexer (Ascend CANN page
  §2.1 "Core Pipeline Operator Fusion").
* :func:`indexer_topk` -- ``idx[t, :K]`` in (score desc, position asc) order,
  ``-1`` padded, plus ``{S_(K), S_(K+1)}`` per row (Day-0 accelerator page
  §3.1 "Integration of the Index Selection Operator").
* :func:`sparse_attn` -- fp64 ``out[t, h, :d_v]``, ``lse[t, h]`` and the sum of
  the softmax weights, over the rows ``idx`` selects (lightweight indexer page
  §1, "sparse flash attention").
* :func:`block_summaries`, :func:`summary_case`, :func:`hierarchical_topk` --
  hierarchical (coarse -> fine) selection: blocks shortlisted by the indexer
  score of their mean key, then the indexer's Top-K over the tokens of the
  shortlisted blocks (Day-0 accelerator page §3.1; adaptation page §3.1).
* :func:`cache_append` -- the caches after writing new tokens' indexer keys and
  latent rows into their paged slots (FP8 keys: block requantisation; FP8
  latent rows: per-row tile quantisation), the step before the path (Ascend
  adaptation page §2.2, cache-update flow).

A case whose ``spec.kv`` is ``"fp8"`` stores its latent rows as FP8 records
(Ascend CANN page §3, FP8 block quantisation in the attention stage): per row,
the e4m3 codes, one fp32 scale per 128-element tile, zero padding to 16 bytes.

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

MODES = {"f32": 0, "bf16": 1, "bf16_kfp8": 2, "mxfp8": 3}


class ODims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("mode", "B", "max_blocks", "num_blocks", "block_size", "H_I", "d_I", "H", "d", "d_v", "K")]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (next to the source)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_to_f64.restype = ctypes.c_double
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_mx_quantize32.restype = ctypes.c_int
    lib.oracle_mx_quantize32.argtypes = [P, P]
    lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    lib.oracle_block_summaries.restype = ctypes.c_int
    lib.oracle_block_summaries.argtypes = [ctypes.POINTER(ODims), P, P, P, P, P]
    lib.oracle_cache_append.restype = ctypes.c_int
    lib.oracle_cache_append.argtypes = [ctypes.POINTER(ODims), P, P, P, P, P, P, ctypes.c_int, P, P, P]
    lib.oracle_index_scores.restype = ctypes.c_int
    lib.oracle_index_scores.argtypes = [ctypes.POINTER(ODims), P, P, P, P, P, P, P, P, ctypes.c_int,
                                        ctypes.c_int64, P, ctypes.c_int]
    lib.oracle_indexer_topk.restype = ctypes.c_int
    lib.oracle_indexer_topk.argtypes = [ctypes.POINTER(ODims), P, P, P, P, P, P, P, P, ctypes.c_int, P, P,
                                        ctypes.c_int]
    lib.oracle_sparse_attn.restype = ctypes.c_int
    lib.oracle_sparse_attn.argtypes = [ctypes.POINTER(ODims), P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double, P, P, P, ctypes.c_int]
    return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _scale(case):
    """The key-scale array in its storage type: fp32 per block (FP8 keys) or E8M0 bytes (MXFP8)."""
    if case.k_I_scale is None:
        return None
    if case.spec.mode == "mxfp8":
        return np.ascontiguousarray(case.k_I_scale, dtype=np.uint8)
    return np.ascontiguousarray(case.k_I_scale, dtype=np.float32)


def mx_quantize32(v) -> tuple:
    """(shared exponent X, 32 e4m3 codes) of 32 fp32 values (OCP MX, E4M3 elements)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    codes = np.zeros(32, np.uint8)
    X = _load().oracle_mx_quantize32(_ptr(v), _ptr(codes))
    return int(X), codes


KV_FP8 = 16  # mode flag: latent rows stored as FP8 records (e4m3 codes + one fp32 scale per 128 elements)


def kv_fp8(case) -> bool:
    return getattr(case.spec, "kv", "act") == "fp8"


def dims_of(case, K=None) -> ODims:
    s = case.spec
    mode = MODES[s.mode] | (KV_FP8 if kv_fp8(case) else 0)
    return ODims(mode, s.B, case.max_blocks, case.num_blocks, s.block_size, s.H_I, s.d_I, s.H, s.d,
                 s.d_v, s.K if K is None else K)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits))


def e4m3_to_f64(code: int) -> float:
    return _load().oracle_e4m3_to_f64(int(code))


def _rows(case, rows):
    """Query-side arrays restricted to the query rows ``rows`` (all rows if None)."""
    if rows is None:
        return case.q_I, case.w, case.q, case.q_seq, case.q_pos
    rows = np.asarray(rows, dtype=np.int64)
    return case.q_I[rows], case.w[rows], case.q[rows], case.q_seq[rows], case.q_pos[rows]


def index_scores(case, rows=None, threads=None) -> np.ndarray:
    """fp64 indexer scores ``S[r, s]`` for the query rows ``rows`` (NaN where s > q_pos)."""
    lib = _load()
    q_I, w, _, q_seq, q_pos = _rows(case, rows)
    T = len(q_seq)
    stride = int(q_pos.max()) + 1 if T else 1
    S = np.full((T, stride), np.nan, dtype=np.float64)
    D = dims_of(case)
    kdt = {"f32": np.float32, "bf16": np.uint16, "bf16_kfp8": np.uint8, "mxfp8": np.uint8}[case.spec.mode]
    adt = np.float32 if case.spec.mode == "f32" else np.uint16
    rc = lib.oracle_index_scores(ctypes.byref(D), _ptr(_c(q_I, adt)), _ptr(_c(w, np.float32)),
                                 _ptr(_c(case.k_I, kdt)), _ptr(_scale(case)),
                                 _ptr(_c(case.block_table, np.int32)), _ptr(_c(case.seq_lens, np.int32)),
                                 _ptr(_c(q_seq, np.int32)), _ptr(_c(q_pos, np.int32)), T, stride, _ptr(S),
                                 threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_index_scores failed: {rc}")
    return S


def indexer_topk(case, rows=None, K=None, threads=None):
    """(idx[r, K] int32 in (score desc, pos asc) order, kth[r, 2] = {S_(K), S_(K+1)})."""
    lib = _load()
    q_I, w, _, q_seq, q_pos = _rows(case, rows)
    T = len(q_seq)
    D = dims_of(case, K)
    idx = np.full((T, D.K), -1, dtype=np.int32)
    kth = np.full((T, 2), np.nan, dtype=np.float64)
    kdt = {"f32": np.float32, "bf16": np.uint16, "bf16_kfp8": np.uint8, "mxfp8": np.uint8}[case.spec.mode]
    adt = np.float32 if case.spec.mode == "f32" else np.uint16
    keep = [_c(q_I, adt), _c(w, np.float32), _c(case.k_I, kdt), _scale(case),
            _c(case.block_table, np.int32), _c(case.seq_lens, np.int32), _c(q_seq, np.int32), _c(q_pos, np.int32)]
    rc = lib.oracle_indexer_topk(ctypes.byref(D), *[_ptr(a) for a in keep], T, _ptr(idx), _ptr(kth),
                                 threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_indexer_topk failed: {rc}")
    return idx, kth


def sparse_attn(case, idx, rows=None, sm_scale=None, threads=None):
    """(out[r, H, d_v] f64, lse[r, H] f64, psum[r, H] f64) over the positions in ``idx[r]``."""
    lib = _load()
    _, _, q, q_seq, _ = _rows(case, rows)
    T = len(q_seq)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    assert idx.shape[0] == T
    s = case.spec
    D = dims_of(case)
    out = np.zeros((T, s.H, s.d_v), dtype=np.float64)
    lse = np.zeros((T, s.H), dtype=np.float64)
    psum = np.zeros((T, s.H), dtype=np.float64)
    adt = np.float32 if s.mode == "f32" else np.uint16
    kvdt = np.uint8 if kv_fp8(case) else adt
    keep = [_c(q, adt), _c(case.kv, kvdt), _c(case.block_table, np.int32), _c(case.seq_lens, np.int32),
            _c(q_seq, np.int32)]
    rc = lib.oracle_sparse_attn(ctypes.byref(D), *[_ptr(a) for a in keep], _ptr(idx), idx.shape[1], T,
                                s.sm_scale if sm_scale is None else float(sm_scale), _ptr(out), _ptr(lse),
                                _ptr(psum), threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_sparse_attn failed: {rc}")
    return out, lse, psum


def f32_to_e4m3(x: float) -> int:
    """OCP e4m3 code of an fp32 value (round to nearest even, saturating at +-448)."""
    return int(_load().oracle_f32_to_e4m3(float(x)))


def cache_append(case, k_new, kv_new, rows=None):
    """(k_I, k_I_scale, kv) after appending new tokens: row r of k_new / kv_new is the token at
    position case.q_pos[r] of sequence case.q_seq[r] (all rows, or the rows ``rows``). The
    case's arrays are not modified; updated copies are returned."""
    lib = _load()
    s = case.spec
    q_seq = case.q_seq if rows is None else case.q_seq[np.asarray(rows)]
    q_pos = case.q_pos if rows is None else case.q_pos[np.asarray(rows)]
    T = len(q_seq)
    k_I = np.ascontiguousarray(case.k_I).copy()
    kv = np.ascontiguousarray(case.kv).copy()
    scale = None if case.k_I_scale is None else _scale(case).copy()
    kdt = np.float32 if s.mode == "f32" else np.uint16
    adt = np.float32 if s.mode == "f32" else np.uint16
    keep = [_c(k_new, kdt), _c(kv_new, adt), _c(case.block_table, np.int32), _c(case.seq_lens, np.int32),
            _c(q_seq, np.int32), _c(q_pos, np.int32)]
    rc = lib.oracle_cache_append(ctypes.byref(dims_of(case)), *[_ptr(a) for a in keep], T, _ptr(k_I), _ptr(scale),
                                 _ptr(kv))
    if rc:
        raise RuntimeError(f"oracle_cache_append failed: {rc}")
    return k_I, scale, kv


def block_summaries(case) -> np.ndarray:
    """bf16 bits [B][max_blocks][d_I]: the mean key of every valid 64-token block (zeros elsewhere)."""
    lib = _load()
    s = case.spec
    out = np.zeros((s.B, case.max_blocks, s.d_I), dtype=np.uint16)
    kdt = {"f32": np.float32, "bf16": np.uint16, "bf16_kfp8": np.uint8, "mxfp8": np.uint8}[s.mode]
    keep = [_c(case.k_I, kdt), _scale(case), _c(case.block_table, np.int32),
            _c(case.seq_lens, np.int32)]
    rc = lib.oracle_block_summaries(ctypes.byref(dims_of(case)), *[_ptr(a) for a in keep], _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_block_summaries failed: {rc}")
    return out


def summary_case(case, summaries, n_sel: int):
    """The coarse stage as an indexer problem: sequence b's block summaries are its "keys" at
    logical positions 0..ceil(L_b/64)-1, stored densely (64 summaries per summary block), with a
    query row at position pos(t) // 64 and Top-K = n_sel."""
    import types
    s = case.spec
    bs = s.block_size
    mb2 = (case.max_blocks + bs - 1) // bs
    lens = ((case.seq_lens.astype(np.int64) + bs - 1) // bs).astype(np.int32)
    keys = np.zeros((s.B * mb2 * bs, s.d_I), dtype=np.uint16)
    keys.reshape(s.B, mb2 * bs, s.d_I)[:, : case.max_blocks] = summaries
    table = (np.arange(s.B)[:, None] * mb2 + np.arange(mb2)[None, :]).astype(np.int32)
    spec2 = types.SimpleNamespace(mode="bf16", B=s.B, T=s.T, H_I=s.H_I, d_I=s.d_I, H=s.H, d=s.d, d_v=s.d_v, K=n_sel,
                                  block_size=bs, sm_scale=s.sm_scale, new_tokens=s.new_tokens)
    return types.SimpleNamespace(spec=spec2, block_table=table, seq_lens=lens, q_seq=case.q_seq,
                                 q_pos=(case.q_pos // bs).astype(np.int32), q_I=case.q_I, w=case.w,
                                 k_I=keys.reshape(s.B * mb2, bs, s.d_I), k_I_scale=None, max_blocks=mb2,
                                 num_blocks=s.B * mb2, q=case.q, kv=case.kv)


def hierarchical_topk(case, n_sel: int, rows=None, threads=None):
    """(idx[r, K] ascending positions -1 padded, blocks[r, n_sel] ascending logical blocks -1 padded)
    of hierarchical selection: the n_sel blocks with the largest summary scores (ties to the lower
    block), then the K largest token scores (ties to the lower position) among the tokens of those
    blocks inside the causal prefix."""
    s = case.spec
    bs = s.block_size
    sel = np.arange(s.T) if rows is None else np.asarray(rows)
    summ = block_summaries(case)
    c2 = summary_case(case, summ, n_sel)
    bidx, _ = indexer_topk(c2, rows=sel, threads=threads)
    S = index_scores(case, rows=sel, threads=threads)
    idx = np.full((len(sel), s.K), -1, np.int32)
    blocks = np.full((len(sel), n_sel), -1, np.int32)
    for r, t in enumerate(sel):
        n = int(case.q_pos[t]) + 1
        bl = np.sort(bidx[r][bidx[r] >= 0])
        blocks[r, : len(bl)] = bl
        pos = np.concatenate([np.arange(b * bs, min((b + 1) * bs, n)) for b in bl]) if len(bl) else np.zeros(0, np.int64)
        sc = S[r, pos]
        order = np.lexsort((pos, -sc))[: s.K]
        chosen = np.sort(pos[order])
        idx[r, : len(chosen)] = chosen
    return idx, blocks
