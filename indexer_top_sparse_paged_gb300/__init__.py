"""Index-selection sparse attention over a paged KV cache on GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libdsa.so`` (C ABI in ``include/dsa.h``). It only marshals
arguments: torch tensors are passed as device pointers together with the current CUDA stream,
and every step of the computation runs in the library's kernels. There is no fallback: if the
library is missing or fails to load, :func:`lib` raises.

Entry points (same names as the C ABI):

* :func:`indexer_topk` -- lightning indexer + Top-K: ``idx[T][K]`` of the selected positions.
* :func:`sparse_attn` -- sparse attention over the rows ``idx`` selects.
* :func:`decode` -- both, fused on one stream, for one query row per sequence.
* :func:`cache_append` -- new tokens' indexer keys and latent rows into the paged caches (FP8 keys:
  block requantisation; FP8 latent rows: per-tile quantisation).
* :func:`indexer_prolog` -- the cache append and the MXFP8 query quantisation in one launch.
* :func:`block_summaries`, :func:`indexer_topk_hier` -- hierarchical (coarse -> fine) selection over
  per-block summary keys.
* :func:`indexer_topk_noalloc` -- :func:`indexer_topk` with the library's static scratch instead of
  a workspace, for callers that cannot allocate device memory.

Every tensor argument is a contiguous CUDA tensor in the layout ``include/dsa.h`` gives; the
calls are enqueued on the current stream (or ``stream=``). A decode step over a batch of B
sequences, bf16 everywhere, 64 indexer heads of 128, 128 heads over 576-wide latent rows::

    dims = make_dims("bf16", B, max_blocks, num_blocks, H_I=64, d_I=128, H=128, d=576, d_v=512, K=2048)
    ws = workspace(dims, B)                      # sized for calls of B rows (the library checks it)
    idx, out, lse = decode(dims, q_I, w, k_I_cache, None, block_table, seq_lens, q, kv_cache,
                           576 ** -0.5, ws=ws)  # idx [B][K] int32, out [B][128][512] bf16
    assert read_error(ws) == 0                   # device-side fault bits (synchronises)
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")
_lib = None

MODES = {"f32": 0, "bf16": 1, "bf16_kfp8": 2, "mxfp8": 3}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace", 4: "launch", 5: "device fault",
          6: "timeout", 7: "too large for the static scratch"}


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("mode", "B", "max_blocks", "num_blocks", "block_size", "H_I", "d_I", "H", "d", "d_v", "K")]


class DsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {lib().dsa_status_string(status).decode()} (status {status})")


def lib():
    """The loaded libdsa.so (built by ``__graft_entry__.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m indexer_top_sparse_paged_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        D = ctypes.POINTER(Dims)
        L.dsa_workspace_size.restype = SZ
        L.dsa_workspace_size.argtypes = [D, I32]
        L.dsa_workspace_init.restype = ctypes.c_int
        L.dsa_workspace_init.argtypes = [P, SZ, P]
        L.dsa_indexer_topk.restype = ctypes.c_int
        L.dsa_indexer_topk.argtypes = [D, P, P, P, P, P, P, P, P, I32, P, P, SZ, P]
        L.dsa_sparse_attn.restype = ctypes.c_int
        L.dsa_sparse_attn.argtypes = [D, P, P, P, P, P, P, I32, ctypes.c_float, P, P, P, SZ, P]
        L.dsa_decode.restype = ctypes.c_int
        L.dsa_decode.argtypes = [D, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, SZ, P]
        L.dsa_hier_workspace_size.restype = SZ
        L.dsa_hier_workspace_size.argtypes = [D, I32, I32]
        L.dsa_block_summaries.restype = ctypes.c_int
        L.dsa_block_summaries.argtypes = [D, P, P, P, P, P, P, SZ, P]
        L.dsa_block_summaries_append.restype = ctypes.c_int
        L.dsa_block_summaries_append.argtypes = [D, P, P, P, P, P, P, I32, P, P, SZ, P]
        L.dsa_indexer_topk_hier.restype = ctypes.c_int
        L.dsa_indexer_topk_hier.argtypes = [D, P, P, P, P, P, P, P, P, I32, P, I32, P, P, P, SZ, P]
        L.dsa_cache_append.restype = ctypes.c_int
        L.dsa_cache_append.argtypes = [D, P, P, P, P, P, P, I32, P, P, P, P, SZ, P]
        L.dsa_indexer_prolog.restype = ctypes.c_int
        L.dsa_indexer_prolog.argtypes = [D, P, P, P, P, P, P, I32, P, P, P, P, I32, P, P, SZ, P]
        L.dsa_indexer_topk_noalloc.restype = ctypes.c_int
        L.dsa_indexer_topk_noalloc.argtypes = [D, P, P, P, P, P, P, P, P, I32, P, P, P]
        L.dsa_read_error.restype = ctypes.c_int
        L.dsa_read_error.argtypes = [P, ctypes.POINTER(I32), P]
        L.dsa_selftest_wait_timeout.restype = ctypes.c_int
        L.dsa_selftest_wait_timeout.argtypes = [P, SZ, P]
        L.dsa_last_launch_count.restype = I32
        L.dsa_last_launch_count.argtypes = []
        L.dsa_status_string.restype = ctypes.c_char_p
        L.dsa_status_string.argtypes = [ctypes.c_int]
        L.dsa_version.restype = I32
        L.dsa_version.argtypes = []
        _lib = L
    return _lib


KV_FP8 = 0x10  # DSA_KV_FP8: the latent cache holds FP8 records (e4m3 codes, one fp32 scale per 128 elements)
Q_MX_READY = 0x20  # DSA_Q_MX_READY: q_I already holds MXFP8 values (from indexer_prolog)


def kv_record_bytes(d: int) -> int:
    """DSA_KV_FP8_RECORD_BYTES(d): bytes of one FP8 latent record."""
    return (d + 4 * ((d + 127) // 128) + 15) // 16 * 16


def make_dims(mode: str, B: int, max_blocks: int, num_blocks: int, H_I: int, d_I: int, H: int, d: int, d_v: int,
              K: int, block_size: int = 64, kv: str = "act", q_ready: bool = False) -> Dims:
    """kv="fp8" sets DSA_KV_FP8 (the latent cache holds FP8 records); q_ready sets DSA_Q_MX_READY."""
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    if q_ready:
        m |= Q_MX_READY
    if kv == "fp8":
        m |= KV_FP8
    elif kv != "act":
        raise ValueError(f"unknown latent-cache storage {kv!r}")
    return Dims(m, B, max_blocks, num_blocks, block_size, H_I, d_I, H, d, d_v, K)


def _p(t):
    """The device address of a tensor argument (None: NULL). The library reads and writes densely
    packed data through raw device pointers, so a strided view or a host tensor is refused here:
    passed on, it would be read with the wrong layout or dereferenced on the GPU as a bad address."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous (the library reads densely packed rows)")
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors (the library takes device pointers)")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise DsaError(fn, status)


def _check_out(dims: Dims, T: int, out, lse):
    """The output buffers the library writes must have its dtype and size (it takes raw pointers)."""
    odt = torch.float32 if dims.mode == MODES["f32"] else torch.bfloat16
    if out.dtype != odt or out.numel() < T * dims.H * dims.d_v or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {odt} tensor of T x H x d_v elements")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() < T * dims.H or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 tensor of T x H elements")


def _check_idx(dims: Dims, T: int, idx):
    if idx.dtype != torch.int32 or idx.numel() < T * dims.K or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous int32 tensor of T x K elements")


def workspace_size(dims: Dims, T: int) -> int:
    return int(lib().dsa_workspace_size(ctypes.byref(dims), T))


def workspace(dims: Dims, T: int, device="cuda", stream=None) -> torch.Tensor:
    """Allocates (with torch) and initialises a workspace for calls with T query rows."""
    n = workspace_size(dims, T)
    if n == 0:
        raise ValueError("invalid dims")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off: off + n]
    _check("dsa_workspace_init", lib().dsa_workspace_init(_p(ws), n, _stream(stream)))
    return ws


def indexer_topk(dims: Dims, q_I, w, k_I_cache, k_I_scale, block_table, seq_lens, q_seq=None, q_pos=None, *, ws,
                 idx=None, stream=None) -> torch.Tensor:
    """idx[T][K] int32: the Top-K causal positions of every query row (ascending, -1 padded)."""
    T = q_I.shape[0]
    if idx is None:
        idx = torch.empty((T, dims.K), dtype=torch.int32, device=q_I.device)
    _check_idx(dims, T, idx)
    st = lib().dsa_indexer_topk(ctypes.byref(dims), _p(q_I), _p(w), _p(k_I_cache), _p(k_I_scale), _p(block_table),
                                _p(seq_lens), _p(q_seq), _p(q_pos), T, _p(idx), _p(ws), ws.numel(), _stream(stream))
    _check("dsa_indexer_topk", st)
    return idx


def indexer_topk_noalloc(dims: Dims, q_I, w, k_I_cache, k_I_scale, block_table, seq_lens, q_seq=None, q_pos=None,
                         *, idx=None, fault_word=None, stream=None) -> torch.Tensor:
    """As :func:`indexer_topk`, without a workspace: the library's static scratch is used.

    ``fault_word`` (optional int32 device tensor of one element) receives the call's fault bits.
    Calls must be ordered on one stream (they share the scratch).
    """
    T = q_I.shape[0]
    if idx is None:
        idx = torch.empty((T, dims.K), dtype=torch.int32, device=q_I.device)
    _check_idx(dims, T, idx)
    st = lib().dsa_indexer_topk_noalloc(ctypes.byref(dims), _p(q_I), _p(w), _p(k_I_cache), _p(k_I_scale),
                                        _p(block_table), _p(seq_lens), _p(q_seq), _p(q_pos), T, _p(idx),
                                        _p(fault_word), _stream(stream))
    _check("dsa_indexer_topk_noalloc", st)
    return idx


def sparse_attn(dims: Dims, q, kv_cache, block_table, seq_lens, idx, sm_scale: float, q_seq=None, *, ws, out=None,
                lse=None, stream=None):
    """(out[T][H][d_v], lse[T][H]) of softmax attention over the rows idx selects."""
    T = q.shape[0]
    odt = torch.float32 if dims.mode == MODES["f32"] else torch.bfloat16
    if out is None:
        out = torch.empty((T, dims.H, dims.d_v), dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((T, dims.H), dtype=torch.float32, device=q.device)
    _check_out(dims, T, out, lse)
    st = lib().dsa_sparse_attn(ctypes.byref(dims), _p(q), _p(kv_cache), _p(block_table), _p(seq_lens), _p(q_seq),
                               _p(idx), T, float(sm_scale), _p(out), _p(lse), _p(ws), ws.numel(), _stream(stream))
    _check("dsa_sparse_attn", st)
    return out, lse


def decode(dims: Dims, q_I, w, k_I_cache, k_I_scale, block_table, seq_lens, q, kv_cache, sm_scale: float, *, ws,
           idx=None, out=None, lse=None, want_idx: bool = True, stream=None):
    """Fused decode step (one query row per sequence): (idx or None, out, lse)."""
    T = dims.B
    odt = torch.float32 if dims.mode == MODES["f32"] else torch.bfloat16
    if idx is None and want_idx:
        idx = torch.empty((T, dims.K), dtype=torch.int32, device=q.device)
    if out is None:
        out = torch.empty((T, dims.H, dims.d_v), dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((T, dims.H), dtype=torch.float32, device=q.device)
    _check_out(dims, T, out, lse)
    if idx is not None and (idx.dtype != torch.int32 or idx.numel() < T * dims.K or not idx.is_contiguous()):
        raise ValueError("idx must be a contiguous int32 tensor of T x K elements")
    st = lib().dsa_decode(ctypes.byref(dims), _p(q_I), _p(w), _p(k_I_cache), _p(k_I_scale), _p(block_table),
                          _p(seq_lens), _p(q), _p(kv_cache), float(sm_scale), _p(idx), _p(out), _p(lse), _p(ws),
                          ws.numel(), _stream(stream))
    _check("dsa_decode", st)
    return idx, out, lse


def cache_append(dims: Dims, k_I_new, kv_new, block_table, seq_lens, k_I_cache, k_I_scale, kv_cache, q_seq=None,
                 q_pos=None, *, ws, stream=None) -> None:
    """Writes new tokens (rows of k_I_new / kv_new) into the paged caches in place."""
    T = kv_new.shape[0]
    st = lib().dsa_cache_append(ctypes.byref(dims), _p(k_I_new), _p(kv_new), _p(block_table), _p(seq_lens), _p(q_seq),
                                _p(q_pos), T, _p(k_I_cache), _p(k_I_scale), _p(kv_cache), _p(ws), ws.numel(),
                                _stream(stream))
    _check("dsa_cache_append", st)


def indexer_prolog(dims: Dims, k_I_new, kv_new, block_table, seq_lens, k_I_cache, k_I_scale, kv_cache, q_I=None,
                   q_seq=None, q_pos=None, *, ws, q_out=None, stream=None):
    """One launch: the cache append of the new tokens (as cache_append) and, when q_I is given
    (DSA_MXFP8), its MXFP8 quantisation into q_out (returned; bf16, q_I's shape)."""
    T_new = 0 if kv_new is None else kv_new.shape[0]
    T_q = 0
    if q_I is not None:
        T_q = q_I.shape[0]
        if q_out is None:
            q_out = torch.empty_like(q_I)
        if q_out.dtype != torch.bfloat16 or q_out.numel() < q_I.numel() or not q_out.is_contiguous():
            raise ValueError("q_out must be a contiguous bf16 tensor of q_I's size")
    st = lib().dsa_indexer_prolog(ctypes.byref(dims), _p(k_I_new), _p(kv_new), _p(block_table), _p(seq_lens),
                                  _p(q_seq), _p(q_pos), T_new, _p(k_I_cache), _p(k_I_scale), _p(kv_cache), _p(q_I), T_q,
                                  _p(q_out), _p(ws), ws.numel(), _stream(stream))
    _check("dsa_indexer_prolog", st)
    return q_out


def summaries_buffer(dims: Dims, device="cuda") -> torch.Tensor:
    """A bf16 [B][pages * 64][d_I] tensor for dsa_block_summaries (pages = ceil(max_blocks / 64))."""
    pages = (dims.max_blocks + 63) // 64
    return torch.zeros((dims.B, pages * 64, dims.d_I), dtype=torch.bfloat16, device=device)


def block_summaries(dims: Dims, k_I_cache, k_I_scale, block_table, seq_lens, summaries, *, ws, stream=None) -> None:
    """Writes the mean key of every valid 64-token block into ``summaries``."""
    st = lib().dsa_block_summaries(ctypes.byref(dims), _p(k_I_cache), _p(k_I_scale), _p(block_table), _p(seq_lens),
                                   _p(summaries), _p(ws), ws.numel(), _stream(stream))
    _check("dsa_block_summaries", st)


def block_summaries_append(dims: Dims, k_I_cache, k_I_scale, block_table, seq_lens, T: int, summaries, q_seq=None,
                           q_pos=None, *, ws, stream=None) -> None:
    """Recomputes the summaries of the blocks that T appended tokens touched."""
    st = lib().dsa_block_summaries_append(ctypes.byref(dims), _p(k_I_cache), _p(k_I_scale), _p(block_table),
                                          _p(seq_lens), _p(q_seq), _p(q_pos), T, _p(summaries), _p(ws), ws.numel(),
                                          _stream(stream))
    _check("dsa_block_summaries_append", st)


def hier_workspace(dims: Dims, T: int, n_sel: int, device="cuda", stream=None) -> torch.Tensor:
    n = int(lib().dsa_hier_workspace_size(ctypes.byref(dims), T, n_sel))
    if n == 0:
        raise ValueError("invalid dims")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off: off + n]
    _check("dsa_workspace_init", lib().dsa_workspace_init(_p(ws), n, _stream(stream)))
    return ws


def indexer_topk_hier(dims: Dims, q_I, w, k_I_cache, k_I_scale, block_table, seq_lens, summaries, n_sel: int,
                      q_seq=None, q_pos=None, *, ws, idx=None, blocks=None, stream=None):
    """(idx[T][K], blocks[T][n_sel]) of hierarchical selection (coarse blocks, then fine tokens)."""
    T = q_I.shape[0]
    if idx is None:
        idx = torch.empty((T, dims.K), dtype=torch.int32, device=q_I.device)
    if blocks is None:
        blocks = torch.empty((T, n_sel), dtype=torch.int32, device=q_I.device)
    st = lib().dsa_indexer_topk_hier(ctypes.byref(dims), _p(q_I), _p(w), _p(k_I_cache), _p(k_I_scale), _p(block_table),
                                     _p(seq_lens), _p(q_seq), _p(q_pos), T, _p(summaries), n_sel, _p(idx), _p(blocks),
                                     _p(ws), ws.numel(), _stream(stream))
    _check("dsa_indexer_topk_hier", st)
    return idx, blocks


def read_error(ws, stream=None) -> int:
    """Synchronises the stream and returns (then clears) the device fault bits of ``ws``."""
    bits = ctypes.c_int32(0)
    st = lib().dsa_read_error(_p(ws), ctypes.byref(bits), _stream(stream))
    if st not in (0, 5, 6):
        raise DsaError("dsa_read_error", st)
    return int(bits.value)


def selftest_wait_timeout(ws, stream=None) -> None:
    """Runs the bounded-wait self-test (its wait runs out after about a second and sets the
    timeout bit of ``ws``; read it with :func:`read_error`)."""
    _check("dsa_selftest_wait_timeout", lib().dsa_selftest_wait_timeout(_p(ws), ws.numel(), _stream(stream)))


def last_launch_count() -> int:
    return int(lib().dsa_last_launch_count())
