"""GPU-side test helpers: move a generated case to the device and call the library through its
C ABI (the Python binding only marshals pointers)."""
from __future__ import annotations

import numpy as np
import torch

import indexer_top_sparse_paged_gb300 as dsa
import oracle
from cases import check_index_row, kv_fp8_decode, np_bf16

ATOL = {"f32": 1e-4, "bf16": 2e-2, "bf16_kfp8": 2e-2, "mxfp8": 2e-2}
LSE_TOL = {"f32": 1e-4, "bf16": 2e-3, "bf16_kfp8": 2e-3, "mxfp8": 2e-3}


def _t(a, dev):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


class Dev:
    """Device copies of one case plus its dims and a workspace."""

    def __init__(self, case, device="cuda", T=None):
        s = case.spec
        self.case = case
        self.dims = dsa.make_dims(s.mode, s.B, case.max_blocks, case.num_blocks, s.H_I, s.d_I, s.H, s.d, s.d_v, s.K,
                                  kv=s.kv)
        self.q_I = _t(case.q_I, device)
        self.w = _t(case.w, device)
        self.k_I = _t(case.k_I, device)
        self.k_I_scale = _t(case.k_I_scale, device)
        self.q = _t(case.q, device)
        self.kv = _t(case.kv, device)
        self.block_table = _t(case.block_table, device)
        self.seq_lens = _t(case.seq_lens, device)
        self.q_seq = _t(case.q_seq, device)
        self.q_pos = _t(case.q_pos, device)
        self.T = s.T if T is None else T
        self.ws = dsa.workspace(self.dims, self.T, device)
        self.decode_shaped = all(n == 1 for n in s.new_tokens)

    def indexer(self, explicit_rows: bool = True) -> np.ndarray:
        if explicit_rows:
            idx = dsa.indexer_topk(self.dims, self.q_I, self.w, self.k_I, self.k_I_scale, self.block_table,
                                   self.seq_lens, self.q_seq, self.q_pos, ws=self.ws)
        else:
            idx = dsa.indexer_topk(self.dims, self.q_I, self.w, self.k_I, self.k_I_scale, self.block_table,
                                   self.seq_lens, ws=self.ws)
        torch.cuda.synchronize()
        return idx.cpu().numpy()

    def attn(self, idx_np: np.ndarray):
        idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int32)).cuda()
        out, lse = dsa.sparse_attn(self.dims, self.q, self.kv, self.block_table, self.seq_lens, idx,
                                   self.case.spec.sm_scale, q_seq=self.q_seq, ws=self.ws)
        torch.cuda.synchronize()
        return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)

    def decode(self):
        idx, out, lse = dsa.decode(self.dims, self.q_I, self.w, self.k_I, self.k_I_scale, self.block_table,
                                   self.seq_lens, self.q, self.kv, self.case.spec.sm_scale, ws=self.ws)
        torch.cuda.synchronize()
        return idx.cpu().numpy(), out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)

    def faults(self) -> int:
        return dsa.read_error(self.ws)


def assert_index_parity(case, gpu_idx, rows=None, K=None):
    """Every row passes the index rule against the fp64 oracle (exact where the K-th gap > 1e-3)."""
    K = case.spec.K if K is None else K
    sel = np.arange(case.spec.T) if rows is None else np.asarray(rows)
    S = oracle.index_scores(case, rows=sel)
    o_idx, kth = oracle.indexer_topk(case, rows=sel)
    bad = []
    exact_rows = 0
    for r, t in enumerate(sel):
        n = int(case.q_pos[t]) + 1
        n = max(n, 0)
        g = gpu_idx[t]
        valid = g[g >= 0]
        # valid entries first, ascending, then -1
        m = len(valid)
        if not (np.all(g[:m] >= 0) and np.all(g[m:] == -1) and np.all(np.diff(valid) > 0)):
            bad.append((int(t), "layout: expected ascending positions then -1"))
            continue
        msg = check_index_row(g, o_idx[r], S[r, :n], K, kth[r] if n > K else None)
        if msg:
            bad.append((int(t), msg))
        if n > K:
            sk, sk1 = kth[r]
            if sk != 0 and (sk - sk1) / abs(sk) > 1e-3:
                exact_rows += 1
    assert not bad, f"index parity failed on {len(bad)} rows: {bad[:5]}"
    return exact_rows


def kv_fp8_logit_bound(case, gpu_idx, rows):
    """With an FP8 latent cache the GPU rounds every element code * scale to bf16 (relative error at
    most 2^-8) before its products, so each logit z_i = sm_scale * q . k_i moves by at most
    sm_scale * 2^-8 * sum_c |q_c| |k_ic|, and lse = log sum exp z by at most the largest of those:
    the bound per (row, head), from the exactly decoded rows."""
    s = case.spec
    bound = np.zeros((len(rows), s.H))
    for n, t in enumerate(rows):
        sel = gpu_idx[t][gpu_idx[t] >= 0]
        if len(sel) == 0:
            continue
        b, bs = int(case.q_seq[t]), s.block_size
        k = np.abs(kv_fp8_decode(case.kv[case.block_table[b, sel // bs], sel % bs], s.d))  # [n, d]
        q = np.abs(np_bf16(case.q[t]))                                  # [H, d]
        bound[n] = s.sm_scale * 2.0 ** -8 * (q @ k.T).max(axis=1)
    return bound


def assert_attn_parity(case, gpu_idx, out, lse, rows=None):
    mode = case.spec.mode
    sel = np.arange(case.spec.T) if rows is None else np.asarray(rows)
    o_out, o_lse, psum = oracle.sparse_attn(case, gpu_idx[sel], rows=sel)
    err = np.abs(out[sel] - o_out).max() if len(sel) else 0.0
    assert err <= ATOL[mode], f"attention max-abs error {err:.3g} > {ATOL[mode]}"
    fin = np.isfinite(o_lse)
    assert np.array_equal(np.isfinite(lse[sel]), fin), "lse finiteness differs"
    if fin.any():
        tol = np.full(o_lse.shape, LSE_TOL[mode])
        if case.spec.kv == "fp8":
            tol = tol + kv_fp8_logit_bound(case, gpu_idx, sel)
        lerr = np.abs(lse[sel][fin] - o_lse[fin])
        assert np.all(lerr <= tol[fin]), f"lse error {lerr.max():.3g} over its bound {tol[fin][np.argmax(lerr - tol[fin])]:.3g}"
    return float(err)
