"""Benchmark of the decode step of index-selection sparse attention (indexer + Top-K + sparse
attention over a paged KV cache) on GB300, through the library's C ABI.

Default workload: decode, bf16, batch 32, context lengths uniform in [16384, 32768], 64 indexer
heads of 128, Top-K 2048, 128 query heads over a 576-wide latent cache (V = first 512 columns),
64-token blocks, shuffled block table. One step = one dsa_decode call on a batch resident in HBM.
The same JSON line carries the chunked-prefill throughput (2 x 4096 new tokens on a 61,440-token
prefix: indexer + sparse attention calls) under "prefill".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own batch (weak scaling, no collective on the data path);
timing is bracketed by a barrier + synchronize and the maximum over ranks is reported.
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "decode indexer+sparse-attn µs/step & HBM GB/s (%roofline); prefill tokens/s"
WORKLOAD = ("decode_bf16_b32: batch 32, context U{16384..32768}, indexer 64x128 bf16, Top-K 2048, "
            "128 heads x 576 latent (V = 512 cols), 64-token blocks, shuffled block table")
L2_FLUSH_BYTES = 256 << 20
PROFILE = os.path.join(ROOT, "profiles", "indexer_tc_decode_bf16_b32.md")


# ------------------------------------------------------------------------------------------------
# algorithmic traffic of one decode step (the method's own bytes: every causal key once, the
# selected rows once, queries, weights, block-table entries, indices and outputs)
# ------------------------------------------------------------------------------------------------

def _decode_rows(case, rows):
    return np.arange(case.spec.T) if rows is None else np.asarray(rows, dtype=np.int64)


def indexer_bytes(case, rows=None) -> int:
    """Algorithmic bytes of the indexer over decode rows (one query row per sequence): every causal
    key once (with its scales), the row's query and head weights, its block-table entries and
    sequence length, and the K indices written."""
    s = case.spec
    rows = _decode_rows(case, rows)
    key_b = {"f32": 4, "bf16": 2, "bf16_kfp8": 1, "mxfp8": 1}[s.mode] * s.d_I
    n = (case.q_pos[rows].astype(np.int64) + 1).clip(min=0)
    blocks = (n + 63) // 64
    b = int(n.sum()) * key_b
    if s.mode == "bf16_kfp8":
        b += int(blocks.sum()) * 4                              # fp32 scale per block
    if s.mode == "mxfp8":
        b += int(n.sum()) * (s.d_I // 32)                       # E8M0 byte per 32 elements
    act = 4 if s.mode == "f32" else 2
    T = len(rows)
    b += T * s.H_I * s.d_I * act + T * s.H_I * 4               # q_I, w
    b += int(blocks.sum()) * 4 + T * 4                          # block-table entries, seq_lens
    b += T * s.K * 4                                            # idx written
    return b


def attn_bytes(case, rows=None) -> int:
    """Algorithmic bytes of sparse attention: the selected latent rows once, their indices and
    block-table entries, the queries, outputs and log-sum-exps."""
    s = case.spec
    rows = _decode_rows(case, rows)
    act = 4 if s.mode == "f32" else 2
    n_sel = int(np.minimum((case.q_pos[rows].astype(np.int64) + 1).clip(min=0), s.K).sum())
    T = len(rows)
    row_b = s.d + 4 * ((s.d + 127) // 128) if s.kv == "fp8" else s.d * act  # FP8 record: codes + tile scales
    b = n_sel * row_b                                           # gathered rows
    b += T * s.K * 4 + n_sel * 4                                # idx read + table entries
    b += T * s.H * s.d * act + T * s.H * s.d_v * act            # q, out
    b += T * s.H * 4                                            # lse
    return b


def indexer_flops(case, rows=None) -> int:
    """Tensor flops of the indexer scores: every causal (row, key) pair, H_I x d_I MACs."""
    s = case.spec
    rows = _decode_rows(case, rows)
    n = (case.q_pos[rows].astype(np.int64) + 1).clip(min=0)
    return int(n.sum()) * s.H_I * s.d_I * 2


def attn_flops(case, rows=None) -> int:
    """Tensor flops of sparse attention: QK^T over d and PV over d_v for every selected row."""
    s = case.spec
    rows = _decode_rows(case, rows)
    n = np.minimum((case.q_pos[rows].astype(np.int64) + 1).clip(min=0), s.K)
    return int(n.sum()) * s.H * (s.d + s.d_v) * 2


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# every source file the measured indexer call (decode, bf16 keys) is built from: host-side launch
# configuration and workspace layout, the indexer kernel, the merge and their shared headers
TRAFFIC_SOURCES = ("dsa_api.cu", "internal.h", "common.cuh", "ptx.cuh", "indexer_tc.cu", "topk_merge.cu")


def code_only(src: str) -> str:
    """C/C++/CUDA source without its comments, trailing blanks and empty lines (string and
    character literals are kept whole), so that a comment edit leaves the digest unchanged."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def kernel_digest() -> str:
    """SHA-256 prefix over the code (comments removed) of every source of the measured call."""
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        src = open(os.path.join(ROOT, "indexer_top_sparse_paged_gb300", "csrc", f), encoding="utf-8").read()
        h.update(code_only(src).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per indexer launch from the committed ncu summary, if it is for this kernel source."""
    if not os.path.exists(PROFILE):
        return None
    vals = {}
    for line in open(PROFILE):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_digest") != kernel_digest():
        return None
    try:
        return int(vals["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------------------------------------
# multi-rank aggregation (N independent replicas, one GPU each; no collective on the data path)
# ------------------------------------------------------------------------------------------------

def reduce_across_ranks(values, op: str, world: int, device):
    """Element-wise max or sum of `values` over the ranks (every rank calls it; world 1: unchanged)."""
    if world == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    red = torch.distributed.ReduceOp.MAX if op == "max" else torch.distributed.ReduceOp.SUM
    torch.distributed.all_reduce(t, op=red)
    return [float(v) for v in t]


def job_throughput(total_bytes: float, slowest_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return total_bytes / (slowest_ms * 1e-3) / 1e9


# ------------------------------------------------------------------------------------------------
# clock sampling during the timed region
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm, smax, util = float(r[0]), float(r[1]), float(r[2])
            except ValueError:
                continue
            mx = smax
            if util > 0:
                mhz.append(sm)
            for n, v in zip(names, r[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples_under_load": len(mhz)}


# ------------------------------------------------------------------------------------------------
# our implementation
# ------------------------------------------------------------------------------------------------

def to_dev(a, dev):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


class Resident:
    """One workload's inputs in device memory and a workspace (inputs copied once, untimed)."""

    def __init__(self, case, dev):
        import indexer_top_sparse_paged_gb300 as dsa
        s = case.spec
        self.case, self.dev = case, dev
        self.dims = dsa.make_dims(s.mode, s.B, case.max_blocks, case.num_blocks, s.H_I, s.d_I, s.H, s.d, s.d_v, s.K,
                                  kv=s.kv)
        self.q_I, self.w, self.k_I = to_dev(case.q_I, dev), to_dev(case.w, dev), to_dev(case.k_I, dev)
        self.ksc = to_dev(case.k_I_scale, dev) if case.k_I_scale is not None else None
        self.q, self.kv = to_dev(case.q, dev), to_dev(case.kv, dev)
        self.bt, self.sl = to_dev(case.block_table, dev), to_dev(case.seq_lens, dev)
        self.qs, self.qp = to_dev(case.q_seq, dev), to_dev(case.q_pos, dev)
        self.ws = dsa.workspace(self.dims, s.T, dev)
        self.idx = torch.empty((s.T, s.K), dtype=torch.int32, device=dev)
        odt = torch.float32 if s.mode == "f32" else torch.bfloat16
        self.out = torch.empty((s.T, s.H, s.d_v), dtype=odt, device=dev)
        self.lse = torch.empty((s.T, s.H), dtype=torch.float32, device=dev)

    def indexer(self):
        import indexer_top_sparse_paged_gb300 as dsa
        dsa.indexer_topk(self.dims, self.q_I, self.w, self.k_I, self.ksc, self.bt, self.sl, self.qs, self.qp,
                         ws=self.ws, idx=self.idx)

    def attn(self):
        import indexer_top_sparse_paged_gb300 as dsa
        dsa.sparse_attn(self.dims, self.q, self.kv, self.bt, self.sl, self.idx, self.case.spec.sm_scale, q_seq=self.qs,
                        ws=self.ws, out=self.out, lse=self.lse)


def run_prefill(steps: int, warmup: int, dev, flush):
    """Chunked prefill (2 x 4096 new tokens on 61,440 cached, Top-K 2048): indexer and sparse
    attention calls timed with CUDA events on the current stream, L2 flushed before each."""
    import indexer_top_sparse_paged_gb300 as dsa
    spec, seed = W.named(4)
    case = W.generate(spec, seed)
    r = Resident(case, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, warmup)):
        r.indexer()
        r.attn()
    torch.cuda.synchronize(dev)
    if dsa.read_error(r.ws) != 0:
        raise RuntimeError("device fault bits set during the prefill warm-up")
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        r.indexer()
        ev[i][1].record(stream)
        r.attn()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    if dsa.read_error(r.ws) != 0:
        raise RuntimeError("device fault bits set during the prefill timing")
    idx_ms = statistics.median(a.elapsed_time(b) for a, b, _ in ev)
    att_ms = statistics.median(b.elapsed_time(c) for _, b, c in ev)
    peak, kind = measured_tensor_peak()
    fi, fa = indexer_flops(case), attn_flops(case)
    res = {
        "workload": "prefill_2x4096_64k: 2 sequences x 4096 new tokens at positions 61440..65535, indexer 64x128 bf16, "
                    "Top-K 2048 per row, 128 heads x 576 latent",
        "tokens_per_s": round(spec.T / ((idx_ms + att_ms) * 1e-3), 1),
        "indexer_ms": round(idx_ms, 3),
        "attn_ms": round(att_ms, 3),
        "indexer_tflops": round(fi / (idx_ms * 1e-3) / 1e12, 1),
        "attn_tflops": round(fa / (att_ms * 1e-3) / 1e12, 1),
        "tensor_peak_tflops": peak,
        "indexer_tensor_frac_of_" + kind: round(fi / (idx_ms * 1e-3) / 1e12 / peak, 4),
        "attn_tensor_frac_of_" + kind: round(fa / (att_ms * 1e-3) / 1e12 / peak, 4),
        "indexer_flops": fi,
        "attn_flops": fa,
        "steps": steps,
        "l2": "flushed (256 MiB write) before every timed step",
        "gpu_launches_per_step": None,
    }
    r.indexer()
    n_idx = dsa.last_launch_count()
    r.attn()
    res["gpu_launches_per_step"] = n_idx + dsa.last_launch_count()
    del r
    torch.cuda.empty_cache()
    # the indexer over the same keys stored in the two 8-bit formats (scores on the same GEMM)
    res["indexer_key_formats"] = {}
    for mode in ("bf16_kfp8", "mxfp8"):
        r = Resident(W.with_key_format(case, mode), dev)
        for _ in range(3):
            r.indexer()
        evk = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            evk[i][0].record(stream)
            r.indexer()
            evk[i][1].record(stream)
        torch.cuda.synchronize(dev)
        if dsa.read_error(r.ws) != 0:
            raise RuntimeError(f"device fault bits set while timing the {mode} prefill indexer")
        ms = statistics.median(a.elapsed_time(b) for a, b in evk)
        res["indexer_key_formats"][mode] = {"indexer_ms": round(ms, 3),
                                            "indexer_tflops": round(fi / (ms * 1e-3) / 1e12, 1)}
        del r
        torch.cuda.empty_cache()
    return res


def run_key_formats(case, steps: int, dev, flush):
    """The decode indexer over the same keys re-stored in the two 8-bit formats (FP8 e4m3 with a
    per-block scale, MXFP8): CUDA-event time per call with L2 flushed, algorithmic bytes, HBM
    fraction. The attention half of the step does not read the indexer keys."""
    import indexer_top_sparse_paged_gb300 as dsa
    peak, kind = measured_peaks()
    res = {}
    stream = torch.cuda.current_stream(dev)
    for mode in ("bf16_kfp8", "mxfp8"):
        c = W.with_key_format(case, mode)
        s = c.spec
        dims = dsa.make_dims(mode, s.B, c.max_blocks, c.num_blocks, s.H_I, s.d_I, s.H, s.d, s.d_v, s.K)
        q_I, w, k_I, ksc = to_dev(c.q_I, dev), to_dev(c.w, dev), to_dev(c.k_I, dev), to_dev(c.k_I_scale, dev)
        bt, sl = to_dev(c.block_table, dev), to_dev(c.seq_lens, dev)
        ws = dsa.workspace(dims, s.T, dev)
        idx = torch.empty((s.T, s.K), dtype=torch.int32, device=dev)
        for _ in range(3):
            dsa.indexer_topk(dims, q_I, w, k_I, ksc, bt, sl, ws=ws, idx=idx)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            dsa.indexer_topk(dims, q_I, w, k_I, ksc, bt, sl, ws=ws, idx=idx)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        if dsa.read_error(ws) != 0:
            raise RuntimeError(f"device fault bits set while timing the {mode} indexer")
        us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
        ib = indexer_bytes(c)
        res[mode] = {"indexer_us": round(us, 2), "indexer_bytes": ib, "gbs": round(ib / (us * 1e-6) / 1e9, 1),
                     "hbm_frac_of_" + kind: round(ib / (us * 1e-6) / 1e9 / peak, 4),
                     "gpu_launches": dsa.last_launch_count()}
        del q_I, w, k_I, ksc, bt, sl, ws, idx
    torch.cuda.empty_cache()
    return res


def _med_us(fn, steps: int, flush, stream) -> float:
    """Median CUDA-event time of fn() in microseconds, L2 flushed (256 MiB write) before each call."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3


def _hbm(nbytes: int, us: float, peak: float, kind: str) -> dict:
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"bytes": nbytes, "gbs": round(gbs, 1), "hbm_frac_of_" + kind: round(gbs / peak, 4)}


def _tensor(flops: int, us: float, peak: float, kind: str) -> dict:
    tf = flops / (us * 1e-6) / 1e12
    return {"flops": flops, "tflops": round(tf, 1), "tensor_frac_of_" + kind: round(tf / peak, 4)}


class _Rows:
    """A contiguous range of query rows of a resident workload, as views (no copies)."""

    def __init__(self, r: "Resident", lo: int, hi: int):
        self.r, self.lo, self.hi = r, lo, hi
        self.idx = r.idx[lo:hi]

    def indexer(self):
        import indexer_top_sparse_paged_gb300 as dsa
        r = self.r
        dsa.indexer_topk(r.dims, r.q_I[self.lo:self.hi], r.w[self.lo:self.hi], r.k_I, r.ksc, r.bt, r.sl,
                         r.qs[self.lo:self.hi], r.qp[self.lo:self.hi], ws=r.ws, idx=self.idx)

    def attn(self):
        import indexer_top_sparse_paged_gb300 as dsa
        r = self.r
        dsa.sparse_attn(r.dims, r.q[self.lo:self.hi], r.kv, r.bt, r.sl, self.idx, r.case.spec.sm_scale,
                        q_seq=r.qs[self.lo:self.hi], ws=r.ws, out=r.out[self.lo:self.hi], lse=r.lse[self.lo:self.hi])


def run_workloads(steps: int, dev, flush) -> dict:
    """The other named workloads at full size, each call timed on its own (median CUDA-event time,
    L2 flushed before each call), with its algorithmic bytes or flops and the fraction of the
    measured peak:
      1  tiny decode, fp32 (L = 2048, K = 256): launch- and latency-bound, reported in microseconds;
      3  1M-token decode with FP8 indexer keys: HBM-bound;
      5  mixed serving batch (64 decode rows, contexts log-uniform in [1K, 256K], plus one 2048-token
         chunk at 128K, FP8 keys): the whole step (one indexer call and one attention call over all
         2112 rows), and its decode rows and chunk rows as separate calls."""
    import indexer_top_sparse_paged_gb300 as dsa
    hbm_peak, hk = measured_peaks()
    tc_peak, tk = measured_tensor_peak()
    stream = torch.cuda.current_stream(dev)
    out = {}
    for n in (1, 3, 5):
        t0 = time.time()
        spec, seed = W.named(n)
        case = W.generate(spec, seed)
        gen_s = time.time() - t0
        r = Resident(case, dev)
        s = case.spec
        for _ in range(3):
            r.indexer()
            r.attn()
        torch.cuda.synchronize(dev)
        if dsa.read_error(r.ws) != 0:
            raise RuntimeError(f"device fault bits set during the warm-up of workload {n}")
        res = {"workload": s.name, "T": s.T, "B": s.B, "K": s.K, "mode": s.mode, "generate_s": round(gen_s, 1)}
        if n in (1, 3):
            res["indexer_us"] = round(_med_us(r.indexer, steps, flush, stream), 2)
            res["attn_us"] = round(_med_us(r.attn, steps, flush, stream), 2)

            def step():
                dsa.decode(r.dims, r.q_I, r.w, r.k_I, r.ksc, r.bt, r.sl, r.q, r.kv, s.sm_scale, ws=r.ws, idx=r.idx,
                           out=r.out, lse=r.lse)
            res["step_us"] = round(_med_us(step, steps, flush, stream), 2)
            res["step_launches"] = dsa.last_launch_count()
            ib, ab = indexer_bytes(case), attn_bytes(case)
            res["step"] = _hbm(ib + ab, res["step_us"], hbm_peak, hk)
            res["indexer"] = _hbm(ib, res["indexer_us"], hbm_peak, hk)
            res["attn"] = _hbm(ab, res["attn_us"], hbm_peak, hk)
        else:
            n_dec = int(sum(1 for x in s.new_tokens if x == 1))
            dec, chunk = _Rows(r, 0, n_dec), _Rows(r, n_dec, s.T)
            res["total_step_us"] = round(_med_us(lambda: (r.indexer(), r.attn()), steps, flush, stream), 2)
            res["total_indexer_us"] = round(_med_us(r.indexer, steps, flush, stream), 2)
            res["total_attn_us"] = round(_med_us(r.attn, steps, flush, stream), 2)
            drows = np.arange(n_dec)
            d = {"rows": n_dec, "indexer_us": round(_med_us(dec.indexer, steps, flush, stream), 2),
                 "attn_us": round(_med_us(dec.attn, steps, flush, stream), 2)}
            d["step_us"] = round(_med_us(lambda: (dec.indexer(), dec.attn()), steps, flush, stream), 2)
            d.update(_hbm(indexer_bytes(case, drows) + attn_bytes(case, drows), d["step_us"], hbm_peak, hk))
            crows = np.arange(n_dec, s.T)
            c = {"rows": s.T - n_dec, "indexer_us": round(_med_us(chunk.indexer, steps, flush, stream), 2),
                 "attn_us": round(_med_us(chunk.attn, steps, flush, stream), 2)}
            c["tokens_per_s"] = round(c["rows"] / ((c["indexer_us"] + c["attn_us"]) * 1e-6), 1)
            c["indexer"] = _tensor(indexer_flops(case, crows), c["indexer_us"], tc_peak, tk)
            c["attn"] = _tensor(attn_flops(case, crows), c["attn_us"], tc_peak, tk)
            res["decode_rows"] = d
            res["chunk_rows"] = c
        if dsa.read_error(r.ws) != 0:
            raise RuntimeError(f"device fault bits set while timing workload {n}")
        out[str(n)] = res
        del r, case
        torch.cuda.empty_cache()
    out["method"] = ("median CUDA-event time per call over %d calls, L2 flushed (256 MiB write) before each; "
                     "bytes and flops are the method's own (every causal key once, the selected rows once)" % steps)
    return out


def run_latent_formats(case, steps: int, dev, flush) -> dict:
    """The decode workload with its latent rows stored as FP8 records (e4m3 codes, one fp32 scale per
    128 elements): the attention call alone, and the whole decode step with bf16 and with FP8
    indexer keys (CUDA events, L2 flushed before each call, medians)."""
    import indexer_top_sparse_paged_gb300 as dsa
    peak, kind = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    res = {}
    for keys in ("bf16", "bf16_kfp8"):
        c = W.with_kv_format(case if keys == "bf16" else W.with_key_format(case, keys), "fp8")
        r = Resident(c, dev)
        s = c.spec

        def step():
            dsa.decode(r.dims, r.q_I, r.w, r.k_I, r.ksc, r.bt, r.sl, r.q, r.kv, s.sm_scale, ws=r.ws, idx=r.idx,
                       out=r.out, lse=r.lse)
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
        step_us = _med_us(step, steps, flush, stream)
        ent = {"step_us": round(step_us, 2), "step_launches": dsa.last_launch_count()}
        ent.update(_hbm(indexer_bytes(c) + attn_bytes(c), step_us, peak, kind))
        if keys == "bf16":
            au = _med_us(r.attn, steps, flush, stream)
            ent["attn_us"] = round(au, 2)
            ent["attn"] = _hbm(attn_bytes(c), au, peak, kind)
        if dsa.read_error(r.ws) != 0:
            raise RuntimeError("device fault bits set while timing the FP8 latent cache")
        res["keys_" + keys] = ent
        del r
        torch.cuda.empty_cache()
    res["record_bytes"] = dsa.kv_record_bytes(case.spec.d)
    return res


def run_ours(args, rank, world):
    import indexer_top_sparse_paged_gb300 as dsa

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    spec, seed = W.named(2)
    case = W.generate(spec, seed + 1000 * rank)
    s = case.spec
    dims = dsa.make_dims(s.mode, s.B, case.max_blocks, case.num_blocks, s.H_I, s.d_I, s.H, s.d, s.d_v, s.K)
    q_I, w, k_I = to_dev(case.q_I, dev), to_dev(case.w, dev), to_dev(case.k_I, dev)
    q, kv = to_dev(case.q, dev), to_dev(case.kv, dev)
    bt, sl = to_dev(case.block_table, dev), to_dev(case.seq_lens, dev)
    ws = dsa.workspace(dims, s.T, dev)
    idx = torch.empty((s.T, s.K), dtype=torch.int32, device=dev)
    out = torch.empty((s.T, s.H, s.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((s.T, s.H), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        dsa.decode(dims, q_I, w, k_I, None, bt, sl, q, kv, s.sm_scale, ws=ws, idx=idx, out=out, lse=lse)
        return dsa.last_launch_count()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if dsa.read_error(ws) != 0:
        raise RuntimeError("device fault bits set during warm-up")

    sampler = ClockSampler(dev.index)
    sampler.start()
    t_burst = time.time()
    while time.time() - t_burst < 0.6:   # load the GPU so the sampler sees clocks under load
        for _ in range(20):
            flush.zero_()
            step()
        torch.cuda.synchronize(dev)

    # --- timed region: K steps, L2 flushed before each, CUDA events on the launching stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches = 0
    barrier()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        launches += step()
        ev[i][1].record(stream)
    barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # --- per-stage breakdown (same work, split into its two ABI calls) for the roofline
    ev3 = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev3[i][0].record(stream)
        dsa.indexer_topk(dims, q_I, w, k_I, None, bt, sl, ws=ws, idx=idx)
        ev3[i][1].record(stream)
        dsa.sparse_attn(dims, q, kv, bt, sl, idx, s.sm_scale, ws=ws, out=out, lse=lse)
        ev3[i][2].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    idx_ms = [a.elapsed_time(b) for a, b, _ in ev3]
    att_ms = [b.elapsed_time(c) for _, b, c in ev3]

    # --- end to end through the public API with host buffers (pinned), copies inside the region:
    #     the step's inputs travel in one staging buffer (one host->device copy), and out and idx
    #     come back in one (one device->host copy)
    def packed(arrays):
        offs, off = [], 0
        for a in arrays:
            offs.append(off)
            off = (off + a.nbytes + 255) // 256 * 256
        return offs, off

    host_in = [np.ascontiguousarray(a) for a in (case.q_I, case.w, case.q, case.block_table, case.seq_lens)]
    in_offs, in_bytes = packed(host_in)
    h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    for a, o in zip(host_in, in_offs):
        h_in[o:o + a.nbytes].copy_(torch.from_numpy(a.view(np.uint8).reshape(-1)))
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)

    def view(buf, o, dtype, shape):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        return buf[o:o + n].view(dtype).view(shape)

    e_qI = view(d_in, in_offs[0], torch.bfloat16, case.q_I.shape)
    e_w = view(d_in, in_offs[1], torch.float32, case.w.shape)
    e_q = view(d_in, in_offs[2], torch.bfloat16, case.q.shape)
    e_bt = view(d_in, in_offs[3], torch.int32, case.block_table.shape)
    e_sl = view(d_in, in_offs[4], torch.int32, case.seq_lens.shape)
    o_off1 = (s.T * s.H * s.d_v * 2 + 255) // 256 * 256
    o_bytes = o_off1 + s.T * s.K * 4
    d_out = torch.empty(o_bytes, dtype=torch.uint8, device=dev)
    e_out = view(d_out, 0, torch.bfloat16, (s.T, s.H, s.d_v))
    e_idx = view(d_out, o_off1, torch.int32, (s.T, s.K))
    h_out = torch.empty(o_bytes, dtype=torch.uint8).pin_memory()
    h2d = sum(a.nbytes for a in host_in)
    d2h = s.T * s.H * s.d_v * 2 + s.T * s.K * 4

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        dsa.decode(dims, e_qI, e_w, k_I, None, e_bt, e_sl, e_q, kv, s.sm_scale, ws=ws, idx=e_idx, out=e_out, lse=lse)
        h_out.copy_(d_out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        flush.zero_()
        e2e_ev[i][0].record(stream)
        e2e_step()
        e2e_ev[i][1].record(stream)
    barrier()
    e2e_ms = [a.elapsed_time(b) for a, b in e2e_ev]
    # the host copy of the last step's result is the device result
    got_idx = h_out[o_off1:o_off1 + s.T * s.K * 4].view(torch.int32).view(s.T, s.K)
    if not torch.equal(got_idx, idx.cpu()):
        raise RuntimeError("end-to-end indices differ from the device-resident step's")

    if dsa.read_error(ws) != 0:
        raise RuntimeError("device fault bits set during the timed region")

    # --- cache append of the step's new tokens (the step before the path; runs after the decode
    #     timing because it rewrites the caches in place)
    rng = np.random.default_rng(77)
    k_new = to_dev(W.to_bf16_bits(rng.standard_normal((s.T, s.d_I), dtype=np.float32)), dev)
    kv_new = to_dev(W.to_bf16_bits(rng.standard_normal((s.T, s.d), dtype=np.float32)), dev)
    app_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        app_ev[i][0].record(stream)
        dsa.cache_append(dims, k_new, kv_new, bt, sl, k_I, None, kv, ws=ws)
        app_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if dsa.read_error(ws) != 0:
        raise RuntimeError("device fault bits set during the cache append")
    app_us = statistics.median(a.elapsed_time(b) for a, b in app_ev) * 1e3
    app_bytes = 2 * s.T * (s.d_I + s.d) * 2  # new rows read + cache rows written (bf16)

    ib, ab = indexer_bytes(case), attn_bytes(case)
    step_bytes = ib + ab
    # per-step medians (CUDA events), the slowest rank's; the K bracketed steps' total beside them
    total_ms, e2e_total, ms_per_step, e2e_med = reduce_across_ranks(
        [sum(step_ms), sum(e2e_ms), statistics.median(step_ms), statistics.median(e2e_ms)], "max", world, dev)
    (job_bytes,) = reduce_across_ranks([step_bytes], "sum", world, dev)
    value = job_throughput(job_bytes, ms_per_step)
    e2e_value = job_throughput(job_bytes, e2e_med)
    peak, peak_kind = measured_peaks()
    idx_avg = statistics.median(idx_ms)
    achieved = ib / (idx_avg * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "timing": "median of the K per-step CUDA-event times (slowest rank); mean over the K bracketed steps "
                  f"{total_ms / args.steps * 1e3:.2f} us",
        "hbm_frac_of_" + peak_kind: round(value / world / peak, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) values, U(0,1) head weights, shuffled block table)",
        "config": {"workload": WORKLOAD, "global_batch": s.B * world, "seq_len": "16384..32768",
                   "parallelism": f"replicas x{world}", "l2": "flushed (256 MiB write) before every timed step",
                   "step_bytes": step_bytes, "indexer_bytes": ib, "attention_bytes": ab},
        "breakdown_us": {"indexer_topk": round(idx_avg * 1e3, 2), "sparse_attn": round(statistics.median(att_ms) * 1e3, 2)},
        "roofline": {"kernel": "dsa_indexer_topk (indexer_tc_kernel + topk_merge)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
                     "algorithmic_bytes_per_launch": ib},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_med, 5)},
        "gpu_launches": launches,
        "clocks": clocks,
        "cache_append": {"us": round(app_us, 2), "rows": s.T, "bytes": app_bytes,
                         "note": "dsa_cache_append of the batch's new keys and latent rows (launch-bound at 32 rows)"},
    }
    res["indexer_key_formats"] = run_key_formats(case, max(3, min(args.steps, 20)), dev, flush)
    res["latent_fp8"] = run_latent_formats(case, max(3, min(args.steps, 20)), dev, flush)
    if not args.no_prefill:
        res["prefill"] = run_prefill(max(3, min(args.steps, 10)), args.warmup, dev, flush)
    if not args.no_workloads:
        res["workloads"] = run_workloads(max(3, min(args.steps, 20)), dev, flush)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(case)
    return res


# ------------------------------------------------------------------------------------------------
# oracle (CPU) baseline
# ------------------------------------------------------------------------------------------------

def sample_case(case, n_seq: int):
    """The first n_seq sequences of a decode case (a bounded sample of the same workload)."""
    sub = W.Case(case.spec, case.seed, case.block_table[:n_seq], case.seq_lens[:n_seq], case.q_seq[:n_seq],
                 case.q_pos[:n_seq], case.q_I[:n_seq], case.w[:n_seq], case.k_I, case.k_I_scale, case.q[:n_seq],
                 case.kv)
    sub.spec = W.Spec(case.spec.name, case.spec.mode, list(case.spec.seq_lens[:n_seq]), [1] * n_seq,
                      case.spec.H_I, case.spec.d_I, case.spec.H, case.spec.d, case.spec.d_v, case.spec.K)
    return sub


def time_oracle(sub, threads: int) -> float:
    import oracle
    t0 = time.perf_counter()
    idx, _ = oracle.indexer_topk(sub, threads=threads)
    oracle.sparse_attn(sub, idx, threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(case, n_seq: int = 32, n_seq_single: int = 8):
    """The oracle as it stands on the host cores: all 32 decode rows with one thread per core, and
    a sample of the rows on one thread."""
    threads = os.cpu_count() or 1
    sub = sample_case(case, n_seq)
    dt = time_oracle(sub, threads)
    b = indexer_bytes(sub) + attn_bytes(sub)
    sub1 = sample_case(case, n_seq_single)
    dt1 = time_oracle(sub1, 1)
    b1 = indexer_bytes(sub1) + attn_bytes(sub1)
    return {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_seq} of the 32 decode sequences (indexer + Top-K + attention, fp64), {dt:.2f} s",
            "single_thread": {"value": round(b1 / dt1 / 1e9, 5), "unit": "GB/s", "cores": 1,
                              "sample": f"the first {n_seq_single} of the 32 decode sequences, {dt1:.2f} s"}}


def run_reference(args, rank, world):
    spec, seed = W.named(2)
    case = W.generate(spec, seed)
    threads = os.cpu_count() or 1
    sub = sample_case(case, 2)
    for _ in range(max(0, min(args.warmup, 1))):
        time_oracle(sub, threads)
    times = [time_oracle(sub, threads) for _ in range(args.steps)]
    b = indexer_bytes(sub) + attn_bytes(sub)
    total = sum(times)
    value = b * args.steps / total / 1e9
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) values, U(0,1) head weights, shuffled block table)",
        "config": {"workload": WORKLOAD, "global_batch": s_b(case), "seq_len": "16384..32768",
                   "parallelism": "cpu oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": "2 of the 32 decode sequences per step (indexer + Top-K + attention, fp64)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile(args):
    """warmup + 1 steps of one case and nothing else (for ncu):
      decode         the default workload (fused decode steps),
      prefill        the chunked prefill workload at full size (indexer + attention calls),
      prefill-small  2 x 2048 new tokens on 16,384 (a small case of the prefill kernels),
      decode-fp8     the default workload's keys stored as FP8 e4m3 with a per-block scale,
      decode-mx      the default workload's keys stored as MXFP8,
      decode-kv8     the default workload's latent rows stored as FP8 records."""
    import indexer_top_sparse_paged_gb300 as dsa

    dev = torch.device("cuda", 0)
    if args.profile in ("prefill", "prefill-small"):
        spec, seed = W.named(4)
        if args.profile == "prefill-small":
            spec = W.prefill_chunk(B=2, new=2048, total=16384)
        r = Resident(W.generate(spec, seed), dev)
        for _ in range(args.warmup + 1):
            r.indexer()
            r.attn()
        torch.cuda.synchronize(dev)
        assert dsa.read_error(r.ws) == 0
        return
    spec, seed = W.named(2)
    case = W.generate(spec, seed)
    if args.profile in ("decode-fp8", "decode-mx"):
        case = W.with_key_format(case, "bf16_kfp8" if args.profile == "decode-fp8" else "mxfp8")
    if args.profile == "decode-kv8":
        case = W.with_kv_format(case, "fp8")
    s = case.spec
    dims = dsa.make_dims(s.mode, s.B, case.max_blocks, case.num_blocks, s.H_I, s.d_I, s.H, s.d, s.d_v, s.K, kv=s.kv)
    q_I, w, k_I = to_dev(case.q_I, dev), to_dev(case.w, dev), to_dev(case.k_I, dev)
    ksc = to_dev(case.k_I_scale, dev) if case.k_I_scale is not None else None
    q, kv = to_dev(case.q, dev), to_dev(case.kv, dev)
    bt, sl = to_dev(case.block_table, dev), to_dev(case.seq_lens, dev)
    ws = dsa.workspace(dims, s.T, dev)
    for _ in range(args.warmup + 1):
        dsa.decode(dims, q_I, w, k_I, ksc, bt, sl, q, kv, s.sm_scale, ws=ws)
    torch.cuda.synchronize(dev)
    assert dsa.read_error(ws) == 0


def s_b(case):
    return case.spec.B


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the chunked-prefill measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the tiny, 1M-token and mixed-batch workloads (measured after the headline)")
    ap.add_argument("--profile", nargs="?", const="decode",
                    choices=["decode", "prefill", "prefill-small", "decode-fp8", "decode-mx", "decode-kv8"],
                    help="only run --warmup + 1 steps of one case (a short command for ncu captures)")
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
