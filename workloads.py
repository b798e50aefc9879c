"""Seeded synthetic inputs for index-selection sparse attention over a paged KV cache.

This module is shared by the fp64 oracle (``oracle/``) and the CUDA path
(``indexer_top_sparse_paged_gb300``) and holds none of the method's arithmetic:
it only draws random values, rounds them to their storage types and lays them
out in a paged cache.

* Values: ``q, kv, q_I, k_I ~ N(0,1)``; head weights ``w ~ U(0,1)`` (fp32).
* Storage: fp32, bf16 (round to nearest even) or OCP FP8 e4m3 indexer keys with
  one fp32 scale per 64-token physical block (``scale = amax/448``, codes
  rounded to nearest even, saturating at 448), or MXFP8 indexer keys (OCP
  Microscaling: e4m3 codes with one E8M0 scale byte per 32 elements of a key,
  quantised from the bf16-rounded draw).
* Paging: every sequence's logical 64-token blocks are placed in a pool of
  physical blocks by a seeded random permutation (plus a few spare blocks),
  recorded in ``block_table[B][max_blocks]``; unused table entries are -1.
  Cache slots that hold no token (the tail of a sequence's last block and the
  spare blocks) are filled with a large finite poison value (64.0 / e4m3 code
  0x7E), so a kernel that reads them gives visibly wrong results.
* Queries: a sequence ``b`` with ``n_b`` query tokens has them at absolute
  positions ``L_b - n_b .. L_b - 1`` (decode: ``n_b = 1``); their keys are
  already in the cache.

The five named workloads follow the problem statement of "index-selection
sparse attention for long-context decode and prefill" (lightweight indexer
page, §2.1 "Core Pipeline Operator Fusion" and the Day-0 GPU guide §3): tiny
fp32 decode, bf16 decode at batch 32, 1M-token decode with FP8 indexer keys,
chunked prefill and a mixed serving batch.  Seeds are the workload numbers
1..5 and the generator is NumPy's PCG64, so every machine draws the same bits.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 64
POISON = 64.0
POISON_E4M3 = 0x7E  # 448: the largest finite e4m3 code


@dataclass
class Spec:
    """Shapes of one workload.

    ``seq_lens[b]`` counts the cached positions of sequence ``b`` including its
    new tokens; ``new_tokens[b]`` is the number of query tokens of ``b``.
    """

    name: str
    mode: str  # "f32" | "bf16" | "bf16_kfp8" | "mxfp8"
    seq_lens: list
    new_tokens: list
    H_I: int
    d_I: int
    H: int
    d: int
    d_v: int
    K: int
    block_size: int = BLOCK
    spare_blocks: int = 3
    meta: dict = field(default_factory=dict)
    kv: str = "act"  # latent rows: "act" (the mode's activation type) | "fp8" (FP8 records, bf16 modes)

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def T(self) -> int:
        return int(sum(self.new_tokens))

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# ----------------------------------------------------------------------------
# named workloads
# ----------------------------------------------------------------------------

def tiny_decode_f32(L: int = 2048) -> Spec:
    return Spec("tiny_decode_f32", "f32", [L], [1], H_I=4, d_I=64, H=8, d=128, d_v=128, K=256)


def decode_bf16_b32(rng: np.random.Generator, B: int = 32, lo: int = 16384, hi: int = 32768) -> Spec:
    lens = [int(x) for x in rng.integers(lo, hi, size=B, endpoint=True)]
    return Spec("decode_bf16_b32", "bf16", lens, [1] * B, H_I=64, d_I=128, H=128, d=576, d_v=512, K=2048)


def decode_1m_fp8(L: int = 1 << 20) -> Spec:
    return Spec("decode_1m_fp8", "bf16_kfp8", [L], [1], H_I=64, d_I=128, H=128, d=576, d_v=512, K=2048)


def prefill_chunk(B: int = 2, new: int = 4096, total: int = 65536, mode: str = "bf16") -> Spec:
    return Spec("prefill_2x4096_64k", mode, [total] * B, [new] * B, H_I=64, d_I=128, H=128, d=576, d_v=512, K=2048)


def mixed_batch(rng: np.random.Generator, n_dec: int = 64, lo: int = 1024, hi: int = 262144,
                chunk: int = 2048, chunk_total: int = 131072) -> Spec:
    u = rng.uniform(math.log(lo), math.log(hi), size=n_dec)
    lens = [int(round(math.exp(x))) for x in u] + [chunk_total]
    return Spec("mixed_64dec_2048pre", "bf16_kfp8", lens, [1] * n_dec + [chunk],
                H_I=64, d_I=128, H=128, d=576, d_v=512, K=2048)


def named(n: int) -> tuple[Spec, int]:
    """Workload number ``n`` (1..5) and its seed."""
    rng = np.random.default_rng(1000 + n)  # lengths draw on their own stream
    if n == 1:
        return tiny_decode_f32(), 1
    if n == 2:
        return decode_bf16_b32(rng), 2
    if n == 3:
        return decode_1m_fp8(), 3
    if n == 4:
        return prefill_chunk(), 4
    if n == 5:
        return mixed_batch(rng), 5
    raise ValueError(n)


# ----------------------------------------------------------------------------
# storage rounding (input preparation only)
# ----------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """fp32 -> OCP e4m3 codes, round to nearest even, saturating at +-448."""
    x = np.clip(np.asarray(x, dtype=np.float32), -448.0, 448.0)
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def kv_record_bytes(d: int) -> int:
    """Bytes of one FP8 latent record: d e4m3 codes, one fp32 scale per 128 elements, padded to 16."""
    return (d + 4 * ((d + 127) // 128) + 15) // 16 * 16


def to_kv_fp8_records(x: np.ndarray) -> np.ndarray:
    """fp32 rows ``[..., d]`` -> FP8 latent records ``[..., kv_record_bytes(d)]`` (uint8).

    Each tile of 128 consecutive elements (the last one the remaining d mod 128) is quantised on its
    own, in fp32: ``scale = amax / 448`` (1 when amax is 0), codes ``RNE_e4m3(x / scale)``
    saturating at 448. A record holds the d codes, then the fp32 scales, then zero bytes.
    """
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    nt = (d + 127) // 128
    out = np.zeros(x.shape[:-1] + (kv_record_bytes(d),), dtype=np.uint8)
    scales = np.empty(x.shape[:-1] + (nt,), dtype=np.float32)
    for j in range(nt):
        tile = x[..., 128 * j: min(d, 128 * j + 128)]
        amax = np.abs(tile).max(axis=-1)
        sc = (amax / np.float32(448.0)).astype(np.float32)
        sc[sc == 0] = 1.0
        scales[..., j] = sc
        out[..., 128 * j: 128 * j + tile.shape[-1]] = to_e4m3_codes(tile / sc[..., None])
    out[..., d: d + 4 * nt] = scales.view(np.uint8).reshape(x.shape[:-1] + (4 * nt,))
    return out


def kv_fp8_poison(d: int) -> np.ndarray:
    """The record of an empty slot: every code 448 (0x7E), every scale 1."""
    rec = np.zeros(kv_record_bytes(d), dtype=np.uint8)
    rec[:d] = POISON_E4M3
    nt = (d + 127) // 128
    rec[d: d + 4 * nt] = np.ones(nt, np.float32).view(np.uint8)
    return rec


def to_mx_e4m3(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 ``[..., n]`` (n a multiple of 32) -> (e4m3 codes ``[..., n]``, E8M0 bytes ``[..., n/32]``).

    OCP Microscaling with E4M3 elements: each group of 32 shares the exponent
    ``X = floor(log2(amax)) - 8`` (clamped to [-127, 127]; -127 for an all-zero
    group), stored as the byte ``X + 127``; the elements are ``x * 2^-X``
    rounded to e4m3 (nearest even, saturating at 448).
    """
    x = np.asarray(x, dtype=np.float32)
    g = x.reshape(x.shape[:-1] + (-1, 32))
    amax = np.abs(g).max(axis=-1)
    _, e = np.frexp(amax)  # amax = f * 2^e with f in [0.5, 1)
    X = np.clip(np.where(amax > 0, e.astype(np.int64) - 9, -127), -127, 127)
    scaled = np.ldexp(g, (-X)[..., None]).astype(np.float32)
    return to_e4m3_codes(scaled).reshape(x.shape), (X + 127).astype(np.uint8)


# ----------------------------------------------------------------------------
# case generation
# ----------------------------------------------------------------------------

@dataclass
class Case:
    spec: Spec
    seed: int
    block_table: np.ndarray  # int32 [B][max_blocks]
    seq_lens: np.ndarray     # int32 [B]
    q_seq: np.ndarray        # int32 [T]
    q_pos: np.ndarray        # int32 [T]
    q_I: np.ndarray          # f32 [T,H_I,d_I] or u16 bf16 bits
    w: np.ndarray            # f32 [T,H_I]
    k_I: np.ndarray          # f32/u16/u8 [NB,64,d_I]
    k_I_scale: np.ndarray | None  # f32 [NB] (FP8 keys) | u8 [NB,64,d_I/32] E8M0 (MXFP8 keys)
    q: np.ndarray            # f32 [T,H,d] or u16
    kv: np.ndarray           # f32 [NB,64,d] or u16

    @property
    def num_blocks(self) -> int:
        return int(self.k_I.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def _normal(rng, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _store(x: np.ndarray, mode: str) -> np.ndarray:
    return x.astype(np.float32) if mode == "f32" else to_bf16_bits(x)


def _poison_value(mode: str):
    return np.float32(POISON) if mode == "f32" else to_bf16_bits(np.array([POISON], np.float32))[0]


def generate(spec: Spec, seed: int, chunk_blocks: int = 1024) -> Case:
    """Draw every input of ``spec`` from PCG64(seed).

    Draw order: block-table permutation, q_I, w, q, then per chunk of logical
    blocks k_I and kv (so the host never holds a full fp32 copy of the cache).
    """
    rng = np.random.default_rng(seed)
    bs = spec.block_size
    lens = np.asarray(spec.seq_lens, dtype=np.int64)
    nblk = (lens + bs - 1) // bs
    n_logical = int(nblk.sum())
    NB = n_logical + spec.spare_blocks
    max_blocks = max(1, int(nblk.max()) if len(nblk) else 1)

    perm = rng.permutation(NB).astype(np.int32)
    table = np.full((spec.B, max_blocks), -1, dtype=np.int32)
    first = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int64)
    for b in range(spec.B):
        table[b, : nblk[b]] = perm[first[b] : first[b + 1]]

    q_seq = np.concatenate([np.full(n, b, np.int32) for b, n in enumerate(spec.new_tokens)]) if spec.T else np.zeros(0, np.int32)
    q_pos = np.concatenate([np.arange(L - n, L, dtype=np.int32) for L, n in zip(spec.seq_lens, spec.new_tokens)]) if spec.T else np.zeros(0, np.int32)

    T = spec.T
    q_I = _store(_normal(rng, (T, spec.H_I, spec.d_I)), spec.mode)
    w = rng.uniform(0.0, 1.0, size=(T, spec.H_I)).astype(np.float32)
    q = _store(_normal(rng, (T, spec.H, spec.d)), spec.mode)

    fp8 = spec.mode == "bf16_kfp8"
    mx = spec.mode == "mxfp8"
    kdt = np.float32 if spec.mode == "f32" else (np.uint8 if fp8 or mx else np.uint16)
    vdt = np.float32 if spec.mode == "f32" else np.uint16
    k_I = np.empty((NB, bs, spec.d_I), dtype=kdt)
    kv_fp8 = spec.kv == "fp8"
    assert spec.kv in ("act", "fp8") and not (kv_fp8 and spec.mode == "f32")
    kv = np.empty((NB, bs, kv_record_bytes(spec.d)), dtype=np.uint8) if kv_fp8 else np.empty((NB, bs, spec.d), dtype=vdt)
    scale = np.ones(NB, dtype=np.float32) if fp8 else None
    if mx:
        scale = np.full((NB, bs, spec.d_I // 32), 127, dtype=np.uint8)

    # logical block list in (sequence, block) order -> physical slot
    phys_of_logical = perm[:n_logical]
    for c0 in range(0, n_logical, chunk_blocks):
        c1 = min(n_logical, c0 + chunk_blocks)
        dst = phys_of_logical[c0:c1]
        kx = _normal(rng, (c1 - c0, bs, spec.d_I))
        if fp8:
            amax = np.abs(kx).reshape(c1 - c0, -1).max(axis=1)
            s = (amax / np.float32(448.0)).astype(np.float32)
            s[s == 0] = 1.0
            k_I[dst] = to_e4m3_codes(kx / s[:, None, None])
            scale[dst] = s
        elif mx:
            k_I[dst], scale[dst] = to_mx_e4m3(bf16_bits_to_f32(to_bf16_bits(kx)))
        else:
            k_I[dst] = _store(kx, spec.mode)
        vx = _normal(rng, (c1 - c0, bs, spec.d))
        # FP8 latent rows: quantised from their bf16 values (what a cache append receives)
        kv[dst] = to_kv_fp8_records(bf16_bits_to_f32(to_bf16_bits(vx))) if kv_fp8 else _store(vx, spec.mode)

    # poison: spare blocks and the tail slots of each sequence's last block
    kpois = np.uint8(POISON_E4M3) if fp8 or mx else _poison_value(spec.mode)
    vpois = kv_fp8_poison(spec.d) if kv_fp8 else _poison_value(spec.mode)
    spare = perm[n_logical:]
    k_I[spare] = kpois
    kv[spare] = vpois
    if mx:
        scale[spare] = 127
    for b in range(spec.B):
        L = int(lens[b])
        if L % bs:
            pb = table[b, L // bs]
            k_I[pb, L % bs :] = kpois
            kv[pb, L % bs :] = vpois
            if mx:
                scale[pb, L % bs :] = 127

    return Case(spec, seed, table, lens.astype(np.int32), q_seq, q_pos, q_I, w, k_I, scale, q, kv)


def with_key_format(case: Case, mode: str) -> Case:
    """The same case with its bf16 indexer keys re-stored as ``"bf16_kfp8"`` (e4m3 codes with one
    fp32 scale per physical block, amax / 448 over the block's tokens) or ``"mxfp8"`` (OCP MX codes
    and E8M0 bytes per 32 elements). Slots that hold no token get the poison code; every other
    input (queries, weights, latent cache, block table) is shared with ``case``."""
    import dataclasses
    assert case.spec.mode == "bf16" and mode in ("bf16_kfp8", "mxfp8")
    bs = case.spec.block_size
    x = bf16_bits_to_f32(case.k_I)
    valid = np.zeros(x.shape[:2], dtype=bool)
    for b, L in enumerate(case.seq_lens.tolist()):
        nblk = (L + bs - 1) // bs
        blks = case.block_table[b, :nblk]
        valid[blks] = True
        if L % bs:
            valid[blks[-1], L % bs:] = False
    x[~valid] = 0.0
    if mode == "mxfp8":
        codes, scale = to_mx_e4m3(x)
        scale[~valid] = 127
    else:
        amax = np.abs(x).reshape(x.shape[0], -1).max(axis=1)
        scale = (amax / np.float32(448.0)).astype(np.float32)
        scale[scale == 0] = 1.0
        codes = to_e4m3_codes(x / scale[:, None, None])
    codes[~valid] = POISON_E4M3
    return dataclasses.replace(case, spec=dataclasses.replace(case.spec, mode=mode), k_I=codes, k_I_scale=scale)


def with_kv_format(case: Case, kv: str) -> Case:
    """The same case with its bf16 latent rows re-stored as FP8 records (``kv="fp8"``): every tile of
    128 elements of a row quantised on its own (``to_kv_fp8_records``); slots that hold no token get
    the poison record. Every other input is shared with ``case``."""
    import dataclasses
    assert case.spec.mode != "f32" and case.spec.kv == "act" and kv == "fp8"
    bs = case.spec.block_size
    recs = to_kv_fp8_records(bf16_bits_to_f32(case.kv))
    valid = np.zeros(case.kv.shape[:2], dtype=bool)
    for b, L in enumerate(case.seq_lens.tolist()):
        nblk = (L + bs - 1) // bs
        blks = case.block_table[b, :nblk]
        valid[blks] = True
        if L % bs:
            valid[blks[-1], L % bs:] = False
    recs[~valid] = kv_fp8_poison(case.spec.d)
    return dataclasses.replace(case, spec=dataclasses.replace(case.spec, kv=kv), kv=recs)


def repage(case: Case, seed: int) -> Case:
    """Same logical content under another physical block permutation."""
    rng = np.random.default_rng(seed)
    NB = case.num_blocks
    perm = rng.permutation(NB).astype(np.int32)  # old physical -> new physical
    table = case.block_table.copy()
    valid = table >= 0
    table[valid] = perm[table[valid]]
    k_I = np.empty_like(case.k_I)
    kv = np.empty_like(case.kv)
    k_I[perm] = case.k_I
    kv[perm] = case.kv
    scale = None
    if case.k_I_scale is not None:
        scale = np.empty_like(case.k_I_scale)
        scale[perm] = case.k_I_scale
    return Case(case.spec, case.seed, table, case.seq_lens.copy(), case.q_seq.copy(), case.q_pos.copy(),
                case.q_I.copy(), case.w.copy(), k_I, scale, case.q.copy(), kv)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact widening, for test-side data edits)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
