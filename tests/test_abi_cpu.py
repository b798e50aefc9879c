"""The C-ABI library builds for sm_103a, loads, exports every symbol include/dsa.h declares, and
rejects bad arguments on the host before any launch (no GPU needed: nothing here computes)."""
import ctypes
import os
import re

import pytest

import indexer_top_sparse_paged_gb300 as dsa
from indexer_top_sparse_paged_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def L():
    build_library()
    return dsa.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("dsa_indexer_topk", "dsa_sparse_attn", "dsa_decode", "dsa_workspace_size", "dsa_read_error",
              "dsa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_symbols():
        assert hasattr(L, n), f"{n} declared in dsa.h but not exported"


def test_status_strings_and_version(L):
    for code in range(8):
        assert L.dsa_status_string(code)
    assert L.dsa_version() >= 100
    assert L.dsa_last_launch_count() == 0


def _dims(**kw):
    d = dict(mode="bf16", B=2, max_blocks=4, num_blocks=8, H_I=64, d_I=128, H=128, d=576, d_v=512, K=256)
    d.update(kw)
    return dsa.make_dims(**d)


def test_workspace_size_rejects_bad_dims(L):
    assert L.dsa_workspace_size(None, 2) == 0
    assert L.dsa_workspace_size(ctypes.byref(_dims(block_size=32)), 2) == 0
    assert L.dsa_workspace_size(ctypes.byref(_dims(K=0)), 2) == 0
    assert L.dsa_workspace_size(ctypes.byref(_dims(K=4096)), 2) == 0
    assert L.dsa_workspace_size(ctypes.byref(_dims()), 2) > 0


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation first


def test_indexer_rejects_null_and_unsupported(L):
    d = _dims()
    args = [FAKE] * 8
    # null q_I
    st = L.dsa_indexer_topk(ctypes.byref(d), None, *args[1:8], 2, FAKE, FAKE, 1 << 30, None)
    assert st == 1
    # unsupported block size and K
    for bad in (_dims(block_size=16), _dims(K=3000), _dims(mode=7)):
        assert L.dsa_indexer_topk(ctypes.byref(bad), *args, 2, FAKE, FAKE, 1 << 30, None) == 2
    # unsupported small shape (d_I not a multiple of 8 in bf16)
    assert L.dsa_indexer_topk(ctypes.byref(_dims(H_I=4, d_I=12)), *args, 2, FAKE, FAKE, 1 << 30, None) == 2
    # FP8 keys need their scales
    st = L.dsa_indexer_topk(ctypes.byref(_dims(mode="bf16_kfp8")), FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE,
                            2, FAKE, FAKE, 1 << 30, None)
    assert st == 1
    # T != B without q_seq
    assert L.dsa_indexer_topk(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 3, FAKE, FAKE,
                              1 << 30, None) == 1
    # misaligned pointer
    assert L.dsa_indexer_topk(ctypes.byref(d), ctypes.c_void_p((1 << 20) + 4), *args[1:8], 2, FAKE, FAKE, 1 << 30,
                              None) == 1
    # missing / misaligned / small workspace
    assert L.dsa_indexer_topk(ctypes.byref(d), *args, 2, FAKE, None, 1 << 30, None) == 3
    assert L.dsa_indexer_topk(ctypes.byref(d), *args, 2, FAKE, ctypes.c_void_p((1 << 20) + 16), 1 << 30, None) == 3
    assert L.dsa_indexer_topk(ctypes.byref(d), *args, 2, FAKE, FAKE, 100, None) == 3


def test_attention_and_decode_reject_bad_args(L):
    d = _dims()
    st = L.dsa_sparse_attn(ctypes.byref(d), None, FAKE, FAKE, FAKE, FAKE, FAKE, 2, ctypes.c_float(0.04), FAKE, None,
                           FAKE, 1 << 30, None)
    assert st == 1
    assert L.dsa_sparse_attn(ctypes.byref(_dims(d_v=600)), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2,
                             ctypes.c_float(0.04), FAKE, None, FAKE, 1 << 30, None) == 1
    st = L.dsa_decode(ctypes.byref(d), FAKE, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, ctypes.c_float(0.04), None,
                      FAKE, None, FAKE, 1 << 30, None)
    assert st == 1
    assert L.dsa_read_error(None, None, None) == 3
    assert L.dsa_workspace_init(None, 256, None) == 3


def test_noalloc_rejects_before_any_device_work(L):
    d = _dims()
    # null input, misaligned fault word
    assert L.dsa_indexer_topk_noalloc(ctypes.byref(d), None, FAKE, FAKE, None, FAKE, FAKE, None, None, 2, FAKE,
                                      None, None) == 1
    assert L.dsa_indexer_topk_noalloc(ctypes.byref(d), FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None, 2, FAKE,
                                      ctypes.c_void_p((1 << 20) + 2), None) == 1
    # more rows than the static scratch holds (K = 2048: (G + T) * 16 KiB > 16 MiB)
    big = _dims(B=4096, K=2048)
    assert L.dsa_workspace_size(ctypes.byref(big), 4096) > 16 << 20
    assert L.dsa_indexer_topk_noalloc(ctypes.byref(big), FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None, 4096, FAKE,
                                      None, None) == 7


def test_mxfp8_argument_checks(L):
    args = [FAKE] * 8
    mx = _dims(mode="mxfp8")
    # MXFP8 keys need their E8M0 scales, 16-byte aligned (they are fetched with bulk copies)
    for bad_scale in (None, ctypes.c_void_p((1 << 20) + 4)):
        st = L.dsa_indexer_topk(ctypes.byref(mx), FAKE, FAKE, FAKE, bad_scale, FAKE, FAKE, FAKE, FAKE, 2, FAKE, FAKE,
                                1 << 30, None)
        assert st == 1
    # groups of 32: d_I must be a multiple of 32 (CUDA-core shapes)
    small = _dims(mode="mxfp8", H_I=8, d_I=48)
    assert L.dsa_indexer_topk(ctypes.byref(small), *args, 2, FAKE, FAKE, 1 << 30, None) == 2
    st = L.dsa_cache_append(ctypes.byref(small), FAKE, FAKE, FAKE, FAKE, None, None, 2, FAKE, FAKE, FAKE, FAKE, 1 << 30,
                            None)
    assert st == 2
    # the workspace holds the quantised query: T x H_I x d_I bf16 more than for bf16 keys
    T = 2
    extra = L.dsa_workspace_size(ctypes.byref(mx), T) - L.dsa_workspace_size(ctypes.byref(_dims()), T)
    assert extra >= T * 64 * 128 * 2


def test_header_is_plain_c(tmp_path):
    """include/dsa.h is a C header (no C++ or CUDA types in the signatures): a C11 translation unit
    that includes it and takes every entry point's address compiles."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_dsa.c"
    names = declared_symbols()
    src.write_text('#include "dsa.h"\nvoid* entry_points[] = {' + ", ".join(f"(void*)&{n}" for n in names) + "};\n")
    subprocess.check_call([cc, "-std=c11", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.dirname(HEADER), str(src)])


def test_calls_with_no_rows_launch_nothing(L):
    """T = 0 is a valid call: arguments are checked, nothing is launched (no device needed)."""
    d = _dims()
    st = L.dsa_indexer_topk(ctypes.byref(d), FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, 1 << 30,
                            None)
    assert st == 0 and L.dsa_last_launch_count() == 0
    st = L.dsa_sparse_attn(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, ctypes.c_float(0.04), FAKE, None,
                           FAKE, 1 << 30, None)
    assert st == 0 and L.dsa_last_launch_count() == 0
    # the entry point without a workspace: no kernel, and its static scratch is not touched
    st = L.dsa_indexer_topk_noalloc(ctypes.byref(d), FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 0, FAKE, None,
                                    None)
    assert st == 0 and L.dsa_last_launch_count() == 0


def _noalloc_prefix_bytes(T: int, K: int, G: int, mx: bool = False, H_I: int = 64, d_I: int = 128) -> int:
    """Bytes of scratch the indexer path uses for T rows: the workspace regions before the
    indices (error word, work plan, merge counters, candidate counts and lists, the MX query)."""
    a256 = lambda x: (x + 255) // 256 * 256
    off = 256
    off = a256(off + 4 * (T + 1))                    # tile prefix
    off = a256(off + 4 * (T + 1))                    # merge-group prefix
    off = a256(off + 4 * 3 * (T + (G + 7) // 8 + 1))  # merge-tree counters
    off = a256(off + 4 * (G + T))                    # candidate counts
    off = a256(off + 8 * (G + T) * K)                # candidate lists
    off = a256(off + 8 * (G + T))                    # the sample estimate of each list
    if mx:
        off = a256(off + 2 * T * H_I * d_I)          # the MX-quantised query (bf16)
    return off


def _noalloc_rows_limit(K: int, G: int, mx: bool = False) -> int:
    T = 0
    while _noalloc_prefix_bytes(T + 1, K, G, mx) <= 16 << 20:
        T += 1
    return T


def test_noalloc_row_limit_is_the_documented_one(L):
    """The largest call dsa_indexer_topk_noalloc accepts follows from its scratch layout, and the
    header states that number for K = 2048 on 152 SMs. The library is probed with null buffers:
    a call over the limit is rejected as too large before its pointers are looked at, one within
    the limit as an invalid argument -- neither launches anything."""
    import torch
    G = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    for mode, K in (("bf16", 2048), ("bf16", 512), ("mxfp8", 2048)):
        t_max = _noalloc_rows_limit(K, G, mode == "mxfp8")
        for T, want in ((t_max, 1), (t_max + 1, 7)):
            d = _dims(mode=mode, B=T, K=K)
            st = L.dsa_indexer_topk_noalloc(ctypes.byref(d), None, None, None, None, None, None, None, None, T, None,
                                            None, None)
            assert st == want, (mode, K, T, st)
    documented = re.search(r"K = 2048: T <= (\d+)[\s*]+rows", open(HEADER).read())
    assert documented and int(documented.group(1)) == _noalloc_rows_limit(2048, 152)


def test_fp8_latent_flag_checks(L):
    """DSA_KV_FP8 goes with the bf16 modes and rows of a multiple of 16 elements; the workspace does
    not depend on it; other bits of the mode are rejected."""
    fp8 = _dims(mode="bf16", kv="fp8")
    assert fp8.mode == 1 | 0x10
    assert L.dsa_workspace_size(ctypes.byref(fp8), 2) == L.dsa_workspace_size(ctypes.byref(_dims()), 2)
    assert L.dsa_workspace_size(ctypes.byref(_dims(mode="f32", H_I=4, d_I=64, H=8, d=128, d_v=128, kv="fp8")), 2) == 0
    assert L.dsa_workspace_size(ctypes.byref(_dims(d=584, kv="fp8")), 2) == 0          # 584 % 16 != 0
    bad = _dims()
    bad.mode = 1 | 0x20
    assert L.dsa_workspace_size(ctypes.byref(bad), 2) == 0
    st = L.dsa_sparse_attn(ctypes.byref(_dims(mode="f32", H_I=4, d_I=64, H=8, d=128, d_v=128, kv="fp8")), FAKE, FAKE,
                           FAKE, FAKE, FAKE, FAKE, 2, ctypes.c_float(0.04), FAKE, None, FAKE, 1 << 30, None)
    assert st == 2
    assert dsa.kv_record_bytes(576) == 608 and dsa.kv_record_bytes(128) == 144 and dsa.kv_record_bytes(80) == 96


def test_binding_refuses_host_and_strided_tensors(L):
    """The binding hands raw device pointers to the library: a host tensor or a strided view is
    refused in Python, before anything reaches the library or a GPU."""
    import torch
    d = _dims(B=1, K=64)
    T = 1
    ws = torch.zeros(1024, dtype=torch.uint8)
    q_I = torch.zeros((T, 64, 128), dtype=torch.bfloat16)
    w = torch.zeros((T, 64), dtype=torch.float32)
    k_I = torch.zeros((8, 64, 128), dtype=torch.bfloat16)
    bt = torch.zeros((1, 4), dtype=torch.int32)
    sl = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.indexer_topk(d, q_I, w, k_I, None, bt, sl, ws=ws)
    with pytest.raises(ValueError, match="contiguous"):
        dsa.indexer_topk(d, q_I.transpose(1, 2), w, k_I, None, bt, sl, ws=ws)
    q = torch.zeros((T, 128, 576), dtype=torch.bfloat16)
    kv = torch.zeros((8, 64, 576), dtype=torch.bfloat16)
    idx = torch.zeros((T, 64), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.sparse_attn(d, q, kv, bt, sl, idx, 0.04, ws=ws)
    with pytest.raises(ValueError, match="contiguous"):
        dsa.decode(d, q_I[:, ::2], w, k_I, None, bt, sl, q, kv, 0.04, ws=ws)
    assert L.dsa_last_launch_count() == 0
