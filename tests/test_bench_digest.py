"""The source digest that ties the committed ncu traffic figure to the measured indexer code:
comment and layout edits leave it unchanged, any code edit changes it, and a profile summary
whose digest does not match is not used."""
import os
import shutil

import bench

SRC = os.path.join(bench.ROOT, "indexer_top_sparse_paged_gb300", "csrc")


def test_code_only_removes_comments_and_keeps_literals():
    src = ('int a = 1;  // one\n'
           '/* block\n   comment */ int b = 2;\n'
           '\n'
           'const char* s = "not // a comment /* either */";\n'
           "char c = '/';  char q = '\\'';\n"
           'const char* e = "quote \\" // still a string";\n')
    out = bench.code_only(src)
    assert "one" not in out and "block" not in out
    assert "int a = 1;" in out and "int b = 2;" in out
    assert '"not // a comment /* either */"' in out
    assert "'/'" in out and "'\\''" in out
    assert '"quote \\" // still a string"' in out
    assert "\n\n" not in out


def _tree(tmp_path, edit=None):
    """A copy of the measured sources under tmp_path (one file optionally edited); returns its root."""
    root = tmp_path / "root"
    csrc = root / "indexer_top_sparse_paged_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.TRAFFIC_SOURCES:
        shutil.copy(os.path.join(SRC, f), csrc / f)
    if edit:
        f, old, new = edit
        text = (csrc / f).read_text()
        assert old in text
        (csrc / f).write_text(text.replace(old, new, 1))
    return str(root)


def test_digest_ignores_comments_but_not_code(tmp_path, monkeypatch):
    base = bench.kernel_digest()
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "a"))
    assert bench.kernel_digest() == base
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "b", ("indexer_tc.cu", "namespace tcidx {",
                                                               "namespace tcidx {  // a new remark\n\n")))
    assert bench.kernel_digest() == base
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "c", ("topk_merge.cu", "#include", "#include <cstdint>\n#include")))
    assert bench.kernel_digest() != base


def test_stale_profile_gives_no_traffic(tmp_path, monkeypatch):
    prof = tmp_path / "p.md"
    prof.write_text("- kernel_source_digest: %s\n- dram_bytes_per_full_launch: 123\n" % bench.kernel_digest())
    monkeypatch.setattr(bench, "PROFILE", str(prof))
    assert bench.profiled_traffic() == 123
    prof.write_text("- kernel_source_digest: 0000000000000000\n- dram_bytes_per_full_launch: 123\n")
    assert bench.profiled_traffic() is None
