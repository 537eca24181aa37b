"""bench.py's record of profiled DRAM traffic is keyed on the expert kernel's
sources with comments and blank lines removed: comment edits keep the record,
code edits drop it."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_kernel_source_hash_ignores_comments(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    srcs = []
    for path in bench.KERNEL_SRC:
        dst = tmp_path / os.path.basename(path)
        shutil.copy(path, dst)
        srcs.append(str(dst))
    monkeypatch.setattr(bench, "KERNEL_SRC", srcs)
    h0 = bench.kernel_source_hash()
    with open(srcs[0], "a") as f:
        f.write("\n// a comment\n/* a block\n   comment */\n\n")
    assert bench.kernel_source_hash() == h0
    with open(srcs[0], "a") as f:
        f.write("static const int kUnusedForTheTest = 1;\n")
    assert bench.kernel_source_hash() != h0
