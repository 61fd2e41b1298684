"""bench.py's host helpers on the CPU: the code hash that keys captured DRAM traffic."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_text_drops_comments_and_layout_but_keeps_literals():
    a = bench.code_text('int a = 1; // one\n/* block\n comment */ float  b = "x  // y";')
    b = bench.code_text('int a = 1;\n\n   float b = "x  // y";  // other words\n')
    assert a == b
    assert '"x  // y"' in a
    assert bench.code_text("a/**/b") == "a b"  # a comment still separates tokens


def test_hash_follows_code_not_comments():
    csrc = os.path.join(ROOT, "shared_prefix_paged_attn_b300", "csrc")
    files = {f: open(os.path.join(csrc, f), encoding="utf-8").read() for f in os.listdir(csrc)}
    base = bench.kernel_source_hash(read=lambda f: files[f])
    assert base == bench.kernel_source_hash()
    name = "merge_kernel.cuh"
    commented = dict(files, **{name: "// a new comment\n" + files[name]})
    assert bench.kernel_source_hash(read=lambda f: commented[f]) == base
    changed = dict(files, **{name: files[name].replace("kThreads = 256", "kThreads = 128")})
    assert changed[name] != files[name]
    assert bench.kernel_source_hash(read=lambda f: changed[f]) != base
    # the compaction op is not part of the decode's hash
    other = dict(files, **{"compact.cu": files["compact.cu"] + "\nint x;\n"})
    assert bench.kernel_source_hash(read=lambda f: other[f]) == base
