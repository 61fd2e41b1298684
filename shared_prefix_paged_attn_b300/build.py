"""Builds ``libforkattn.so`` (the C-ABI library) in-tree with nvcc for sm_103a."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libforkattn.so")
# the same sources with device bounds checks on every page id and row record from the plan
LIB_CHECKED = os.path.join(HERE, "libforkattn_checked.so")
SOURCES = ["plan.cpp", "decode.cu", "compact.cu", "score.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _newest_source_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(os.path.dirname(HERE), "include", "fork_attn.h"))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    out = LIB_CHECKED if checked else LIB
    if not force and os.path.exists(out) and os.path.getmtime(out) >= _newest_source_mtime():
        return out
    cmd = ["nvcc", *ARCH, "-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-Wall", "-o", out]
    if checked:
        cmd.append("-DFORK_ATTN_CHECKED")
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, checked="--checked" in sys.argv))
