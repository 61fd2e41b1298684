"""The C-ABI library loads without a GPU and exports every function include/*.h declares."""
import ctypes
import glob
import os
import re

import pytest

from shared_prefix_paged_attn_b300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fork_attn_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(_lib.LIB_PATH)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fork_attn_plan_create", "fork_attn_decode", "fork_attn_plan_upload",
                 "fork_attn_strerror"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_strerror_names_every_status(lib):
    _lib.load()
    for code in range(0, -11, -1):
        s = _lib.load().fork_attn_strerror(code).decode()
        assert s and s != "unknown status"
    assert _lib.load().fork_attn_strerror(-999).decode() == "unknown status"


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(_lib, "_LIB", None)
    with pytest.raises(ImportError):
        _lib.load()


def test_checked_build_exports_the_same_symbols():
    # the library with device bounds checks is the same C ABI
    import ctypes
    from shared_prefix_paged_attn_b300 import _lib, build
    path = build.build(checked=True)
    lib = ctypes.CDLL(path)
    for name in _lib.SIGNATURES:
        assert hasattr(lib, name), name


def test_merge_parts_and_scoring_refuse_bad_arguments_before_any_launch():
    import ctypes
    from shared_prefix_paged_attn_b300 import _lib
    import shared_prefix_paged_attn_b300 as fa
    from shared_prefix_paged_attn_b300 import workloads as W
    lib = _lib.load()
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    assert lib.fork_attn_merge_parts(None, p, 1, 4, p, fa.FA_F32, p, None) == -1
    assert lib.fork_attn_merge_parts(p, p, 0, 4, p, fa.FA_F32, p, None) == -2
    assert lib.fork_attn_merge_parts(p, p, 1, -1, p, fa.FA_F32, p, None) == -2
    assert lib.fork_attn_merge_parts(p, p, 1, 4, p, 7, p, None) == -2
    assert lib.fork_attn_merge_parts(ctypes.c_void_p((1 << 20) + 4), p, 1, 4, p, fa.FA_F32, p, None) == -5
    assert lib.fork_attn_merge_parts(p, p, 1, 0, p, fa.FA_F32, p, None) == 0  # nothing to do
    # scoring calls want a representatives plan, uploaded
    w = W.make(1, values=False)
    plan = fa.plan_for(w)
    assert lib.fork_attn_score(p, p, plan.handle, p, p, None) == -2
    assert lib.fork_attn_score_lse(p, p, plan.handle, p, None) == -2
    assert lib.fork_attn_topk(plan.handle, p, p, p, None) == -2
    reps = fa.plan_for(W.with_representatives(W.make(1), reps=4), representatives=1)
    assert lib.fork_attn_score(p, p, reps.handle, p, p, None) == -6
    assert lib.fork_attn_score_lse(p, p, reps.handle, p, None) == -6
    assert lib.fork_attn_topk(reps.handle, p, p, p, None) == -6
    assert lib.fork_attn_score(None, p, reps.handle, p, p, None) == -1
