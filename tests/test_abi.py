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
