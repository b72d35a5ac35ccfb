"""The C-ABI library loads on a machine without a GPU and exports every entry
point that include/fs.h declares (no compute calls)."""
import os
import re

import pytest

from continuous_transformer_decode_gb300 import build, fs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(fs_\w+)\s*\(", src))
    return names


def test_library_builds_and_loads():
    build.build()
    assert fs.lib() is not None


def test_every_declared_symbol_is_exported():
    build.build()
    L = fs.lib()
    declared = _declared()
    assert "fs_decode_step_batch" in declared and "fs_create" in declared
    for name in sorted(declared):
        assert hasattr(L, name), name
    missing = declared - set(fs.exported_symbols())
    assert not missing, missing


def test_errors_without_gpu_are_reported_not_raised():
    # a NULL descriptor is refused before any CUDA call
    import ctypes as C
    h = C.c_void_p()
    rc = fs.lib().fs_create(None, None, C.byref(h))
    assert rc == fs.CODES["FS_ERR_ARG"]
    assert fs.fs_last_error(None)
