"""The C-ABI library loads and exports every entry point include/tcd.h declares
(CPU only: no call here touches the GPU)."""
import ctypes
import os
import re

from conftest import ROOT


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(tc_[a-z0-9_]+)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("tc_compile_trie", "tc_bind_grammar", "tc_step", "tc_decode"):
        assert required in names


def test_library_exports_every_declared_symbol(tcd):
    lib = ctypes.CDLL(tcd.LIB_PATH)
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(tcd):
    assert tcd.status_name(0) == "TC_OK"
    assert tcd.status_name(16) == "TC_ERR_EMPTY_MASK"
    assert tcd.status_name(999) == "TC_ERR_UNKNOWN"
