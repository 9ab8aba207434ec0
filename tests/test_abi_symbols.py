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


def _header_constants():
    """#define and enum constants of include/tcd.h (comments removed)."""
    text = open(os.path.join(ROOT, "include", "tcd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    consts = {n: int(v, 0) for n, v in re.findall(r"#define\s+(TC_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)\b", text)}
    for body in re.findall(r"enum[^{]*\{(.*?)\}", text, flags=re.S):
        for n, v in re.findall(r"\b(TC_[A-Z0-9_]+)\s*=\s*(0x[0-9a-fA-F]+|\d+)", body):
            consts[n] = int(v, 0)
    return consts


def test_binding_constants_match_the_header(tcd):
    """The binding's heads, flags, residencies and status codes are the
    header's values (the binding only marshals; a drifted constant would make
    it ask for another head or flag than it names)."""
    h = _header_constants()
    pairs = {"HEAD_SPARSE": "TC_HEAD_SPARSE", "HEAD_DENSE": "TC_HEAD_DENSE",
             "HEAD_UNION_GEMM": "TC_HEAD_UNION_GEMM", "HEAD_DENSE_GEMM": "TC_HEAD_DENSE_GEMM",
             "FLAG_JUMP_FORWARD": "TC_FLAG_JUMP_FORWARD", "FLAG_FORCED_LOGITS": "TC_FLAG_FORCED_LOGITS",
             "FLAG_ROOT_GEMM": "TC_FLAG_ROOT_GEMM", "BIND_LIVE_COUNTS": "TC_BIND_LIVE_COUNTS",
             "RES_AUTO": "TC_RES_AUTO", "RES_CONST": "TC_RES_CONST", "RES_GLOBAL": "TC_RES_GLOBAL",
             "TC_ERR_EMPTY_MASK": "TC_ERR_EMPTY_MASK", "TC_ERR_NO_LIVE_EDGE": "TC_ERR_NO_LIVE_EDGE",
             "TC_ERR_MAX_STEPS": "TC_ERR_MAX_STEPS", "TC_ERR_BOUNDS": "TC_ERR_BOUNDS"}
    for py, c in pairs.items():
        assert c in h, c
        assert getattr(tcd, py) == h[c], (py, getattr(tcd, py), h[c])
    # the flags are distinct bits, clear of the head values
    flags = [h["TC_FLAG_JUMP_FORWARD"], h["TC_FLAG_FORCED_LOGITS"], h["TC_FLAG_ROOT_GEMM"]]
    assert len(set(flags)) == 3 and all(f & (f - 1) == 0 and f > 3 for f in flags)
