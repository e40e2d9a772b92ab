"""The C-ABI library builds, loads and exports every entry point its header declares.

No compute call is made here: these run without a GPU.
"""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_decode.h")
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def _declared():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(mla_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared()
    for required in ["mla_decode_plan", "mla_decode", "mla_decode_workspace_size",
                     "mla_decode_check", "mla_status_string", "mla_prolog"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    import mla_decode_attention_02_gb300 as m
    lib = m.load_library()
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", m.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mla_[a-z_]+)\b", out))
    assert set(_declared()) <= exported


def test_status_strings():
    import mla_decode_attention_02_gb300 as m
    lib = m.load_library()
    for s in range(7):
        assert lib.mla_status_string(s)
    assert lib.mla_status_string(99) == b"unknown status"


@pytest.mark.parametrize("header", HEADERS, ids=os.path.basename)
def test_header_compiles_as_c(header):
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c",
                         "-I", os.path.dirname(header), header], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr


def test_missing_library_fails_loudly(tmp_path):
    import mla_decode_attention_02_gb300._binding as b
    saved = b._lib
    try:
        b._lib = None
        with pytest.raises(RuntimeError, match="no fallback"):
            b.load_library(str(tmp_path / "nope.so"))
    finally:
        b._lib = saved
