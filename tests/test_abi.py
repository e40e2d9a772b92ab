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


def _prob(batch=2, s_q=1, heads=128, page=64, max_pages=4, flags=0):
    import mla_decode_attention_02_gb300._binding as b
    return b._Problem(batch, s_q, heads, page, max_pages, flags)


def test_prolog_and_epilog_reject_bad_arguments_before_any_cuda_call():
    """Host-side validation of the prolog and epilog entry points (no GPU needed: each call
    fails on its arguments and returns before touching CUDA)."""
    import ctypes
    import mla_decode_attention_02_gb300 as m
    lib = m.load_library()
    A = 0x10000                      # a 16-byte aligned address that is never dereferenced
    ok = [A] * 6
    good = _prob()

    def prolog(prob, ptrs=ok, eps=1e-6, table=A, num_pages=8, status=A):
        return lib.mla_prolog(ctypes.byref(prob) if prob is not None else None, *ptrs, eps, table, A,
                              num_pages, A, A, A, A, status, None)
    assert prolog(None) == 1
    assert prolog(_prob(s_q=3)) == 2
    assert prolog(_prob(heads=64)) == 2
    assert prolog(_prob(page=32)) == 2
    assert prolog(_prob(batch=0)) == 1
    assert prolog(_prob(flags=1)) == 1                                    # decode-only flag
    assert prolog(_prob(batch=1, max_pages=1 << 25)) == 2                 # positions past 2^31
    assert prolog(good, ptrs=[A, A + 8, A, A, A, A]) == 1          # q_pe not 16-byte aligned
    assert prolog(good, eps=-1.0) == 1
    assert prolog(good, eps=float("nan")) == 1
    assert prolog(good, table=None) == 1
    assert prolog(good, num_pages=0) == 1
    assert prolog(good, status=None) == 1
    assert lib.mla_prolog_rope_table(-1.0, A, None) == 1
    assert lib.mla_prolog_rope_table(float("inf"), A, None) == 1
    assert lib.mla_prolog_rope_table(10000.0, None, None) == 1

    assert lib.mla_epilog_uv(None, A, A, A, A, None) == 1
    assert lib.mla_epilog_uv(ctypes.byref(_prob(s_q=3)), A, A, A, A, None) == 2
    assert lib.mla_epilog_uv(ctypes.byref(_prob(flags=1)), A, A, A, A, None) == 1
    assert lib.mla_epilog_uv(ctypes.byref(good), A, A, None, A, None) == 1
    assert lib.mla_epilog_uv(ctypes.byref(good), A, A, A, None, None) == 1
    assert lib.mla_epilog_oproj(0, 7168, A, A, A, A, None) == 1
    assert lib.mla_epilog_oproj(4, 7, A, A, A, A, None) == 1
    assert lib.mla_epilog_oproj(4, 7168, A + 2, A, A, A, None) == 1
    assert lib.mla_epilog_oproj(4, 7168, A, A, A, None, None) == 1         # no status word
    assert lib.mla_epilog_oproj(4, 7168, A, A, A, A + 2, None) == 1        # misaligned status word
    assert lib.mla_cache_quantize_fp8(None, 64, A, None) == 1
    assert lib.mla_cache_quantize_fp8(A, 0, A, None) == 1
    assert lib.mla_cache_quantize_fp8(A, 64, A + 4, None) == 1


def test_decode_entry_points_reject_bad_arguments_before_any_cuda_call():
    """mla_decode_plan, mla_decode, mla_decode_timed, mla_decode_diag, mla_decode_fp8 and
    mla_decode_noalloc refuse null or unaligned pointers, an empty page pool, a non-positive or non-finite scale
    and a workspace below the size any device could need (mla_decode_diag also a wait limit
    outside [1 us, 60 s] and unknown injection bits), before they make a CUDA call (so these
    run without a GPU; a call that passed validation would stop at the first CUDA call
    instead)."""
    import mla_decode_attention_02_gb300 as m
    lib = m.load_library()
    A = 0x10000
    good = _prob()
    big = 1 << 30                       # plenty of workspace bytes

    def plan(prob=good, seq=A, ws=A, nbytes=big):
        return lib.mla_decode_plan(ctypes.byref(prob) if prob is not None else None, seq, ws, nbytes, None)

    def decode(prob=good, ptrs=(A, A, A), num_pages=8, bt=A, scale=0.072, out=(A, A), ws=A,
               nbytes=big, timed="plain", limit=10**6, inject=0):
        args = [ctypes.byref(prob) if prob is not None else None, *ptrs, num_pages, bt, scale, *out, ws,
                nbytes, None]
        if timed == "diag":
            return lib.mla_decode_diag(*args, limit, inject)
        if timed == "fp8":
            return lib.mla_decode_fp8(*args, None)
        return lib.mla_decode_timed(*args, None) if timed == "timed" else lib.mla_decode(*args)

    def noalloc(prob=good, ptrs=(A, A, A), num_pages=8, bt=A, seq=A, scale=0.072, out=(A, A)):
        return lib.mla_decode_noalloc(ctypes.byref(prob) if prob is not None else None, *ptrs,
                                      num_pages, bt, seq, scale, *out, None)

    assert plan(prob=None) == 1
    assert plan(prob=_prob(s_q=3)) == 2
    assert plan(prob=_prob(flags=2)) == 1                                 # unknown flag bit
    assert plan(prob=_prob(flags=1), nbytes=64) == 3                      # the known one passes on
    assert plan(seq=None) == 1
    assert plan(seq=A + 4) == 1
    assert plan(ws=None) == 1
    assert plan(ws=A + 8) == 1
    assert plan(nbytes=64) == 3
    for timed in ("plain", "timed", "diag", "fp8"):
        assert decode(prob=None, timed=timed) == 1
        assert decode(prob=_prob(heads=64), timed=timed) == 2
        assert decode(ptrs=(None, A, A), timed=timed) == 1
        assert decode(ptrs=(A, A + 2, A), timed=timed) == 1
        assert decode(ptrs=(A, A, None), timed=timed) == 1
        assert decode(bt=None, timed=timed) == 1
        assert decode(out=(A, None), timed=timed) == 1
        assert decode(out=(A + 8, A), timed=timed) == 1
        assert decode(ws=None, timed=timed) == 1
        assert decode(num_pages=0, timed=timed) == 1
        assert decode(num_pages=-5, timed=timed) == 1
        assert decode(num_pages=1 << 31, timed=timed) == 1
        for bad in (0.0, -0.072, float("nan"), float("inf"), float("-inf")):
            assert decode(scale=bad, timed=timed) == 1, bad
        assert decode(prob=_prob(flags=-1), timed=timed) == 1
        assert decode(prob=_prob(flags=1), nbytes=1024, timed=timed) == 3
        assert decode(nbytes=1024, timed=timed) == 3
    # the diagnostic entry point also bounds its wait limit and knows one injection bit
    for limit in (0, 999, 60 * 10**9 + 1, 2**64 - 1):
        assert decode(timed="diag", limit=limit) == 1, limit
    for inject in (2, 0x80000000, 0xFFFFFFFF):
        assert decode(timed="diag", inject=inject) == 1, inject
    assert noalloc(prob=None) == 1
    assert noalloc(seq=None) == 1
    assert noalloc(seq=A + 4) == 1
    assert noalloc(out=(A, None)) == 1
    assert noalloc(ptrs=(A, A, None)) == 1
    assert noalloc(num_pages=0) == 1
    assert noalloc(scale=-1.0) == 1
    assert noalloc(scale=float("nan")) == 1
