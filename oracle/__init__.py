"""fp64 CPU oracle for weight-absorbed MLA decode (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding in ``mla_decode_attention_02_gb300``) never does, and shares no
code with it: the arithmetic lives in ``mla_oracle.c``, compiled here with the
host C compiler.

What the oracle computes is stated in the header of ``mla_oracle.c``, with
its sources: "Huawei Ascend servers: DeepSeek V3/R1 inference best practice"
sections 3.2.1 (heads share one compressed cache; decode absorbs the weights),
6.1 (FlashAttention-style exact attention) and 7.2 (the 576/512/128 cost
formula), and the FlashDecoding split described in the Atlas 800I A3
TPOT-jitter troubleshooting post.

Pins (tests that tie it to something other than itself) live in
``tests/test_oracle_pins.py``: the unabsorbed multi-head form, a dense fp64
library softmax on tiny inputs, closed forms, and invariants.

``oracle.prolog`` (numpy, fp64) holds the step before attention: the
absorbed query projection, RoPE, RMSNorm of the new latent and the append
into the paged cache; its pins are in ``tests/test_prolog_pins.py``.
``oracle.epilog`` (numpy, fp64) holds the step after it: the value
up-projection W_UV per head, the output projection W_O, and the same layer
written as plain (unabsorbed) multi-head attention; pins in
``tests/test_epilog_pins.py``.
``oracle.fp8`` holds the e4m3 latent cache format (per-token fp32 scale):
the quantiser, deciding codes in fp32 as the GPU does, and the
dequantisation; pins in ``tests/test_fp8_pins.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmla_oracle.so")

ELEM_BF16 = 0
ELEM_F64 = 1

_ERRORS = {
    1: "invalid argument",
    2: "seq_len smaller than the number of query tokens",
    3: "block_table entry outside the page pool",
    4: "key range outside the visible keys",
    5: "out of memory",
}

_lock = threading.Lock()
_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("s_q", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("d_latent", ctypes.c_int32),
        ("d_rope", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("elem", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("q_latent", ctypes.c_void_p),
        ("q_rope", ctypes.c_void_p),
        ("kv_cache", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile ``mla_oracle.c`` into ``_build/libmla_oracle.so`` (host C compiler)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cc = os.environ.get("CC", "gcc")
    # -ffp-contract=off keeps every product and sum a separately rounded fp64 op.
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.mla_oracle_rows.restype = ctypes.c_int
            lib.mla_oracle_rows.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int64,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int32]
            lib.mla_oracle_merge.restype = ctypes.c_int
            lib.mla_oracle_merge.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _as_np(x, dtype):
    """numpy view of a CPU array/tensor; bf16 tensors become uint16 bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16).numpy().view(np.uint16)
            else:
                x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=dtype)


def decode(q_latent, q_rope, kv_cache, block_table, seq_lens, *, s_q: int, scale: float,
           rows=None, ranges=None, threads: int | None = None):
    """fp64 MLA decode rows.

    q_latent [B][s_q][H][512], q_rope [B][s_q][H][64], kv_cache [P][page][576]:
    either bf16 (torch bf16 tensors or uint16 bit patterns) or float64.
    block_table [B][max_pages] int32, seq_lens [B] int32.

    rows: None for every (b, t, h) in that order, else an (n, 3) int array.
    ranges: None for each row's full visible key range, else an (n, 2) int array
    of [j0, j1) key ranges.  Returns (o [n][512] float64, lse [n] float64); with
    rows=None, o is shaped [B][s_q][H][512] and lse [B][s_q][H].
    """
    lib = _load()
    qd = getattr(q_latent, "dtype", None)
    is_f64 = str(qd) in ("float64", "torch.float64")
    elem = ELEM_F64 if is_f64 else ELEM_BF16
    dt = np.float64 if is_f64 else np.uint16
    ql = _as_np(q_latent, dt)
    qr = _as_np(q_rope, dt)
    kv = _as_np(kv_cache, dt)
    bt = _as_np(block_table, np.int32)
    sl = _as_np(seq_lens, np.int32)
    if ql.ndim != 4 or qr.ndim != 4 or kv.ndim != 3 or bt.ndim != 2 or sl.ndim != 1:
        raise ValueError("oracle: bad input ranks")
    B, S, H, DL = ql.shape
    DR = qr.shape[3]
    if S != s_q or kv.shape[2] != DL + DR or bt.shape[0] != B or sl.shape[0] != B:
        raise ValueError("oracle: inconsistent shapes")
    prob = _Problem(B, s_q, H, DL, DR, kv.shape[1], bt.shape[1], elem, kv.shape[0], float(scale),
                    ql.ctypes.data, qr.ctypes.data, kv.ctypes.data, bt.ctypes.data,
                    sl.ctypes.data)
    if rows is None:
        n = B * S * H
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
        n = rows_arr.shape[0]
    rng_arr = None
    if ranges is not None:
        rng_arr = np.ascontiguousarray(ranges, dtype=np.int64).reshape(-1, 2)
        if rng_arr.shape[0] != n:
            raise ValueError("oracle: ranges must match rows")
    o = np.empty((n, DL), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = lib.mla_oracle_rows(ctypes.byref(prob), n,
                             None if rows_arr is None else rows_arr.ctypes.data,
                             None if rng_arr is None else rng_arr.ctypes.data,
                             o.ctypes.data, lse.ctypes.data,
                             threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")
    if rows is None:
        return o.reshape(B, S, H, DL), lse.reshape(B, S, H)
    return o, lse


def merge(o_parts, lse_parts):
    """LSE merge of partial results over disjoint key ranges.

    o_parts [n][d] float64, lse_parts [n] float64 -> (o [d], lse).
    """
    lib = _load()
    op = np.ascontiguousarray(o_parts, dtype=np.float64)
    lp = np.ascontiguousarray(lse_parts, dtype=np.float64).reshape(-1)
    n, d = op.shape
    if lp.shape[0] != n:
        raise ValueError("oracle: merge shapes")
    o = np.empty((d,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    rc = lib.mla_oracle_merge(n, d, op.ctypes.data, lp.ctypes.data, o.ctypes.data,
                              lse.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")
    return o, float(lse[0])
