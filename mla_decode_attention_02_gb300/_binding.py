"""ctypes binding over libmla_decode.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this
module checks tensor shapes, dtypes and devices, allocates the caller-owned
workspace and outputs with PyTorch, and passes raw pointers and the current
CUDA stream through the C ABI declared in include/mla_decode.h.  There is
no CPU path: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np

NUM_HEADS = 128
D_LATENT = 512
D_ROPE = 64
PAGE_SIZE = 64
DEFAULT_SCALE = 192.0 ** -0.5

MLA_DEV_BAD_PAGE = 0x1
MLA_DEV_BAD_SEQ_LEN = 0x2
MLA_DEV_BAD_PLAN = 0x4
MLA_DEV_TIMEOUT = 0x8

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_decode.so")

_lock = threading.Lock()
_lib = None


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_string(status)} (status {status})")


class _Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("s_q", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("flags", ctypes.c_int32)]


_P = ctypes.POINTER(_Problem)
_vp = ctypes.c_void_p
_SIGS = {
    "mla_decode_workspace_size": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_size_t)]),
    "mla_decode_num_units": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32)]),
    "mla_decode_plan": (ctypes.c_int, [_P, _vp, _vp, ctypes.c_size_t, _vp]),
    "mla_decode": (ctypes.c_int, [_P, _vp, _vp, _vp, ctypes.c_int64, _vp, ctypes.c_float, _vp,
                                  _vp, _vp, ctypes.c_size_t, _vp]),
    "mla_decode_timed": (ctypes.c_int, [_P, _vp, _vp, _vp, ctypes.c_int64, _vp, ctypes.c_float,
                                        _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]),
    "mla_decode_diag": (ctypes.c_int, [_P, _vp, _vp, _vp, ctypes.c_int64, _vp, ctypes.c_float,
                                       _vp, _vp, _vp, ctypes.c_size_t, _vp, ctypes.c_uint64,
                                       ctypes.c_uint32]),
    "mla_decode_fp8": (ctypes.c_int, [_P, _vp, _vp, _vp, ctypes.c_int64, _vp, ctypes.c_float, _vp,
                                      _vp, _vp, ctypes.c_size_t, _vp, _vp]),
    "mla_decode_noalloc": (ctypes.c_int, [_P, _vp, _vp, _vp, ctypes.c_int64, _vp, _vp,
                                          ctypes.c_float, _vp, _vp, _vp]),
    "mla_decode_check": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int32), _vp]),
    "mla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mla_decode_plan_bytes": (ctypes.c_size_t, [_P, ctypes.c_int32]),
    "mla_decode_plan_host": (ctypes.c_int, [_P, _vp, ctypes.c_int32, _vp, ctypes.c_size_t]),
    "mla_prolog": (ctypes.c_int, [_P, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp,
                                  _vp, ctypes.c_int64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mla_prolog_rope_table": (ctypes.c_int, [ctypes.c_double, _vp, _vp]),
    "mla_epilog_uv": (ctypes.c_int, [_P, _vp, _vp, _vp, _vp, _vp]),
    "mla_cache_quantize_fp8": (ctypes.c_int, [_vp, ctypes.c_int64, _vp, _vp]),
    "mla_epilog_oproj": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp]),
}


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libmla_decode.so (built by ``__graft_entry__.build()`` or ``build.py``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build the CUDA library first "
                    "(python -m mla_decode_attention_02_gb300.build); there is no fallback path")
            lib = ctypes.CDLL(p)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _status_string(status: int) -> str:
    try:
        return load_library().mla_status_string(status).decode()
    except Exception:  # pragma: no cover - library not loadable
        return "unknown"


def _check(status: int, what: str) -> None:
    if status != 0:
        raise MLAError(status, what)


MLA_FLAG_POW2_MAX = 0x1


def _problem(batch: int, s_q: int, max_pages: int, flags: int = 0) -> _Problem:
    return _Problem(int(batch), int(s_q), NUM_HEADS, PAGE_SIZE, int(max_pages), int(flags))


def num_units() -> int:
    """Work units (SM groups) the main kernel uses on the current device."""
    u = ctypes.c_int32(0)
    _check(load_library().mla_decode_num_units(ctypes.byref(u)), "mla_decode_num_units")
    return u.value


def workspace_size(batch: int, s_q: int, max_pages: int) -> int:
    n = ctypes.c_size_t(0)
    prob = _problem(batch, s_q, max_pages)
    _check(load_library().mla_decode_workspace_size(ctypes.byref(prob), ctypes.byref(n)),
           "mla_decode_workspace_size")
    return n.value


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _req(t, name, dtype, shape, device):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device.type != "cuda" or (device is not None and t.device != device):
        raise ValueError(f"{name} must be on {device or 'a CUDA device'}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.data_ptr() % 16:
        raise ValueError(f"{name} must be 16-byte aligned")


@dataclass
class Plan:
    """A split-KV schedule in a device workspace (valid for one seq_lens)."""
    batch: int
    s_q: int
    max_pages: int
    workspace: object   # torch.uint8 CUDA tensor, owned by this Plan
    seq_lens: object    # the device seq_lens it was built from

    def problem(self, flags: int = 0) -> _Problem:
        return _problem(self.batch, self.s_q, self.max_pages, flags)


def plan(seq_lens, *, s_q: int, max_pages_per_seq: int, workspace=None, stream=None) -> Plan:
    """Build the split-KV schedule on the device (``mla_decode_plan``)."""
    import torch
    _req(seq_lens, "seq_lens", torch.int32, None, None)
    if seq_lens.dim() != 1:
        raise ValueError("seq_lens must be 1-D [batch]")
    batch = seq_lens.shape[0]
    with torch.cuda.device(seq_lens.device):
        need = workspace_size(batch, s_q, max_pages_per_seq)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=seq_lens.device)
        _req(workspace, "workspace", torch.uint8, None, seq_lens.device)
        prob = _problem(batch, s_q, max_pages_per_seq)
        _check(load_library().mla_decode_plan(ctypes.byref(prob), seq_lens.data_ptr(),
                                              workspace.data_ptr(), workspace.numel(),
                                              _stream_handle(stream)), "mla_decode_plan")
    return Plan(batch, s_q, max_pages_per_seq, workspace, seq_lens)


def decode(p: Plan, q_latent, q_rope, kv_cache, block_table, *, scale: float = DEFAULT_SCALE,
           out=None, lse=None, stream=None, events=None, pow2_max: bool = False):
    """Weight-absorbed MLA decode (``mla_decode``) -> (o_latent bf16, lse fp32).

    events: optional three torch.cuda.Event(enable_timing=True) recorded before the
    main kernel, between the main kernel and the merge, and after the merge
    (``mla_decode_timed``).  pow2_max: power-of-two running maxima
    (MLA_FLAG_POW2_MAX), so that every rescale is by an exact power of two.
    """
    return _decode(p, q_latent, q_rope, kv_cache, block_table, scale, out, lse, stream, events, None,
                   MLA_FLAG_POW2_MAX if pow2_max else 0)


def decode_fp8(p: Plan, q_latent, q_rope, kv_cache_fp8, block_table, *, scale: float = DEFAULT_SCALE,
               out=None, lse=None, stream=None, events=None, pow2_max: bool = False):
    """``mla_decode_fp8``: decode over an fp8 cache (uint8 [num_pages][64][656]) -> (o bf16, lse fp32).

    events and pow2_max as in ``decode``.
    """
    return _decode(p, q_latent, q_rope, kv_cache_fp8, block_table, scale, out, lse, stream, events, None,
                   MLA_FLAG_POW2_MAX if pow2_max else 0, fp8=True)


MLA_INJECT_WITHHOLD_K_LOAD = 0x1


def decode_diag(p: Plan, q_latent, q_rope, kv_cache, block_table, *, wait_limit_ns: int,
                inject: int = 0, scale: float = DEFAULT_SCALE, out=None, lse=None, stream=None):
    """``mla_decode_diag``: decode with a chosen wait limit and an optional injected stall.

    With inject=MLA_INJECT_WITHHOLD_K_LOAD one K-stage load of the unit that runs the
    schedule's first item is never issued, so the kernel's bounded waits run out: check(p) then reports
    MLA_DEV_TIMEOUT and the rows of that unit are unspecified.
    """
    return _decode(p, q_latent, q_rope, kv_cache, block_table, scale, out, lse, stream, None,
                   (int(wait_limit_ns), int(inject)), 0)


def _decode(p, q_latent, q_rope, kv_cache, block_table, scale, out, lse, stream, events, diag, flags,
            fp8=False):
    import torch
    dev = p.workspace.device
    B, S = p.batch, p.s_q
    _req(q_latent, "q_latent", torch.bfloat16, (B, S, NUM_HEADS, D_LATENT), dev)
    _req(q_rope, "q_rope", torch.bfloat16, (B, S, NUM_HEADS, D_ROPE), dev)
    if fp8:
        _req(kv_cache, "kv_cache_fp8", torch.uint8, None, dev)
        if kv_cache.dim() != 3 or tuple(kv_cache.shape[1:]) != (PAGE_SIZE, FP8_ROW_BYTES):
            raise ValueError("kv_cache_fp8 must be [num_pages][64][656] bytes")
    else:
        _req(kv_cache, "kv_cache", torch.bfloat16, None, dev)
        if kv_cache.dim() != 3 or tuple(kv_cache.shape[1:]) != (PAGE_SIZE, D_LATENT + D_ROPE):
            raise ValueError("kv_cache must be [num_pages][64][576]")
    _req(block_table, "block_table", torch.int32, (B, p.max_pages), dev)
    if out is None:
        out = torch.empty((B, S, NUM_HEADS, D_LATENT), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, S, NUM_HEADS), dtype=torch.float32, device=dev)
    _req(out, "out", torch.bfloat16, (B, S, NUM_HEADS, D_LATENT), dev)
    _req(lse, "lse", torch.float32, (B, S, NUM_HEADS), dev)
    prob = p.problem(flags)
    args = [ctypes.byref(prob), q_latent.data_ptr(), q_rope.data_ptr(), kv_cache.data_ptr(),
            kv_cache.shape[0], block_table.data_ptr(), float(scale), out.data_ptr(),
            lse.data_ptr(), p.workspace.data_ptr(), p.workspace.numel(), _stream_handle(stream)]
    handles = None
    if events is not None:
        if len(events) != 3:
            raise ValueError("events must hold three torch.cuda.Event")
        handles = (ctypes.c_void_p * 3)(*[ctypes.c_void_p(e.cuda_event) if e is not None
                                          else None for e in events])
    with torch.cuda.device(dev):
        if fp8:
            _check(load_library().mla_decode_fp8(*args, handles), "mla_decode_fp8")
        elif diag is not None:
            _check(load_library().mla_decode_diag(*args, *diag), "mla_decode_diag")
        elif handles is None:
            _check(load_library().mla_decode(*args), "mla_decode")
        else:
            _check(load_library().mla_decode_timed(*args, handles), "mla_decode_timed")
    return out, lse


NOALLOC_SCRATCH_BYTES = 64 << 20


def decode_noalloc(q_latent, q_rope, kv_cache, block_table, seq_lens, *, s_q: int,
                   scale: float = DEFAULT_SCALE, out=None, lse=None, stream=None):
    """Plan + decode through ``mla_decode_noalloc``: the library allocates nothing.

    For callers that cannot allocate device memory on their decode path; the
    workspace lives in a fixed 64 MiB device array inside the library, shared
    by every call (order calls on one stream).  Problems needing a larger
    workspace raise MLAError (status 3).  out / lse may be passed in so that
    this call allocates nothing on the Python side either.
    """
    import torch
    _req(seq_lens, "seq_lens", torch.int32, None, None)
    dev = seq_lens.device
    B = seq_lens.shape[0]
    _req(q_latent, "q_latent", torch.bfloat16, (B, s_q, NUM_HEADS, D_LATENT), dev)
    _req(q_rope, "q_rope", torch.bfloat16, (B, s_q, NUM_HEADS, D_ROPE), dev)
    _req(kv_cache, "kv_cache", torch.bfloat16, None, dev)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch][max_pages_per_seq]")
    _req(block_table, "block_table", torch.int32, None, dev)
    if out is None:
        out = torch.empty((B, s_q, NUM_HEADS, D_LATENT), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, s_q, NUM_HEADS), dtype=torch.float32, device=dev)
    _req(out, "out", torch.bfloat16, (B, s_q, NUM_HEADS, D_LATENT), dev)
    _req(lse, "lse", torch.float32, (B, s_q, NUM_HEADS), dev)
    prob = _problem(B, s_q, block_table.shape[1])
    with torch.cuda.device(dev):
        _check(load_library().mla_decode_noalloc(
            ctypes.byref(prob), q_latent.data_ptr(), q_rope.data_ptr(), kv_cache.data_ptr(),
            kv_cache.shape[0], block_table.data_ptr(), seq_lens.data_ptr(), float(scale),
            out.data_ptr(), lse.data_ptr(), _stream_handle(stream)), "mla_decode_noalloc")
    return out, lse


D_NOPE = 128
DEFAULT_ROPE_BASE = 10000.0
DEFAULT_RMS_EPS = 1e-6


ROPE_TABLE_FLOATS = 64
_rope_tables = {}


def rope_table(rope_base: float = DEFAULT_ROPE_BASE, device=None, stream=None):
    """The rotary table of ``mla_prolog_rope_table`` (float32 [64] on the device), built on the GPU."""
    import torch
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        table = torch.empty(ROPE_TABLE_FLOATS, dtype=torch.float32, device=dev)
        _check(load_library().mla_prolog_rope_table(float(rope_base), table.data_ptr(),
                                                    _stream_handle(stream)), "mla_prolog_rope_table")
    return table


def prolog(q_nope, q_pe, kv_latent, k_pe, w_uk, kv_norm_weight, kv_cache, block_table, seq_lens, *,
           rope_base: float = DEFAULT_ROPE_BASE, rms_eps: float = DEFAULT_RMS_EPS, table=None,
           q_latent=None, q_rope=None, status=None, stream=None):
    """The MLA prolog slice (``mla_prolog``): absorbed query, RoPE, cache append.

    Shapes: q_nope [B][s_q][128][128], q_pe [B][s_q][128][64], kv_latent [B][s_q][512],
    k_pe [B][s_q][64], w_uk [128][128][512], kv_norm_weight [512] (all bf16);
    kv_cache [pages][64][576] bf16 is updated in place; block_table [B][max_pages]
    and seq_lens [B] int32.  table: a rope_table() tensor; without one, the table of
    rope_base is built once per device and kept.  Returns (q_latent, q_rope, status):
    status is a one-element int32 device tensor of MLA_DEV_* bits (zeroed here, on the
    stream, unless the caller passes its own).
    """
    import torch
    if q_nope.dim() != 4:
        raise ValueError("q_nope must be [batch][s_q][heads][128]")
    B, S = q_nope.shape[0], q_nope.shape[1]
    dev = q_nope.device
    _req(q_nope, "q_nope", torch.bfloat16, (B, S, NUM_HEADS, D_NOPE), dev)
    _req(q_pe, "q_pe", torch.bfloat16, (B, S, NUM_HEADS, D_ROPE), dev)
    _req(kv_latent, "kv_latent", torch.bfloat16, (B, S, D_LATENT), dev)
    _req(k_pe, "k_pe", torch.bfloat16, (B, S, D_ROPE), dev)
    _req(w_uk, "w_uk", torch.bfloat16, (NUM_HEADS, D_NOPE, D_LATENT), dev)
    _req(kv_norm_weight, "kv_norm_weight", torch.bfloat16, (D_LATENT,), dev)
    _req(kv_cache, "kv_cache", torch.bfloat16, None, dev)
    if kv_cache.dim() != 3 or tuple(kv_cache.shape[1:]) != (PAGE_SIZE, D_LATENT + D_ROPE):
        raise ValueError("kv_cache must be [num_pages][64][576]")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch][max_pages_per_seq]")
    _req(block_table, "block_table", torch.int32, None, dev)
    _req(seq_lens, "seq_lens", torch.int32, (B,), dev)
    if q_latent is None:
        q_latent = torch.empty((B, S, NUM_HEADS, D_LATENT), dtype=torch.bfloat16, device=dev)
    if q_rope is None:
        q_rope = torch.empty((B, S, NUM_HEADS, D_ROPE), dtype=torch.bfloat16, device=dev)
    _req(q_latent, "q_latent", torch.bfloat16, (B, S, NUM_HEADS, D_LATENT), dev)
    _req(q_rope, "q_rope", torch.bfloat16, (B, S, NUM_HEADS, D_ROPE), dev)
    with torch.cuda.device(dev):
        if table is None:
            key = (dev.index, float(rope_base))
            table = _rope_tables.get(key)
            if table is None:
                # the kept table must hold its values for every later call on any stream
                if torch.cuda.is_current_stream_capturing():
                    raise RuntimeError("prolog: build the rotary table with rope_table() before "
                                       "capturing a CUDA graph, and pass it as table=")
                table = rope_table(rope_base, dev, stream)
                (stream if stream is not None else torch.cuda.current_stream()).synchronize()
                _rope_tables[key] = table
        _req(table, "table", torch.float32, (ROPE_TABLE_FLOATS,), dev)
        if status is None:
            status = torch.zeros(1, dtype=torch.int32, device=dev)
        _req(status, "status", torch.int32, (1,), dev)
        prob = _problem(B, S, block_table.shape[1])
        _check(load_library().mla_prolog(
            ctypes.byref(prob), q_nope.data_ptr(), q_pe.data_ptr(), kv_latent.data_ptr(),
            k_pe.data_ptr(), w_uk.data_ptr(), kv_norm_weight.data_ptr(), float(rms_eps),
            table.data_ptr(), kv_cache.data_ptr(), kv_cache.shape[0], block_table.data_ptr(),
            seq_lens.data_ptr(), q_latent.data_ptr(), q_rope.data_ptr(), status.data_ptr(),
            _stream_handle(stream)), "mla_prolog")
    return q_latent, q_rope, status


D_V = 128
HIDDEN = 7168


def epilog_uv(o_latent, w_uv, *, o_v=None, status=None, stream=None):
    """The value up-projection (``mla_epilog_uv``): o_v[t][h] = W_UV[h] . o_latent[t][h].

    o_latent [B][s_q][128][512] and w_uv [128][128][512] bf16 -> (o_v [B][s_q][128][128] bf16,
    status: one-element int32 device tensor of MLA_DEV_* bits).
    """
    import torch
    if o_latent.dim() != 4:
        raise ValueError("o_latent must be [batch][s_q][heads][512]")
    B, S = o_latent.shape[0], o_latent.shape[1]
    dev = o_latent.device
    _req(o_latent, "o_latent", torch.bfloat16, (B, S, NUM_HEADS, D_LATENT), dev)
    _req(w_uv, "w_uv", torch.bfloat16, (NUM_HEADS, D_V, D_LATENT), dev)
    if o_v is None:
        o_v = torch.empty((B, S, NUM_HEADS, D_V), dtype=torch.bfloat16, device=dev)
    _req(o_v, "o_v", torch.bfloat16, (B, S, NUM_HEADS, D_V), dev)
    with torch.cuda.device(dev):
        if status is None:
            status = torch.zeros(1, dtype=torch.int32, device=dev)
        _req(status, "status", torch.int32, (1,), dev)
        prob = _problem(B, S, 1)
        _check(load_library().mla_epilog_uv(ctypes.byref(prob), o_latent.data_ptr(), w_uv.data_ptr(),
                                            o_v.data_ptr(), status.data_ptr(), _stream_handle(stream)),
               "mla_epilog_uv")
    return o_v, status


def epilog_oproj(o_v, w_o, *, out=None, status=None, stream=None):
    """The output projection (``mla_epilog_oproj``, a tensor-core kernel): out = o_v . W_O^T.

    o_v [..][128][128] bf16 viewed as [tokens][16384], w_o [hidden][16384] bf16 ->
    out [tokens][hidden] bf16.  status: optional int32 device tensor of one element that
    the call ORs MLA_DEV_TIMEOUT into if a bounded wait in the kernel runs out.
    """
    import torch
    dev = o_v.device
    tokens = o_v.numel() // (NUM_HEADS * D_V)
    if tokens * NUM_HEADS * D_V != o_v.numel() or tokens < 1:
        raise ValueError("o_v must hold whole [128][128] token rows")
    _req(o_v, "o_v", torch.bfloat16, None, dev)
    if w_o.dim() != 2 or w_o.shape[1] != NUM_HEADS * D_V:
        raise ValueError("w_o must be [hidden][16384]")
    _req(w_o, "w_o", torch.bfloat16, None, dev)
    hidden = w_o.shape[0]
    if out is None:
        out = torch.empty((tokens, hidden), dtype=torch.bfloat16, device=dev)
    _req(out, "out", torch.bfloat16, (tokens, hidden), dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    _req(status, "status", torch.int32, None, dev)
    with torch.cuda.device(dev):
        _check(load_library().mla_epilog_oproj(int(tokens), int(hidden), o_v.data_ptr(), w_o.data_ptr(),
                                               out.data_ptr(), status.data_ptr(), _stream_handle(stream)),
               "mla_epilog_oproj")
    return out


FP8_ROW_BYTES = 656


def quantize_cache_fp8(kv_cache, *, out=None, stream=None):
    """The fp8 (e4m3) cache of a bf16 cache (``mla_cache_quantize_fp8``).

    kv_cache [..][576] bf16 -> uint8 [..][656]: per row the 512 e4m3 codes of c_kv / s,
    k_rope / s (bf16), s (fp32), zero padding.
    """
    import torch
    if kv_cache.shape[-1] != D_LATENT + D_ROPE:
        raise ValueError("kv_cache rows must hold 576 values")
    _req(kv_cache, "kv_cache", torch.bfloat16, None, None)
    dev = kv_cache.device
    shape = tuple(kv_cache.shape[:-1]) + (FP8_ROW_BYTES,)
    if out is None:
        out = torch.empty(shape, dtype=torch.uint8, device=dev)
    _req(out, "out", torch.uint8, shape, dev)
    rows = kv_cache.numel() // (D_LATENT + D_ROPE)
    with torch.cuda.device(dev):
        _check(load_library().mla_cache_quantize_fp8(kv_cache.data_ptr(), int(rows), out.data_ptr(),
                                                     _stream_handle(stream)), "mla_cache_quantize_fp8")
    return out


def check(p: Plan, stream=None) -> int:
    """Synchronise and return the device status bits (0 = no input error seen)."""
    import torch
    v = ctypes.c_int32(0)
    with torch.cuda.device(p.workspace.device):
        rc = load_library().mla_decode_check(p.workspace.data_ptr(), ctypes.byref(v),
                                             _stream_handle(stream))
    if rc not in (0, 5, 6):
        _check(rc, "mla_decode_check")
    return v.value


# ----------------------------------------------------------------------------- host planner

def _align(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def plan_layout(batch: int, s_q: int, units: int) -> dict:
    """Byte offsets of the schedule regions (mirrors plan_layout in csrc/mla_internal.h)."""
    rows = batch * s_q
    max_items = rows + units
    off = 64
    L = {"num_rows": rows, "max_items": max_items, "items": off}
    off += 16 * max_items
    L["item_unit"] = off
    off += 4 * max_items
    L["unit_begin"] = off
    off += 4 * (units + 1)
    L["row_nparts"] = off
    off += 4 * rows
    L["row_part0"] = off
    off += 4 * rows
    L["row_item0"] = off
    off += 4 * rows
    off = _align(off, 8)
    L["row_pos"] = off
    off += 8 * rows
    L["plan_end"] = off
    return L


_HDR = np.dtype([("magic", "<u4"), ("batch", "<i4"), ("s_q", "<i4"), ("max_pages", "<i4"),
                 ("num_units", "<i4"), ("num_rows", "<i4"), ("max_items", "<i4"),
                 ("num_items", "<i4"), ("num_parts", "<i4"), ("status", "<i4"),
                 ("split", "<i4"), ("min_split", "<i4"), ("total_cost", "<i8"),
                 ("target", "<i8")])


def parse_plan(buf, batch: int, s_q: int, units: int) -> dict:
    """Decode schedule bytes (host copy of a workspace prefix) into numpy arrays."""
    b = np.frombuffer(bytes(buf), dtype=np.uint8)
    L = plan_layout(batch, s_q, units)
    hdr = b[:64].view(_HDR)[0]
    n = int(hdr["num_items"])
    R = L["num_rows"]
    items = b[L["items"]:L["items"] + 16 * n].view("<i4").reshape(n, 4)
    return {
        "header": {k: int(hdr[k]) for k in _HDR.names},
        "items": items.copy(),   # columns: row, kv_begin, kv_end, part
        "item_unit": b[L["item_unit"]:L["item_unit"] + 4 * n].view("<i4").copy(),
        "unit_begin": b[L["unit_begin"]:L["unit_begin"] + 4 * (units + 1)].view("<i4").copy(),
        "row_nparts": b[L["row_nparts"]:L["row_nparts"] + 4 * R].view("<i4").copy(),
        "row_part0": b[L["row_part0"]:L["row_part0"] + 4 * R].view("<i4").copy(),
        "row_item0": b[L["row_item0"]:L["row_item0"] + 4 * R].view("<i4").copy(),
        "row_pos": b[L["row_pos"]:L["row_pos"] + 8 * R].view("<i8").copy(),
    }


def plan_host(seq_lens, *, s_q: int, max_pages_per_seq: int, num_units: int) -> dict:
    """Run the planner's algorithm on the CPU (``mla_decode_plan_host``) and parse it."""
    lib = load_library()
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    prob = _problem(sl.shape[0], s_q, max_pages_per_seq)
    nbytes = lib.mla_decode_plan_bytes(ctypes.byref(prob), int(num_units))
    if nbytes == 0:  # invalid problem: let the planner entry point name the reason
        _check(lib.mla_decode_plan_host(ctypes.byref(prob), sl.ctypes.data, int(num_units),
                                        None, 0), "mla_decode_plan_host")
        raise MLAError(1, "mla_decode_plan_bytes")
    buf = np.zeros(nbytes, dtype=np.uint8)
    _check(lib.mla_decode_plan_host(ctypes.byref(prob), sl.ctypes.data, int(num_units),
                                    buf.ctypes.data, nbytes), "mla_decode_plan_host")
    return parse_plan(buf.tobytes(), sl.shape[0], s_q, num_units)


def plan_device_bytes(p: Plan) -> bytes:
    """Host copy of a device schedule (for tests)."""
    L = plan_layout(p.batch, p.s_q, num_units())
    return p.workspace[:L["plan_end"]].cpu().numpy().tobytes()
