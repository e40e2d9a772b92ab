"""Seeded synthetic inputs for MLA decode (shared by the tests, the smoke check and the bench).

This module only draws random inputs and lays them out; it holds none of the
attention arithmetic, so the CUDA path and the fp64 oracle can both consume
what it produces without sharing any of the method.

Shapes (row-major):
    q_latent    [B][s_q][128][512] bf16 ~ N(0, 1)
    q_rope      [B][s_q][128][64]  bf16 ~ N(0, 1)
    kv_cache    [P][64][576]       bf16 ~ N(0, 1)   (row = c_kv[0:512] || k_rope[512:576])
    block_table [B][max_pages]     int32, a seeded random permutation of the page pool, -1 padded
    seq_lens    [B]                int32

The page pool holds exactly sum_b ceil(L_b / 64) pages (plus ``extra_pages``
unused pages when asked).  With ``poison=True`` every cache slot past a
request's length in its last page, and every unused page, holds NaN, so any
read of a masked key shows up in the result.

Workloads (the pages' decode shapes; see the design notes for the citations):
    tiny      B=4,   s_q=1, seq_lens {1, 63, 64, 200} shuffled
    uniform   B=64,  s_q=1, all 4096
    mtp       B=128, s_q=2, seq_lens uniform in [1024, 8192]
    mixed     B=64,  s_q=1, 26 x 20480 + 38 x 400 interleaved at random
    long      B=4,   s_q=1, 4 x 262144
    long1m    B=1,   s_q=1, 1 x 1048576

Prolog inputs (the step before attention, ``prolog_tensors``):
    q_nope [B][s_q][128][128], q_pe [B][s_q][128][64], kv_latent [B][s_q][512],
    k_pe [B][s_q][64] bf16 ~ N(0, 1); w_uk [128][128][512] bf16 ~ N(0, 1/128)
    (random weights, unit-variance outputs); kv_norm_weight [512] bf16 ~ 1 + N(0, 0.1^2).
``sparse_cache`` builds a pool and block table for the append alone: the
slots of the step's new tokens get distinct pages, every other table entry a
random page (so positions up to millions need no million-token pool).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

NUM_HEADS = 128
D_LATENT = 512
D_ROPE = 64
D_ROW = D_LATENT + D_ROPE
D_NOPE = 128
D_V = 128
HIDDEN = 7168
PAGE = 64
SCALE = 192.0 ** -0.5
ROPE_BASE = 10000.0      # DeepSeek V3/R1 rotary base
RMS_EPS = 1e-6           # DeepSeek V3/R1 RMSNorm epsilon


@dataclass
class Workload:
    name: str
    seed: int
    batch: int
    s_q: int
    seq_lens: list = field(default_factory=list)


def _seq_lens(name: str, gen: torch.Generator) -> tuple[int, int, list]:
    if name == "tiny":
        lens = [1, 63, 64, 200]
        perm = torch.randperm(4, generator=gen).tolist()
        return 4, 1, [lens[i] for i in perm]
    if name == "uniform":
        return 64, 1, [4096] * 64
    if name == "mtp":
        lens = torch.randint(1024, 8193, (128,), generator=gen).tolist()
        return 128, 2, lens
    if name == "mixed":
        lens = [20480] * 26 + [400] * 38
        perm = torch.randperm(64, generator=gen).tolist()
        return 64, 1, [lens[i] for i in perm]
    if name == "long":
        return 4, 1, [262144] * 4
    if name == "long1m":
        return 1, 1, [1048576]
    raise KeyError(name)


SEEDS = {"tiny": 1, "uniform": 2, "mtp": 3, "mixed": 4, "long": 5, "long1m": 6}


def workload(name: str) -> Workload:
    gen = torch.Generator().manual_seed(SEEDS[name])
    b, s, lens = _seq_lens(name, gen)
    return Workload(name, SEEDS[name], b, s, lens)


def custom(seq_lens, s_q: int = 1, seed: int = 0, name: str = "custom") -> Workload:
    return Workload(name, seed, len(seq_lens), s_q, list(int(x) for x in seq_lens))


def _randn_bf16(shape, gen: torch.Generator, chunk: int = 1 << 26, std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) fp32 draws rounded to bf16 (round to nearest even), drawn in chunks."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16)
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        out[i:i + m] = (torch.randn(m, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)
    return out.view(*shape)


def make_inputs(w: Workload, *, poison: bool = False, extra_pages: int = 0,
                max_pages: int | None = None) -> dict:
    """All inputs of one decode step, on the CPU.

    The draw order is fixed: block-table permutation, then q_latent, q_rope,
    kv_cache.  A fresh generator seeded with ``w.seed + 1000`` drives it, so the
    seq_lens draw in ``workload()`` does not shift the tensors.
    """
    gen = torch.Generator().manual_seed(w.seed + 1000)
    pages_per = [(L + PAGE - 1) // PAGE for L in w.seq_lens]
    used = sum(pages_per)
    pool = used + extra_pages
    mp = max(pages_per) if max_pages is None else max_pages
    if mp < max(pages_per):
        raise ValueError("max_pages smaller than the longest request")
    perm = torch.randperm(pool, generator=gen).to(torch.int32)
    block_table = torch.full((w.batch, mp), -1, dtype=torch.int32)
    k = 0
    for b, n in enumerate(pages_per):
        block_table[b, :n] = perm[k:k + n]
        k += n
    q_latent = _randn_bf16((w.batch, w.s_q, NUM_HEADS, D_LATENT), gen)
    q_rope = _randn_bf16((w.batch, w.s_q, NUM_HEADS, D_ROPE), gen)
    kv_cache = _randn_bf16((pool, PAGE, D_ROW), gen)
    if poison:
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
        referenced = torch.zeros(pool, dtype=torch.bool)
        for b, n in enumerate(pages_per):
            pages = block_table[b, :n].long()
            referenced[pages] = True
            tail = w.seq_lens[b] - (n - 1) * PAGE
            if tail < PAGE:
                kv_cache[pages[-1], tail:, :] = nan
        kv_cache[~referenced] = nan
    return {
        "q_latent": q_latent,
        "q_rope": q_rope,
        "kv_cache": kv_cache,
        "block_table": block_table,
        "seq_lens": torch.tensor(w.seq_lens, dtype=torch.int32),
        "s_q": w.s_q,
        "scale": SCALE,
    }


def cache_bytes(seq_lens) -> int:
    """Algorithmic cache bytes one decode step must read: every key row once."""
    return sum(int(L) for L in seq_lens) * D_ROW * 2


FP8_ROW_BYTES = 656   # an fp8 cache row: 512 e4m3 codes, 64 bf16 k_rope / s, fp32 s, padding


def cache_bytes_fp8(seq_lens) -> int:
    """Algorithmic bytes of the same step over the fp8 cache: every 656-byte row once."""
    return sum(int(L) for L in seq_lens) * FP8_ROW_BYTES


def flops(seq_lens, s_q: int) -> int:
    """Tensor FLOPs of one step: 2 * heads * (576 + 512) per (query token, visible key)."""
    per_key = 2 * NUM_HEADS * (D_ROW + D_LATENT)
    return sum(per_key * (int(L) - s_q + 1 + t) for L in seq_lens for t in range(s_q))


def prolog_tensors(batch: int, s_q: int, seed: int) -> dict:
    """Raw per-token inputs and weights of one prolog step (bf16, CPU)."""
    gen = torch.Generator().manual_seed(seed + 2000)
    return {
        "q_nope": _randn_bf16((batch, s_q, NUM_HEADS, D_NOPE), gen),
        "q_pe": _randn_bf16((batch, s_q, NUM_HEADS, D_ROPE), gen),
        "kv_latent": _randn_bf16((batch, s_q, D_LATENT), gen),
        "k_pe": _randn_bf16((batch, s_q, D_ROPE), gen),
        "w_uk": _randn_bf16((NUM_HEADS, D_NOPE, D_LATENT), gen, std=D_NOPE ** -0.5),
        "kv_norm_weight": (1.0 + 0.1 * torch.randn(D_LATENT, generator=gen)).to(torch.bfloat16),
    }


def sparse_cache(seq_lens, s_q: int, seed: int, extra_pages: int = 4) -> dict:
    """Cache pool, block table and seq_lens for an append-only step (see the module notes)."""
    gen = torch.Generator().manual_seed(seed + 3000)
    B = len(seq_lens)
    max_pages = max(1, max((int(L) + PAGE - 1) // PAGE for L in seq_lens))
    slots = sorted({(b, (int(L) - s_q + t) // PAGE) for b, L in enumerate(seq_lens)
                    for t in range(s_q) if int(L) - s_q + t >= 0})
    pool = len(slots) + extra_pages
    block_table = torch.randint(0, pool, (B, max_pages), generator=gen, dtype=torch.int32)
    perm = torch.randperm(pool, generator=gen).to(torch.int32)
    for k, (b, j) in enumerate(slots):
        block_table[b, j] = perm[k]
    return {
        "kv_cache": _randn_bf16((pool, PAGE, D_ROW), gen),
        "block_table": block_table,
        "seq_lens": torch.tensor([int(L) for L in seq_lens], dtype=torch.int32),
    }


def prolog_bytes(batch: int, s_q: int) -> int:
    """Algorithmic HBM bytes of one prolog launch: every input read once, every output written once."""
    T = batch * s_q
    reads = 2 * (T * NUM_HEADS * (D_NOPE + D_ROPE) + NUM_HEADS * D_NOPE * D_LATENT
                 + T * (D_LATENT + D_ROPE) + D_LATENT) + 4 * (batch + T)   # + seq_lens, table entries
    writes = 2 * (T * NUM_HEADS * (D_LATENT + D_ROPE) + T * D_ROW)
    return reads + writes


def prolog_flops(batch: int, s_q: int) -> int:
    """Tensor FLOPs of the absorbed-q contraction: 2 x tokens x heads x 128 x 512."""
    return 2 * batch * s_q * NUM_HEADS * D_NOPE * D_LATENT


def epilog_tensors(tokens: int, seed: int, hidden: int = HIDDEN) -> dict:
    """Inputs and random weights of the step after attention (bf16, CPU): o_latent ~ N(0, 1),
    W_UV ~ N(0, 1/512), W_O ~ N(0, 1/16384), so every projection keeps unit variance."""
    gen = torch.Generator().manual_seed(seed + 4000)
    return {
        "o_latent": _randn_bf16((tokens, NUM_HEADS, D_LATENT), gen),
        "w_uv": _randn_bf16((NUM_HEADS, D_V, D_LATENT), gen, std=D_LATENT ** -0.5),
        "w_o": _randn_bf16((hidden, NUM_HEADS * D_V), gen, std=(NUM_HEADS * D_V) ** -0.5),
    }


def epilog_bytes(tokens: int, hidden: int = HIDDEN) -> tuple:
    """Algorithmic HBM bytes of (the W_UV step, o_proj): every input read once, output written once."""
    uv = 2 * (tokens * NUM_HEADS * (D_LATENT + D_V) + NUM_HEADS * D_V * D_LATENT)
    op = 2 * (tokens * NUM_HEADS * D_V + hidden * NUM_HEADS * D_V + tokens * hidden)
    return uv, op
