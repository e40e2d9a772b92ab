"""fp64 oracle for the MLA prolog slice that feeds the decode path (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs
may import this module; the CUDA library never does.

What it computes (the prolog fused ahead of attention):

* "Huawei Ascend servers: DeepSeek V3/R1 inference best practice", section
  3.2.1: in decode the up-projection of the keys is absorbed into the query, so
  each head's 128-value no-position query becomes a 512-value latent query,
  q_latent[h] = q_nope[h] · W_UK[h] with W_UK[h] of shape 128 x 512 (the
  per-head slice of the key up-projection, rows = no-position dims, columns =
  latent dims).  Section 6.1 names this fused step (MLAProlog).
* "CloudMatrix384 ... (digest)", section 3.2 on MLA optimisation: the prolog
  fuses RMSNorm, the Q/K/V projections and RoPE; the pages give no formula
  for the latter two, so the plain readings are used:
  - RoPE on the 64 position dims, pairs (2i, 2i+1) rotated by the angle
    pos * base^(-2i/64) (base a parameter, 10000 for DeepSeek V3/R1);
  - RMSNorm y = x / sqrt(mean(x^2) + eps) * gamma over the 512 latent values.
* The token's position is its cache slot: with seq_lens counting this step's
  tokens, query token t of request b sits at pos = seq_len - s_q + t, which is
  where its c_kv ‖ k_rope row is appended (page block_table[b][pos // 64],
  row pos % 64).

Every function is written from those definitions with numpy's fp64 routines;
the pins live in ``tests/test_prolog_pins.py`` (an explicit-loop contraction,
the unabsorbed score, complex-exponential rotation, closed forms).
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def absorb_q(q_nope, w_uk) -> np.ndarray:
    """q_latent[t, h, :] = q_nope[t, h, :] · W_UK[h]  ([T, H, dn] x [H, dn, dl] -> [T, H, dl])."""
    q = _f64(q_nope)
    w = _f64(w_uk)
    return np.matmul(q.transpose(1, 0, 2), w).transpose(1, 0, 2)   # per head: [T, dn] @ [dn, dl]


def rope_angles(pos, d_rope: int, base: float) -> np.ndarray:
    """Angle of pair i at each position: pos * base^(-2i/d_rope); shape pos.shape + (d_rope/2,)."""
    i = np.arange(d_rope // 2, dtype=np.float64)
    inv_freq = np.power(float(base), -2.0 * i / d_rope)
    return np.asarray(pos, dtype=np.float64)[..., None] * inv_freq


def rope(x, pos, base: float) -> np.ndarray:
    """Rotate pairs (2i, 2i+1) of the last axis of x by rope_angles(pos); pos broadcasts over x[..., 0]."""
    v = _f64(x)
    ang = rope_angles(pos, v.shape[-1], base)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., 0::2], v[..., 1::2]
    out = np.empty(np.broadcast_shapes(v.shape, ang.shape[:-1] + (v.shape[-1],)))
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def rms_norm(x, gamma, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gamma over the last axis."""
    v = _f64(x)
    g = _f64(gamma)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps) * g


def positions(seq_lens, s_q: int) -> np.ndarray:
    """pos[b, t] = seq_lens[b] - s_q + t: the cache slot and RoPE position of each new token."""
    sl = np.asarray(seq_lens, dtype=np.int64)
    return sl[:, None] - s_q + np.arange(s_q, dtype=np.int64)[None, :]


def prolog(q_nope, q_pe, kv_latent, k_pe, w_uk, kv_norm_weight, kv_cache, block_table, seq_lens, *,
           rope_base: float = 10000.0, rms_eps: float = 1e-6):
    """The whole slice for one decode step.

    q_nope [B][s_q][H][128], q_pe [B][s_q][H][64], kv_latent [B][s_q][512],
    k_pe [B][s_q][64], w_uk [H][128][512], kv_norm_weight [512],
    kv_cache [P][page][576], block_table [B][max_pages], seq_lens [B].

    Returns (q_latent [B][s_q][H][512], q_rope [B][s_q][H][64], cache) in fp64,
    where cache is kv_cache (as fp64) with each new token's normalised latent
    and rotated k_rope written at its slot.  Raises ValueError for a position
    below 0 or past the block table, or a page outside the pool.
    """
    qn = _f64(q_nope)
    B, S, H, DN = qn.shape
    pos = positions(seq_lens, S)
    q_lat = absorb_q(qn.reshape(B * S, H, DN), w_uk).reshape(B, S, H, -1)
    q_rot = rope(q_pe, pos[:, :, None], rope_base)
    c = rms_norm(kv_latent, kv_norm_weight, rms_eps)
    k_rot = rope(k_pe, pos, rope_base)
    cache = _f64(kv_cache).copy()
    bt = np.asarray(block_table)
    page_size = cache.shape[1]
    DL = c.shape[-1]
    for b in range(B):
        for t in range(S):
            p = int(pos[b, t])
            if p < 0 or p // page_size >= bt.shape[1]:
                raise ValueError(f"oracle prolog: position {p} of request {b} outside its block table")
            page = int(bt[b, p // page_size])
            if page < 0 or page >= cache.shape[0]:
                raise ValueError(f"oracle prolog: page {page} outside the pool")
            cache[page, p % page_size, :DL] = c[b, t]
            cache[page, p % page_size, DL:] = k_rot[b, t]
    return q_lat, q_rot, cache
