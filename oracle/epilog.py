"""fp64 oracle for the step after decode attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs
may import this module; the CUDA library never does.

What it computes:

* "Huawei Ascend servers: DeepSeek V3/R1 inference best practice", section
  3.2.1: with the weights absorbed, attention returns each head's output in
  the 512-value latent space; the value up-projection W_UV[h] (128 x 512 per
  head: row v holds the latent weights of value dim v) brings it back to the
  head's 128 value dims, o_v[t][h][v] = sum_c W_UV[h][v][c] * o_latent[t][h][c].
* Sections 3.2.1-3.3 (figures 5-9, "O Proj"): the output projection then maps
  the concatenated heads (128 x 128 = 16384 values) to the hidden size,
  out[t] = W_O . o_v[t] with W_O of shape 7168 x 16384 (DeepSeek V3/R1's
  hidden size; the pages name the projection but print no shape).
* ``unabsorbed_attention`` is the same layer written without absorption, as
  plain multi-head attention with 192-value keys [W_UK[h] c ; k_rope] and
  128-value values W_UV[h] c per cached row, for the GPU check that decode
  followed by the W_UV step equals it.

Pins: ``tests/test_epilog_pins.py``.
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


def uv_project(o_latent, w_uv) -> np.ndarray:
    """o_v[t, h, v] = sum_c W_UV[h, v, c] o_latent[t, h, c]  ([T, H, dl] x [H, dv, dl] -> [T, H, dv])."""
    o = _f64(o_latent)
    w = _f64(w_uv)
    return np.matmul(o.transpose(1, 0, 2), w.transpose(0, 2, 1)).transpose(1, 0, 2)


def o_project(o_v, w_o) -> np.ndarray:
    """out[t] = W_O . concat_h o_v[t, h]  ([T, H, dv] x [hidden, H * dv] -> [T, hidden])."""
    o = _f64(o_v)
    return o.reshape(o.shape[0], -1) @ _f64(w_o).T


def unabsorbed_attention(q_nope, q_rope, latent, k_rope, w_uk, w_uv, scale: float) -> np.ndarray:
    """Plain multi-head attention over one request's visible rows, without absorption.

    q_nope [H, dn], q_rope [H, dr] (one query token), latent [L, dl], k_rope [L, dr],
    w_uk [H, dn, dl], w_uv [H, dv, dl].  Keys of head h: [W_UK[h] c_j ; k_rope_j]
    (dn + dr values), values W_UV[h] c_j; returns o [H, dv].
    """
    qn, qr = _f64(q_nope), _f64(q_rope)
    c, kr = _f64(latent), _f64(k_rope)
    wk, wv = _f64(w_uk), _f64(w_uv)
    H = qn.shape[0]
    out = np.empty((H, wv.shape[1]))
    for h in range(H):
        k_nope = c @ wk[h].T                     # [L, dn]: each cached row up-projected
        v = c @ wv[h].T                          # [L, dv]
        s = scale * (k_nope @ qn[h] + kr @ qr[h])
        p = np.exp(s - s.max())
        out[h] = (p / p.sum()) @ v
    return out
