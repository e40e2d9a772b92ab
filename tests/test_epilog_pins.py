"""Pins for the fp64 epilog oracle (CPU only): explicit loops, index order, the unabsorbed layer."""

import math

import numpy as np
import pytest

import oracle
from oracle import epilog as E
from oracle import prolog as P


def _rng(seed):
    return np.random.default_rng(seed)


def test_uv_project_matches_loops():
    r = _rng(1)
    T, H, DV, DL = 2, 3, 4, 5
    o = r.standard_normal((T, H, DL))
    w = r.standard_normal((H, DV, DL))
    out = E.uv_project(o, w)
    for t in range(T):
        for h in range(H):
            for v in range(DV):
                assert out[t, h, v] == pytest.approx(sum(w[h, v, c] * o[t, h, c] for c in range(DL)),
                                                     rel=1e-13, abs=1e-13)


def test_o_project_matches_loops_and_concat_order():
    r = _rng(2)
    T, H, DV, HID = 2, 3, 4, 5
    o = r.standard_normal((T, H, DV))
    w = r.standard_normal((HID, H * DV))
    out = E.o_project(o, w)
    for t in range(T):
        for n in range(HID):
            acc = 0.0
            for h in range(H):
                for v in range(DV):
                    acc += w[n, h * DV + v] * o[t, h, v]
            assert out[t, n] == pytest.approx(acc, rel=1e-13, abs=1e-13)
    # a single weight at column h * dv + v picks exactly o_v[:, h, v]
    sel = np.zeros((1, H * DV))
    sel[0, 2 * DV + 1] = 1.0
    np.testing.assert_array_equal(E.o_project(o, sel)[:, 0], o[:, 2, 1])


def test_unabsorbed_closed_forms():
    r = _rng(3)
    H, DN, DR, DL, DV = 2, 4, 2, 6, 3
    wk = r.standard_normal((H, DN, DL))
    wv = r.standard_normal((H, DV, DL))
    c = r.standard_normal((1, DL))
    out = E.unabsorbed_attention(r.standard_normal((H, DN)), r.standard_normal((H, DR)), c,
                                 r.standard_normal((1, DR)), wk, wv, 0.3)
    np.testing.assert_allclose(out, np.stack([wv[h] @ c[0] for h in range(H)]), rtol=1e-13)
    # identical rows: every key scores the same, the output is that row's value
    cc = np.repeat(c, 5, axis=0)
    kr = np.zeros((5, DR))
    out = E.unabsorbed_attention(r.standard_normal((H, DN)), r.standard_normal((H, DR)), cc, kr, wk, wv,
                                 0.3)
    np.testing.assert_allclose(out, np.stack([wv[h] @ c[0] for h in range(H)]), rtol=1e-12)


def test_absorbed_decode_then_uv_equals_unabsorbed():
    """Prolog absorb -> decode oracle -> W_UV step equals plain multi-head attention, per token."""
    r = _rng(4)
    H, DN, DR, DL, DV, PG = 4, 8, 8, 16, 8, 4
    seq_lens = [3, 9]
    s_q = 2
    B = len(seq_lens)
    pages = [(L + PG - 1) // PG for L in seq_lens]
    pool = sum(pages)
    perm = r.permutation(pool).astype(np.int32)
    bt = np.full((B, max(pages)), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    cache = r.standard_normal((pool, PG, DL + DR))
    q_nope = r.standard_normal((B, s_q, H, DN))
    q_rope = r.standard_normal((B, s_q, H, DR))
    wk = r.standard_normal((H, DN, DL)) / math.sqrt(DN)
    wv = r.standard_normal((H, DV, DL)) / math.sqrt(DL)
    scale = 1.0 / math.sqrt(DN + DR)
    q_lat = P.absorb_q(q_nope.reshape(B * s_q, H, DN), wk).reshape(B, s_q, H, DL)
    o_lat, _ = oracle.decode(q_lat, q_rope, cache, bt, np.array(seq_lens, dtype=np.int32), s_q=s_q,
                             scale=scale)
    o_v = E.uv_project(o_lat.reshape(B * s_q, H, DL), wv).reshape(B, s_q, H, DV)
    for b, L in enumerate(seq_lens):
        rows = np.stack([cache[bt[b, j // PG], j % PG] for j in range(L)])
        for t in range(s_q):
            vis = L - s_q + 1 + t
            ref = E.unabsorbed_attention(q_nope[b, t], q_rope[b, t], rows[:vis, :DL], rows[:vis, DL:],
                                         wk, wv, scale)
            np.testing.assert_allclose(o_v[b, t], ref, rtol=1e-10, atol=1e-12)
