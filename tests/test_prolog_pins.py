"""Pins for the fp64 prolog oracle (CPU only).

Each test ties the oracle to something other than its own formula: explicit
loops, the unabsorbed attention score, complex-exponential rotation from the
standard library, closed forms and group properties of rotations.
"""

import cmath
import math

import numpy as np
import pytest

from oracle import prolog as P


def _rng(seed):
    return np.random.default_rng(seed)


def test_absorb_matches_explicit_loops():
    r = _rng(1)
    T, H, DN, DL = 2, 3, 4, 5
    q = r.standard_normal((T, H, DN))
    w = r.standard_normal((H, DN, DL))
    out = P.absorb_q(q, w)
    for t in range(T):
        for h in range(H):
            for n in range(DL):
                acc = 0.0
                for k in range(DN):
                    acc += q[t, h, k] * w[h, k, n]
                assert out[t, h, n] == pytest.approx(acc, rel=1e-13, abs=1e-13)


def test_absorbed_score_equals_unabsorbed_score():
    """q_latent[h] · c == q_nope[h] · k_nope[h] with the key up-projected per head: k_nope[h] = W_UK[h] c."""
    r = _rng(2)
    T, H, DN, DL = 3, 4, 16, 24
    q = r.standard_normal((T, H, DN))
    w = r.standard_normal((H, DN, DL)) / math.sqrt(DN)
    c = r.standard_normal((7, DL))
    ql = P.absorb_q(q, w)
    for h in range(H):
        k_nope = c @ w[h].T                      # [7, DN], one up-projected key per latent row
        np.testing.assert_allclose(ql[:, h, :] @ c.T, q[:, h, :] @ k_nope.T, rtol=1e-12, atol=1e-12)


def test_rope_frequencies_closed_form():
    ang = P.rope_angles(np.array(1), 64, 10000.0)
    assert ang.shape == (32,)
    assert ang[0] == 1.0                          # the first pair turns one radian per position
    np.testing.assert_allclose(ang[1:] / ang[:-1], 10000.0 ** (-1.0 / 32), rtol=1e-14)
    assert ang[31] == pytest.approx(10000.0 ** (-31.0 / 32), rel=1e-14)
    np.testing.assert_allclose(P.rope_angles(np.array(37), 64, 10000.0), 37 * ang, rtol=1e-15)


def test_rope_is_complex_rotation_of_interleaved_pairs():
    r = _rng(3)
    x = r.standard_normal(64)
    pos = 123
    out = P.rope(x, pos, 10000.0)
    ang = P.rope_angles(np.array(pos), 64, 10000.0)
    for i in range(32):
        z = complex(x[2 * i], x[2 * i + 1]) * cmath.exp(1j * ang[i])
        assert out[2 * i] == pytest.approx(z.real, abs=1e-12)
        assert out[2 * i + 1] == pytest.approx(z.imag, abs=1e-12)
    e0 = np.zeros(64)
    e0[0] = 1.0
    turned = P.rope(e0, 1, 10000.0)               # pairs are adjacent dims, not halves
    assert turned[0] == pytest.approx(math.cos(1.0)) and turned[1] == pytest.approx(math.sin(1.0))
    assert np.all(turned[2:] == 0.0)


def test_rope_rotation_group_properties():
    r = _rng(4)
    x = r.standard_normal((5, 64))
    k = r.standard_normal((5, 64))
    np.testing.assert_array_equal(P.rope(x, 0, 10000.0), x)
    for m, n in ((3, 11), (1000, 17), (65535, 65530)):
        y = P.rope(x, m, 10000.0)
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
        np.testing.assert_allclose(P.rope(y, n, 10000.0), P.rope(x, m + n, 10000.0), atol=1e-9)
        # relative position: the score of (query at m, key at n) depends only on m - n
        lhs = np.sum(P.rope(x, m, 10000.0) * P.rope(k, n, 10000.0), axis=-1)
        rhs = np.sum(P.rope(x, m - n, 10000.0) * k, axis=-1)
        np.testing.assert_allclose(lhs, rhs, atol=1e-9)


def test_rms_norm_closed_forms():
    a, eps = 0.75, 1e-6
    x = np.full(512, a)
    np.testing.assert_allclose(P.rms_norm(x, np.ones(512), eps), a / math.sqrt(a * a + eps), rtol=1e-15)
    r = _rng(5)
    v = r.standard_normal(512)
    g = r.standard_normal(512)
    y = P.rms_norm(v, np.ones(512), 0.0)
    assert math.sqrt(np.mean(y * y)) == pytest.approx(1.0, rel=1e-13)
    np.testing.assert_allclose(P.rms_norm(7.5 * v, g, 0.0), P.rms_norm(v, g, 0.0), rtol=1e-12)
    np.testing.assert_allclose(P.rms_norm(v, g, 0.0), y * g, rtol=1e-13)


def _small_problem(seed, seq_lens, s_q, H=2, DN=8, DL=16, DR=8, page=4, pool=None, max_pages=None):
    r = _rng(seed)
    B = len(seq_lens)
    pages_per = [(L + page - 1) // page for L in seq_lens]
    pool = pool or sum(pages_per) + 2
    mp = max_pages or max(pages_per)
    perm = r.permutation(pool)
    bt = np.full((B, mp), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[k:k + n]
        k += n
    return dict(q_nope=r.standard_normal((B, s_q, H, DN)), q_pe=r.standard_normal((B, s_q, H, DR)),
                kv_latent=r.standard_normal((B, s_q, DL)), k_pe=r.standard_normal((B, s_q, DR)),
                w_uk=r.standard_normal((H, DN, DL)), kv_norm_weight=r.standard_normal(DL),
                kv_cache=r.standard_normal((pool, page, DL + DR)), block_table=bt,
                seq_lens=np.array(seq_lens, dtype=np.int32))


def test_prolog_appends_at_the_token_positions_only():
    s_q = 2
    inp = _small_problem(6, [5, 2, 9], s_q)
    ql, qr, cache = P.prolog(**inp, rope_base=100.0, rms_eps=1e-6)
    old = inp["kv_cache"]
    page = old.shape[1]
    written = np.zeros(old.shape[:2], dtype=bool)
    for b, L in enumerate(inp["seq_lens"]):
        for t in range(s_q):
            p = L - s_q + t
            pg = inp["block_table"][b, p // page]
            written[pg, p % page] = True
            row = cache[pg, p % page]
            x = inp["kv_latent"][b, t]
            ref_c = x / math.sqrt(float(np.mean(x * x)) + 1e-6) * inp["kv_norm_weight"]
            np.testing.assert_allclose(row[:16], ref_c, rtol=1e-13)
            ref_k = P.rope(inp["k_pe"][b, t], p, 100.0)
            np.testing.assert_allclose(row[16:], ref_k, rtol=1e-13)
            np.testing.assert_allclose(qr[b, t], P.rope(inp["q_pe"][b, t], p, 100.0), rtol=1e-13)
    assert written.sum() == 3 * s_q
    np.testing.assert_array_equal(cache[~written], old[~written])
    assert ql.shape == (3, s_q, 2, 16)


def test_prolog_positions_are_relative_across_offsets():
    """Same raw tokens appended at two different offsets give the same q_rope · k_rope scores."""
    s_q = 2
    a = _small_problem(7, [6], s_q)
    b = dict(a, seq_lens=np.array([11], dtype=np.int32))
    b["block_table"] = np.array([[3, 1, 0]], dtype=np.int32)
    a["block_table"] = np.array([[2, 3]], dtype=np.int32)
    out = []
    for inp in (a, b):
        _, qr, cache = P.prolog(**inp, rope_base=50.0, rms_eps=1e-6)
        L = int(inp["seq_lens"][0])
        rows = []
        for t in range(s_q):
            p = L - s_q + t
            rows.append(cache[inp["block_table"][0, p // 4], p % 4, 16:])
        out.append(np.einsum("thd,jd->thj", qr[0], np.array(rows)))
    np.testing.assert_allclose(out[0], out[1], atol=1e-10)


@pytest.mark.parametrize("seq_lens,bt_fix", [([1], None), ([4], "bad_page"), ([9], "short_table")])
def test_prolog_rejects_bad_slots(seq_lens, bt_fix):
    inp = _small_problem(8, seq_lens if bt_fix != "short_table" else [4], 2)
    if bt_fix == "bad_page":
        inp["block_table"][0, 0] = inp["kv_cache"].shape[0]
    if bt_fix == "short_table":
        inp["seq_lens"] = np.array(seq_lens, dtype=np.int32)
    with pytest.raises(ValueError):
        P.prolog(**inp)
