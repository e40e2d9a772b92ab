"""Pins for the fp64 oracle: each test ties it to something other than itself.

- the unabsorbed multi-head form (weight absorption, "Huawei Ascend servers:
  DeepSeek V3/R1 inference best practice" sections 3.1.2 / 3.2.1): decompress
  K and V with random per-head matrices and run standard attention;
- a dense float64 library softmax (torch) on tiny inputs;
- closed forms (one key, equal rows, zero query, one dominant key);
- invariants (split + merge, page permutation, MTP causality, weights sum to 1).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _f64_problem(rng, lens, s_q=1, H=4, max_pages=None, page=W.PAGE):
    """Random fp64 inputs in the oracle's layout (not bf16: used where exactness matters)."""
    B = len(lens)
    npages = [(L + page - 1) // page for L in lens]
    P = sum(npages)
    mp = max(npages) if max_pages is None else max_pages
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((B, mp), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[k:k + n]
        k += n
    return dict(
        q_latent=rng.standard_normal((B, s_q, H, W.D_LATENT)),
        q_rope=rng.standard_normal((B, s_q, H, W.D_ROPE)),
        kv_cache=rng.standard_normal((P, page, W.D_ROW)),
        block_table=bt,
        seq_lens=np.array(lens, dtype=np.int32),
    )


def _gather_rows(kv, bt_row, L):
    """Dense [L][576] rows of one request, gathered through its block table."""
    page = kv.shape[1]
    idx = np.arange(L)
    return kv[bt_row[idx // page], idx % page]


def _run(inp, s_q, scale=W.SCALE, **kw):
    return oracle.decode(inp["q_latent"], inp["q_rope"], inp["kv_cache"], inp["block_table"],
                         inp["seq_lens"], s_q=s_q, scale=scale, **kw)


# --------------------------------------------------------------------------- unabsorbed form

def test_unabsorbed_mha_equivalence():
    """Absorbed latent attention == standard MHA over decompressed per-head K and V.

    Per head h: K_j = [W_UK^h c_kv_j ; k_rope_j] (128 + 64 = 192 dims),
    V_j = W_UV^h c_kv_j (128 dims), q = [q_nope ; q_rope], scale 1/sqrt(192).
    The absorbed query is q_lat = W_UK^h^T q_nope, and the absorbed output maps
    back through W_UV^h.  Includes an MTP step (s_q = 2, causal inside it).
    """
    rng = np.random.default_rng(11)
    H, d_nope, d_v = 4, 128, 128
    lens = [5, 70, 129]
    s_q = 2
    inp = _f64_problem(rng, lens, s_q=s_q, H=H)
    B = len(lens)
    W_UK = rng.standard_normal((H, d_nope, W.D_LATENT)) / math.sqrt(W.D_LATENT)
    W_UV = rng.standard_normal((H, d_v, W.D_LATENT)) / math.sqrt(W.D_LATENT)
    q_nope = rng.standard_normal((B, s_q, H, d_nope))
    # absorb W_UK into the query
    inp["q_latent"] = np.einsum("bthn,hnd->bthd", q_nope, W_UK)
    o_lat, lse = _run(inp, s_q)

    for b in range(B):
        rows = _gather_rows(inp["kv_cache"], inp["block_table"][b], lens[b])
        c_kv, k_rope = rows[:, :W.D_LATENT], rows[:, W.D_LATENT:]
        for t in range(s_q):
            vis = lens[b] - s_q + 1 + t
            for h in range(H):
                K = np.concatenate([c_kv[:vis] @ W_UK[h].T, k_rope[:vis]], axis=1)  # [vis][192]
                V = c_kv[:vis] @ W_UV[h].T                                          # [vis][128]
                q = np.concatenate([q_nope[b, t, h], inp["q_rope"][b, t, h]])
                s = (K @ q) / math.sqrt(192.0)
                m = s.max()
                p = np.exp(s - m)
                o_ref = (p @ V) / p.sum()
                lse_ref = m + math.log(p.sum())
                np.testing.assert_allclose(W_UV[h] @ o_lat[b, t, h], o_ref, rtol=0, atol=1e-12)
                assert abs(lse[b, t, h] - lse_ref) < 1e-12


# --------------------------------------------------------------------------- library routine

def test_dense_torch_softmax_tiny_config():
    """Tiny workload (bf16 inputs) against torch float64 softmax(QK^T scale) V."""
    w = W.workload("tiny")
    inp = W.make_inputs(w, poison=True, extra_pages=2)
    o, lse = _run(inp, w.s_q)
    kv = inp["kv_cache"].double()
    for b, L in enumerate(w.seq_lens):
        idx = torch.arange(L)
        rows = kv[inp["block_table"][b][idx // W.PAGE].long(), idx % W.PAGE]   # [L][576]
        q = torch.cat([inp["q_latent"][b, 0].double(), inp["q_rope"][b, 0].double()], dim=1)
        s = (q @ rows.T) * W.SCALE                                                # [H][L]
        ref = torch.softmax(s, dim=1) @ rows[:, :W.D_LATENT]
        ref_lse = torch.logsumexp(s, dim=1)
        np.testing.assert_allclose(o[b, 0], ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b, 0], ref_lse.numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- closed forms

def test_single_key_returns_that_row():
    """L = 1: the only key gets weight 1, so o is its latent row and lse its score."""
    w = W.workload("tiny")
    inp = W.make_inputs(w)
    b = w.seq_lens.index(1)
    o, lse = _run(inp, 1)
    row = inp["kv_cache"][inp["block_table"][b, 0].long(), 0].double().numpy()
    q = np.concatenate([inp["q_latent"][b, 0].double().numpy(),
                        inp["q_rope"][b, 0].double().numpy()], axis=1)
    np.testing.assert_array_equal(o[b, 0], np.broadcast_to(row[:W.D_LATENT], (W.NUM_HEADS, W.D_LATENT)))
    np.testing.assert_allclose(lse[b, 0], W.SCALE * (q @ row), rtol=0, atol=1e-12)


def test_equal_rows_and_zero_query():
    rng = np.random.default_rng(5)
    lens = [77, 130]
    inp = _f64_problem(rng, lens, H=3)
    row = rng.standard_normal(W.D_ROW)
    # request 0: every cached row identical -> o = row, lse = s + ln L
    for j in range(lens[0]):
        inp["kv_cache"][inp["block_table"][0][j // W.PAGE], j % W.PAGE] = row
    # request 1: zero query -> uniform weights: o = mean of rows, lse = ln L
    inp["q_latent"][1] = 0.0
    inp["q_rope"][1] = 0.0
    o, lse = _run(inp, 1)
    q0 = np.concatenate([inp["q_latent"][0, 0], inp["q_rope"][0, 0]], axis=1)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(row[:W.D_LATENT], o[0, 0].shape), atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], W.SCALE * (q0 @ row) + math.log(lens[0]), atol=1e-12)
    rows1 = _gather_rows(inp["kv_cache"], inp["block_table"][1], lens[1])
    np.testing.assert_allclose(o[1, 0], np.broadcast_to(rows1[:, :W.D_LATENT].mean(0), o[1, 0].shape),
                               atol=1e-12)
    np.testing.assert_allclose(lse[1, 0], math.log(lens[1]), atol=1e-12)


def test_dominant_key():
    """A key whose score exceeds every other by about 80 takes all the weight (exp(-80) ~ 1e-35)."""
    rng = np.random.default_rng(6)
    lens = [150]
    inp = _f64_problem(rng, lens, H=2)
    j_star = 97
    r = inp["kv_cache"][inp["block_table"][0][j_star // W.PAGE], j_star % W.PAGE]
    inp["q_latent"][0, 0, :] = 0.0
    inp["q_rope"][0, 0, :] = 0.0
    inp["q_latent"][0, 0, :, :] = 60.0 * r[:W.D_LATENT] / np.linalg.norm(r)
    o, lse = _run(inp, 1)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(r[:W.D_LATENT], o[0, 0].shape), atol=1e-12)


# --------------------------------------------------------------------------- invariants

def test_split_merge_equals_unsplit():
    """Partials over any partition of the visible keys merge to the unsplit result."""
    rng = np.random.default_rng(7)
    lens = [1, 64, 65, 300, 1000]
    s_q = 2
    lens[0] = 2  # s_q = 2 needs L >= 2
    inp = _f64_problem(rng, lens, s_q=s_q, H=2)
    o_full, lse_full = _run(inp, s_q)
    for b, L in enumerate(lens):
        for t in range(s_q):
            vis = L - s_q + 1 + t
            for h in range(2):
                n_cuts = int(rng.integers(0, 5))
                cuts = np.sort(rng.integers(0, vis + 1, size=n_cuts))
                bounds = [0, *cuts.tolist(), vis]
                ranges = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
                rows = [(b, t, h)] * len(ranges)
                op, lp = _run(inp, s_q, rows=rows, ranges=ranges)
                om, lm = oracle.merge(op, lp)
                np.testing.assert_allclose(om, o_full[b, t, h], rtol=0, atol=1e-12)
                assert abs(lm - lse_full[b, t, h]) < 1e-12


def test_page_permutation_invariance():
    """Moving pages in the pool and rewriting block_table leaves results bit-identical."""
    w = W.workload("tiny")
    inp = W.make_inputs(w, extra_pages=3)
    o1, l1 = _run(inp, 1)
    P = inp["kv_cache"].shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(99))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    kv2 = inp["kv_cache"][perm]                      # new page i = old page perm[i]
    bt2 = inp["block_table"].clone()
    m = bt2 >= 0
    bt2[m] = inv[bt2[m].long()].to(torch.int32)
    o2, l2 = oracle.decode(inp["q_latent"], inp["q_rope"], kv2, bt2, inp["seq_lens"], s_q=1,
                           scale=W.SCALE)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_mtp_token_matches_single_token_run():
    """Query token t of an s_q = 2 step equals an s_q = 1 step over L - 1 + t keys."""
    w = W.custom([2, 65, 129, 700], s_q=2, seed=12)
    inp = W.make_inputs(w)
    o2, l2 = _run(inp, 2)
    for t in range(2):
        sl = inp["seq_lens"] - 1 + t
        o1, l1 = oracle.decode(inp["q_latent"][:, t:t + 1], inp["q_rope"][:, t:t + 1],
                               inp["kv_cache"], inp["block_table"], sl, s_q=1, scale=W.SCALE)
        np.testing.assert_array_equal(o2[:, t], o1[:, 0])
        np.testing.assert_array_equal(l2[:, t], l1[:, 0])


def test_weights_sum_to_one():
    """With every latent value 1, o = sum_j softmax_j = 1 in every dim."""
    rng = np.random.default_rng(8)
    inp = _f64_problem(rng, [33, 257], H=3)
    inp["kv_cache"][:, :, :W.D_LATENT] = 1.0
    o, _ = _run(inp, 1)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)


def test_merge_closed_forms():
    rng = np.random.default_rng(9)
    o = rng.standard_normal(16)
    om, lm = oracle.merge(np.stack([o, o, o]), np.array([1.5, 1.5, 1.5]))
    np.testing.assert_allclose(om, o, atol=1e-15)
    assert abs(lm - (1.5 + math.log(3))) < 1e-14
    om, lm = oracle.merge(np.stack([o, np.zeros(16)]), np.array([0.25, -np.inf]))
    np.testing.assert_allclose(om, o, atol=1e-15)
    assert lm == 0.25
    om, lm = oracle.merge(np.zeros((0, 16)), np.zeros(0))
    assert lm == -np.inf and not om.any()


def test_errors_are_reported():
    w = W.workload("tiny")
    inp = W.make_inputs(w)
    bad = inp["block_table"].clone()
    bad[0, 0] = 10_000
    with pytest.raises(ValueError, match="page pool"):
        oracle.decode(inp["q_latent"], inp["q_rope"], inp["kv_cache"], bad, inp["seq_lens"],
                      s_q=1, scale=W.SCALE)
    short = torch.tensor([1, 1, 1, 1], dtype=torch.int32)
    with pytest.raises(ValueError, match="seq_len"):
        oracle.decode(inp["q_latent"].repeat(1, 2, 1, 1), inp["q_rope"].repeat(1, 2, 1, 1),
                      inp["kv_cache"], inp["block_table"], short, s_q=2, scale=W.SCALE)
