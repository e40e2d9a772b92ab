"""Decode over the fp8 (e4m3) cache on cuda:0 (``mla_decode_fp8``) against the fp64 oracle.

The parity reference is ``oracle.fp8.decode``: the attention of the dequantised rows, which
is what the kernel computes (its only roundings are the bf16 path's: codes and k_rope / s are
exact bf16 operands, the per-token scale multiplies each fp32 score and is folded into each
weight before the weights are rounded to bf16).  The acceptance bar is the bf16 path's:
o_latent max |err| <= 2e-2 and mean |err| <= 2e-3, lse |err| <= 1e-3.  The gap to the bf16
cache's result is the quantisation error, reported by the bench, not a parity criterion.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, sample_rows, to_device
from oracle import fp8 as F

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import mla_decode_attention_02_gb300 as mla  # noqa: E402


def _quantize(kv):
    """The oracle's quantiser over a cache, a few hundred pages at a time (bounded memory)."""
    out = np.empty(tuple(kv.shape[:-1]) + (F.ROW_BYTES,), dtype=np.uint8)
    for p0 in range(0, kv.shape[0], 256):
        out[p0:p0 + 256] = F.quantize_cache(kv[p0:p0 + 256])
    return out


def _fp8_inputs(w, poison=False, extra_pages=0):
    inp = W.make_inputs(w, extra_pages=extra_pages)
    q8 = _quantize(inp["kv_cache"])                                # [pages][64][656] uint8
    if poison:
        # every slot past a row's end and every unused page: NaN codes and a NaN scale
        pages_per = [(L + 63) // 64 for L in w.seq_lens]
        used = np.zeros(q8.shape[0], dtype=bool)
        for b, n in enumerate(pages_per):
            pg = inp["block_table"][b, :n].numpy()
            used[pg] = True
            tail = w.seq_lens[b] - (n - 1) * 64
            last = q8[pg[-1]]
            last[tail:, :512] = 0x7F
            last[tail:, 640:644] = np.frombuffer(np.float32(np.nan).tobytes(), dtype=np.uint8)
        q8[~used, :, :512] = 0x7F
    inp["kv8"] = torch.from_numpy(q8)
    return inp


def _run(inp, s_q, pow2_max=False):
    d = to_device(inp)
    p = mla.plan(d["seq_lens"], s_q=s_q, max_pages_per_seq=d["block_table"].shape[1])
    o, lse = mla.decode_fp8(p, d["q_latent"], d["q_rope"], d["kv8"], d["block_table"], scale=d["scale"],
                            pow2_max=pow2_max)
    status = mla.check(p)
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy(), status


def _parity_full(inp, s_q, what, pow2_max=False):
    o, lse, status = _run(inp, s_q, pow2_max)
    assert status == 0, f"device status {status:#x}"
    o_ref, lse_ref = F.decode(inp["q_latent"], inp["q_rope"], inp["kv8"].numpy(), inp["block_table"],
                              inp["seq_lens"], s_q=s_q, scale=inp["scale"])
    return assert_close(o, lse, o_ref, lse_ref, what)


def test_fp8_tiny_poisoned():
    _parity_full(_fp8_inputs(W.workload("tiny"), poison=True, extra_pages=3), 1, "fp8 tiny")


@pytest.mark.parametrize("s_q", [1, 2])
def test_fp8_ragged_lengths(s_q):
    lens = [2, 3, 63, 64, 65, 127, 128, 129, 191, 500, 1000, 1537, 3001, 4096]
    _parity_full(_fp8_inputs(W.custom(lens, s_q=s_q, seed=90 + s_q), poison=True, extra_pages=5), s_q,
                 f"fp8 ragged s_q={s_q}")


def test_fp8_many_short_rows_and_splits():
    """Several items per unit (item start) and rows split across units (merge)."""
    rng = np.random.default_rng(93)
    lens = [int(x) for x in rng.integers(1, 300, size=200)] + [30000, 9000]
    _parity_full(_fp8_inputs(W.custom(lens, s_q=1, seed=93)), 1, "fp8 packed + split")


def test_fp8_pow2_max():
    lens = [700, 1500, 64, 3000]
    _parity_full(_fp8_inputs(W.custom(lens, s_q=1, seed=94)), 1, "fp8 pow2", pow2_max=True)


def _oracle_rows(inp, w, rows):
    """The oracle on sampled (b, t, h) rows, each request's pages dequantised on their own
    (a whole full-size cache in fp64 would take gigabytes)."""
    q8 = inp["kv8"].numpy()
    o_ref = np.empty((len(rows), W.D_LATENT))
    lse_ref = np.empty(len(rows))
    for b in sorted(set(rows[:, 0].tolist())):
        L = w.seq_lens[b]
        n = (L + 63) // 64
        pages = inp["block_table"][b, :n].numpy()
        deq = torch.from_numpy(F.dequantize_cache(q8[pages]))           # [n][64][576] fp64
        sel = np.nonzero(rows[:, 0] == b)[0]
        sub = rows[sel].copy()
        sub[:, 0] = 0
        o, l = oracle.decode(inp["q_latent"][b:b + 1].double(), inp["q_rope"][b:b + 1].double(), deq,
                             torch.arange(n, dtype=torch.int32)[None], torch.tensor([L], dtype=torch.int32),
                             s_q=w.s_q, scale=W.SCALE, rows=sub)
        o_ref[sel], lse_ref[sel] = o, l
    return o_ref, lse_ref


@pytest.mark.parametrize("name,nrows", [("uniform", 64), ("mixed", 64), ("mtp", 96)])
def test_fp8_full_size_sampled(name, nrows):
    w = W.workload(name)
    inp = _fp8_inputs(w)
    o, lse, status = _run(inp, w.s_q)
    assert status == 0
    rows = sample_rows(w, nrows, seed=11 + sum(map(ord, name)))
    o_ref, lse_ref = _oracle_rows(inp, w, rows)
    b, t, h = rows[:, 0], rows[:, 1], rows[:, 2]
    assert_close(o[b, t, h], lse[b, t, h], o_ref, lse_ref, "fp8 " + name)


def test_fp8_deterministic_and_quantiser_path():
    """Two runs are bit-identical, and the cache quantised on the GPU gives the same result."""
    w = W.custom([700, 5000, 64, 12000], s_q=1, seed=95)
    inp = _fp8_inputs(w)
    d = to_device(inp)
    p = mla.plan(d["seq_lens"], s_q=1, max_pages_per_seq=d["block_table"].shape[1])
    args = (d["q_latent"], d["q_rope"])
    o1, l1 = mla.decode_fp8(p, *args, d["kv8"], d["block_table"], scale=d["scale"])
    o2, l2 = mla.decode_fp8(p, *args, d["kv8"], d["block_table"], scale=d["scale"])
    kv8_gpu = mla.quantize_cache_fp8(d["kv_cache"])
    o3, l3 = mla.decode_fp8(p, *args, kv8_gpu, d["block_table"], scale=d["scale"])
    assert mla.check(p) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_fp8_bad_page_flagged():
    w = W.custom([300, 200], s_q=1, seed=96)
    inp = _fp8_inputs(w)
    inp["block_table"][0, 2] = inp["kv8"].shape[0] + 7
    o, lse, status = _run(inp, 1)
    assert status & mla.MLA_DEV_BAD_PAGE
    assert np.isnan(lse[0]).all()
    o_ref, lse_ref = F.decode(inp["q_latent"][1:2], inp["q_rope"][1:2], inp["kv8"].numpy(),
                              inp["block_table"][1:2], inp["seq_lens"][1:2], s_q=1, scale=W.SCALE)
    assert_close(o[1:2], lse[1:2], o_ref, lse_ref, "fp8 good row beside a bad one")


def test_fp8_every_code_exact():
    """Every finite e4m3 code, the subnormal ones and both signs included, reaches both
    contractions at its exact value.

    Eight requests of two tokens, each on its own page; token 0 holds the codes (dim d holds
    code d mod 256, the NaN codes 0x7F / 0xFF replaced by 0), token 1 is zero (s = 1).
    Requests 0-3 read the K side: head h of request b has q = 1 on dim 128 b + h and 0
    elsewhere, and token 0's s = 64, so the head's score is value(code) * 64 * scale against
    0 and lse = log(1 + exp(score)); reading the smallest subnormal (2^-9) as a normal
    number would move lse by more than 1e-2.  Requests 4-7 read the V side: q = 0, both
    tokens weigh 1/2, s = 1, so o_latent = value(code) / 2 on every dim, exactly
    representable in bf16.
    """
    B = 8
    lens = [2] * B
    w = W.custom(lens, s_q=1, seed=98)
    inp = W.make_inputs(w)
    codes = np.arange(512) % 256
    codes[(codes == 0x7F) | (codes == 0xFF)] = 0
    q8 = np.zeros((B, 64, F.ROW_BYTES), dtype=np.uint8)
    one = np.frombuffer(np.float32(1.0).tobytes(), dtype=np.uint8)
    q8[:, :, 640:644] = one                                         # every token: s = 1
    q8[:, 0, :512] = codes.astype(np.uint8)
    q8[:4, 0, 640:644] = np.frombuffer(np.float32(64.0).tobytes(), dtype=np.uint8)
    inp["kv8"] = torch.from_numpy(q8)
    bt = torch.zeros_like(inp["block_table"])
    bt[:, 0] = torch.arange(B, dtype=torch.int32)
    inp["block_table"] = bt
    ql = torch.zeros_like(inp["q_latent"])
    for b in range(4):
        ql[b, 0, torch.arange(128), 128 * b + torch.arange(128)] = 1.0
    inp["q_latent"] = ql
    inp["q_rope"] = torch.zeros_like(inp["q_rope"])
    o, lse, status = _run(inp, 1)
    assert status == 0
    o_ref, lse_ref = F.decode(inp["q_latent"], inp["q_rope"], q8, bt, inp["seq_lens"], s_q=1, scale=inp["scale"])
    value = F.e4m3_value(codes.astype(np.uint8))
    # K side: the reference lse is that of the exact code values
    score = value[128 * np.arange(4)[:, None] + np.arange(128)[None, :]] * 64.0 * inp["scale"]
    np.testing.assert_allclose(lse_ref[:4, 0], np.logaddexp(score, 0.0), rtol=0, atol=1e-9)
    assert np.abs(lse[:4, 0] - lse_ref[:4, 0]).max() <= 1e-3
    # V side: exact
    assert np.array_equal(o[4:, 0], np.broadcast_to(value / 2, (4, 128, 512)))
    np.testing.assert_allclose(lse[4:, 0], np.log(2.0), rtol=0, atol=1e-6)
