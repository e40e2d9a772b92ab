"""Power-of-two running maxima (MLA_FLAG_POW2_MAX) against the fp64 oracle.

The AMLA-style mode keeps every running max an integer in log2 units, so each
rescale of P and of the output accumulator is by an exact power of two.  It
computes the same attention, so the acceptance bar is the usual one
(o_latent max |err| <= 2e-2, mean <= 2e-3, lse <= 1e-3).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, oracle_full, run_gpu, sample_rows, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import mla_decode_attention_02_gb300 as mla  # noqa: E402


def _parity(inp, what):
    o, lse, _ = run_gpu(inp, pow2_max=True)
    o_ref, lse_ref = oracle_full(inp)
    return assert_close(o, lse, o_ref, lse_ref, what)


def test_pow2_tiny_poisoned():
    _parity(W.make_inputs(W.workload("tiny"), poison=True, extra_pages=3), "tiny pow2")


@pytest.mark.parametrize("s_q", [1, 2])
def test_pow2_ragged(s_q):
    lens = [2, 3, 63, 64, 65, 127, 128, 129, 191, 500, 1000, 1537, 3001, 4096]
    _parity(W.make_inputs(W.custom(lens, s_q=s_q, seed=80 + s_q), poison=True, extra_pages=5),
            f"ragged s_q={s_q} pow2")


def test_pow2_rising_scores():
    """The running max keeps rising by more than 2^8: the exact power-of-two rescales of O
    and of the lower P half run on many pages.  The scores rise through k_rope (scaled with
    the page index); c_kv is halved so that the peaked rows' outputs (|o| up to about 2.3
    instead of 4.6) leave the bar to the attention's own error: at |o| near 4.6 the bf16
    rounding of the output alone is up to 0.016 of the 0.02, and with power-of-two maxima
    the dominant P of a peaked row is no longer exactly 1, so it is rounded as well."""
    lens = [700, 1500, 3000, 64, 130, 2049]
    w = W.custom(lens, s_q=1, seed=85)
    inp = W.make_inputs(w)
    inp["q_rope"] = (inp["q_rope"].float() * 3).to(torch.bfloat16)
    kv = inp["kv_cache"].float()
    kv[:, :, :W.D_LATENT] *= 0.5
    bt = inp["block_table"]
    for b, L in enumerate(lens):
        for pi in range((L + 63) // 64):
            kv[int(bt[b, pi]), :, W.D_LATENT:] *= 1.0 + pi / 4.0
    inp["kv_cache"] = kv.to(torch.bfloat16)
    _parity(inp, "rising scores pow2")


@pytest.mark.parametrize("name,nrows", [("uniform", 64), ("mixed", 64)])
def test_pow2_full_size_sampled(name, nrows):
    w = W.workload(name)
    inp = W.make_inputs(w)
    o, lse, _ = run_gpu(inp, pow2_max=True)
    rows = sample_rows(w, nrows, seed=7 + sum(map(ord, name)))
    o_ref, lse_ref = oracle.decode(inp["q_latent"], inp["q_rope"], inp["kv_cache"],
                                   inp["block_table"], inp["seq_lens"], s_q=w.s_q,
                                   scale=W.SCALE, rows=rows)
    b, t, h = rows[:, 0], rows[:, 1], rows[:, 2]
    assert_close(o[b, t, h], lse[b, t, h], o_ref, lse_ref, name + " pow2")


def test_pow2_deterministic_and_close_to_default():
    w = W.custom([700, 5000, 64, 12000], s_q=1, seed=86)
    inp = W.make_inputs(w)
    d = to_device(inp)
    p = mla.plan(d["seq_lens"], s_q=1, max_pages_per_seq=d["block_table"].shape[1])
    args = (d["q_latent"], d["q_rope"], d["kv_cache"], d["block_table"])
    o1, l1 = mla.decode(p, *args, scale=d["scale"], pow2_max=True)
    o2, l2 = mla.decode(p, *args, scale=d["scale"], pow2_max=True)
    o0, l0 = mla.decode(p, *args, scale=d["scale"])
    assert mla.check(p) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert (o1.float() - o0.float()).abs().max().item() <= 2e-2
    assert (l1 - l0).abs().max().item() <= 1e-3
