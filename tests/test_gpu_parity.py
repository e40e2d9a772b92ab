"""CUDA path vs the fp64 oracle, through the C ABI, on cuda:0.

Small cases compare every output element; the full-size workloads (in the
launch configuration bench.py times) compare sampled rows that the oracle
computes one by one.  Tolerances are the acceptance bar: o_latent
max |err| <= 2e-2 and mean |err| <= 2e-3, lse |err| <= 1e-3.
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


def _parity_full(w, **kw):
    inp = W.make_inputs(w, **kw)
    o, lse, _ = run_gpu(inp)
    o_ref, lse_ref = oracle_full(inp)
    return assert_close(o, lse, o_ref, lse_ref, w.name)


def test_tiny_poisoned():
    """The tiny workload (seq_lens 1, 63, 64, 200) with NaN in every masked slot and unused page."""
    _parity_full(W.workload("tiny"), poison=True, extra_pages=3)


@pytest.mark.parametrize("s_q", [1, 2])
def test_ragged_lengths(s_q):
    """Lengths around page and tile boundaries, several pages per row, poisoned tails."""
    lens = [2, 3, 63, 64, 65, 127, 128, 129, 191, 500, 1000, 1537, 3001, 4096]
    _parity_full(W.custom(lens, s_q=s_q, seed=20 + s_q), poison=True, extra_pages=5)


def test_split_rows_are_merged():
    """Few long rows: the schedule splits each across many units and the merge runs."""
    w = W.custom([30000, 17, 25000, 9000], s_q=1, seed=31)
    inp = W.make_inputs(w, poison=True)
    d = to_device(inp)
    p = mla.plan(d["seq_lens"], s_q=1, max_pages_per_seq=d["block_table"].shape[1])
    r = mla.parse_plan(mla.plan_device_bytes(p), w.batch, 1, mla.num_units())
    assert r["row_nparts"].max() > 1
    o, lse, _ = run_gpu(inp)
    o_ref, lse_ref = oracle_full(inp)
    assert_close(o, lse, o_ref, lse_ref, "split")


@pytest.mark.parametrize("s_q,batch", [(1, 240), (2, 120)])
def test_many_short_rows_packed(s_q, batch):
    """Many short rows: units run several items back to back (item start: q staged by
    TMA while the previous item drains), single-page items included; every element compared."""
    rng = np.random.default_rng(50 + s_q)
    lens = [int(x) for x in rng.integers(s_q, 300, size=batch)]
    lens[:4] = [s_q, 64, 65, 299]
    w = W.custom(lens, s_q=s_q, seed=51 + s_q)
    inp = W.make_inputs(w, poison=True, extra_pages=4)
    d = to_device(inp)
    p = mla.plan(d["seq_lens"], s_q=s_q, max_pages_per_seq=d["block_table"].shape[1])
    r = mla.parse_plan(mla.plan_device_bytes(p), w.batch, s_q, mla.num_units())
    items_per_unit = np.diff(r["unit_begin"])
    assert items_per_unit.max() >= 3
    _parity_full(w, poison=True, extra_pages=4)


@pytest.mark.parametrize("s_q", [1, 2])
def test_rising_scores_rescale(s_q):
    """Scores that keep rising along each row: each page's k_rope is scaled up with its page
    index (and q_rope by 3), so the running max grows by more than 2^8 again and again and
    the kernel rescales O and the lower P half on many pages.  V (c_kv) is left at N(0, 1),
    so the tolerance still measures the attention, not bf16 rounding of large outputs."""
    lens = [700, 1500, 3000, 64, 130, 2049]
    w = W.custom(lens, s_q=s_q, seed=60 + s_q)
    inp = W.make_inputs(w)
    inp["q_rope"] = (inp["q_rope"].float() * 3).to(torch.bfloat16)
    kv = inp["kv_cache"].float()
    bt = inp["block_table"]
    for b, L in enumerate(lens):
        for pi in range((L + 63) // 64):
            kv[int(bt[b, pi]), :, W.D_LATENT:] *= 1.0 + pi / 4.0
    inp["kv_cache"] = kv.to(torch.bfloat16)
    o, lse, _ = run_gpu(inp)
    o_ref, lse_ref = oracle_full(inp)
    assert_close(o, lse, o_ref, lse_ref, "rising scores")


def test_mtp_small():
    _parity_full(W.custom([2, 64, 65, 1024, 2049, 8192], s_q=2, seed=41), poison=True)


def test_device_plan_matches_host_planner():
    """mla_decode_plan (device) writes the same schedule bytes as the host twin."""
    units = mla.num_units()
    cases = [(W.workload(n).seq_lens, W.workload(n).s_q) for n in
             ("tiny", "uniform", "mtp", "mixed", "long", "long1m")]
    rng = np.random.default_rng(5)
    for _ in range(10):
        B = int(rng.integers(1, 300))
        cases.append((rng.integers(2, 20000, size=B).tolist(), int(rng.integers(1, 3))))
    for lens, s_q in cases:
        mp = max((L + 63) // 64 for L in lens)
        sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
        p = mla.plan(sl, s_q=s_q, max_pages_per_seq=mp)
        dev = mla.parse_plan(mla.plan_device_bytes(p), len(lens), s_q, units)
        host = mla.plan_host(lens, s_q=s_q, max_pages_per_seq=mp, num_units=units)
        assert dev["header"] == host["header"]
        for k in host:
            if k != "header":
                np.testing.assert_array_equal(dev[k], host[k], err_msg=k)


def test_deterministic_and_permutation_invariant():
    """Two runs are bit-identical; moving pages in the pool changes no bit either."""
    w = W.custom([700, 5000, 64, 12000], s_q=1, seed=51)
    inp = W.make_inputs(w, extra_pages=4)
    o1, l1, _ = run_gpu(inp)
    o2, l2, _ = run_gpu(inp)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    P = inp["kv_cache"].shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(7))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    inp2 = dict(inp)
    inp2["kv_cache"] = inp["kv_cache"][perm].contiguous()
    bt = inp["block_table"].clone()
    m = bt >= 0
    bt[m] = inv[bt[m].long()].to(torch.int32)
    inp2["block_table"] = bt
    o3, l3, _ = run_gpu(inp2)
    np.testing.assert_array_equal(o1, o3)
    np.testing.assert_array_equal(l1, l3)


def test_bad_inputs_are_flagged_not_faulted():
    """A block_table entry outside the pool and a too-short seq_len set status bits; rows go NaN."""
    w = W.custom([300, 200, 5], s_q=2, seed=61)
    inp = W.make_inputs(w)
    inp["block_table"][0, 2] = inp["kv_cache"].shape[0] + 1000
    inp["seq_lens"][2] = 1   # < s_q
    o, lse, status = run_gpu(inp, check_status=False)
    assert status & mla.MLA_DEV_BAD_PAGE and status & mla.MLA_DEV_BAD_SEQ_LEN
    assert np.isnan(o[2]).all() and np.isnan(lse[2]).all()
    assert np.isnan(lse[0]).all()
    o_ref, lse_ref = oracle.decode(inp["q_latent"][1:2], inp["q_rope"][1:2], inp["kv_cache"],
                                   inp["block_table"][1:2], inp["seq_lens"][1:2], s_q=2,
                                   scale=W.SCALE)
    assert_close(o[1:2], lse[1:2], o_ref, lse_ref, "good row beside bad ones")


@pytest.mark.parametrize("name,nrows", [("uniform", 96), ("mtp", 160), ("mixed", 96),
                                        ("long", 24), ("long1m", 12)])
def test_full_size_sampled(name, nrows):
    """Full-size workloads in the benchmark's launch configuration, sampled rows vs the oracle."""
    w = W.workload(name)
    inp = W.make_inputs(w)
    o, lse, _ = run_gpu(inp)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = sample_rows(w, nrows, seed=sum(map(ord, name)))
    o_ref, lse_ref = oracle.decode(inp["q_latent"], inp["q_rope"], inp["kv_cache"],
                                   inp["block_table"], inp["seq_lens"], s_q=w.s_q,
                                   scale=W.SCALE, rows=rows)
    b, t, h = rows[:, 0], rows[:, 1], rows[:, 2]
    assert_close(o[b, t, h], lse[b, t, h], o_ref, lse_ref, name)
