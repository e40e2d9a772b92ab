"""The main kernel's time-out path, run without a GPU fault.

mla_decode_diag lowers the limit of the kernel's bounded waits and can
withhold one K-stage load of one work unit, so that the waits for it run out:
the kernel must record MLA_DEV_TIMEOUT, wind down and return (no hang, no
fault), and the next ordinary call on the same context must be exact.
"""

import time

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import assert_close, oracle_full, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import mla_decode_attention_02_gb300 as mla  # noqa: E402

LIMIT_NS = 20_000_000   # 20 ms per wait


def _first_unit_pages(p, w):
    """Pages of the unit that runs the schedule's first item (the one the stall targets)."""
    r = mla.parse_plan(mla.plan_device_bytes(p), w.batch, w.s_q, mla.num_units())
    ub = r["unit_begin"]
    u = int(np.nonzero((ub[:-1] == 0) & (ub[1:] > 0))[0][0])
    items = r["items"][ub[u]:ub[u + 1]]
    return int(sum((e - b + 63) // 64 for _, b, e, _ in items))


def test_injected_stall_times_out_and_the_next_call_is_exact():
    w = W.custom([4096] * 6, s_q=1, seed=71)
    inp = W.make_inputs(w)
    d = to_device(inp)
    mp = d["block_table"].shape[1]
    p = mla.plan(d["seq_lens"], s_q=1, max_pages_per_seq=mp)
    assert _first_unit_pages(p, w) >= 2, "the stalled unit must own a second page"
    args = (d["q_latent"], d["q_rope"], d["kv_cache"], d["block_table"])

    t0 = time.monotonic()
    mla.decode_diag(p, *args, scale=d["scale"], wait_limit_ns=LIMIT_NS,
                    inject=mla.MLA_INJECT_WITHHOLD_K_LOAD)
    status = mla.check(p)   # synchronises: the kernel has returned
    elapsed = time.monotonic() - t0
    assert status & mla.MLA_DEV_TIMEOUT, f"device status {status:#x}"
    assert status & ~mla.MLA_DEV_TIMEOUT == 0, f"device status {status:#x}"
    # a CTA gives up after one limit; the pair's teardown waits at most a few more
    assert elapsed < 2.0, f"time-out path took {elapsed:.3f} s"

    # the context is usable and the next plan + decode (same workspace) is exact
    p = mla.plan(d["seq_lens"], s_q=1, max_pages_per_seq=mp, workspace=p.workspace)
    o, lse = mla.decode(p, *args, scale=d["scale"])
    assert mla.check(p) == 0
    o_ref, lse_ref = oracle_full(inp)
    assert_close(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
                 "after a time-out")

    # without injection the diagnostic entry point is mla_decode, bit for bit
    o2, lse2 = mla.decode_diag(p, *args, scale=d["scale"], wait_limit_ns=2 * 10**9, inject=0)
    assert mla.check(p) == 0
    assert torch.equal(o2, o) and torch.equal(lse2, lse)


def test_short_limit_without_stall_is_exact():
    """A limit of a few milliseconds is far above any wait of a healthy run."""
    w = W.custom([3001, 64, 700], s_q=2, seed=72)
    inp = W.make_inputs(w)
    d = to_device(inp)
    p = mla.plan(d["seq_lens"], s_q=2, max_pages_per_seq=d["block_table"].shape[1])
    o, lse = mla.decode_diag(p, d["q_latent"], d["q_rope"], d["kv_cache"], d["block_table"],
                             scale=d["scale"], wait_limit_ns=5_000_000)
    assert mla.check(p) == 0
    o_ref, lse_ref = oracle_full(inp)
    assert_close(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
                 "5 ms limit")
    assert np.isfinite(lse.cpu().numpy()).all()
