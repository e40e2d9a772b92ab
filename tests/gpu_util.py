"""Helpers shared by the GPU tests: run the CUDA path through the binding, compare with the oracle."""

import numpy as np
import torch

import mla_decode_attention_02_gb300 as mla
import oracle
import workloads as W

# Acceptance bar: max |err| <= 2e-2 and mean |err| <= 2e-3 on o_latent, |err| <= 1e-3 on lse.
O_MAX_ERR = 2e-2
O_MEAN_ERR = 2e-3
LSE_MAX_ERR = 1e-3


def to_device(inp, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_gpu(inp, *, max_pages=None, check_status=True, pow2_max=False):
    """Plan + decode on cuda:0 through the C ABI; returns (o fp64 numpy, lse fp64 numpy, status)."""
    d = to_device(inp)
    mp = d["block_table"].shape[1] if max_pages is None else max_pages
    p = mla.plan(d["seq_lens"], s_q=d["s_q"], max_pages_per_seq=mp)
    o, lse = mla.decode(p, d["q_latent"], d["q_rope"], d["kv_cache"], d["block_table"],
                        scale=d["scale"], pow2_max=pow2_max)
    status = mla.check(p)
    if check_status:
        assert status == 0, f"device status {status:#x}"
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy(), status


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    err = np.abs(o_gpu - o_ref)
    lerr = np.abs(lse_gpu - lse_ref)
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), f"{what}: non-finite output"
    assert err.max() <= O_MAX_ERR, f"{what}: o max err {err.max():.3e}"
    assert err.mean() <= O_MEAN_ERR, f"{what}: o mean err {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX_ERR, f"{what}: lse max err {lerr.max():.3e}"
    return err.max(), err.mean(), lerr.max()


def oracle_full(inp):
    return oracle.decode(inp["q_latent"], inp["q_rope"], inp["kv_cache"], inp["block_table"],
                         inp["seq_lens"], s_q=inp["s_q"], scale=inp["scale"])


def sample_rows(w, n, seed=0):
    """n (b, t, h) rows spread over requests, query tokens and heads."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(min(w.batch, n)):   # every request at least once, then random
        rows.add((b, int(rng.integers(0, w.s_q)), int(rng.integers(0, W.NUM_HEADS))))
    while len(rows) < n:
        rows.add((int(rng.integers(0, w.batch)), int(rng.integers(0, w.s_q)),
                  int(rng.integers(0, W.NUM_HEADS))))
    return np.array(sorted(rows), dtype=np.int32)
