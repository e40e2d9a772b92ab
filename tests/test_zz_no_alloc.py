"""The allocation-free entry point (mla_decode_noalloc) against the regular one.

mla_decode_noalloc serves callers that cannot allocate device memory on
their decode path: it keeps its workspace in a fixed 64 MiB device array
inside the library instead of a caller-allocated buffer.  This file is
collected last so that a failure here does not hide any other test.  It
must pass alone in a fresh process and after the rest of the suite.
"""

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import assert_close, oracle_full, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import mla_decode_attention_02_gb300 as mla  # noqa: E402


def _regular(d):
    p = mla.plan(d["seq_lens"], s_q=d["s_q"], max_pages_per_seq=d["block_table"].shape[1])
    o, lse = mla.decode(p, d["q_latent"], d["q_rope"], d["kv_cache"], d["block_table"],
                        scale=d["scale"])
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _noalloc(d):
    o, lse = mla.decode_noalloc(d["q_latent"], d["q_rope"], d["kv_cache"], d["block_table"],
                                d["seq_lens"], s_q=d["s_q"], scale=d["scale"])
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _identical(a, b):
    (o1, l1), (o2, l2) = a, b
    assert np.isfinite(o2).all() and np.isfinite(l2).all()
    # the same schedule runs through the same kernels: bit for bit equal
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_noalloc_matches_regular_entry_point_twice():
    """Two calls in a row with different batches; each is bit-identical to plan + decode
    (same schedule, same kernels), and the second is also checked against the oracle."""
    cases = [W.custom([1, 63, 64, 200, 3000, 9000], s_q=1, seed=71),
             W.custom([2, 130, 700, 2000], s_q=2, seed=72)]
    for i, w in enumerate(cases):
        inp = W.make_inputs(w, poison=True)
        d = to_device(inp)
        na = _noalloc(d)
        _identical(_regular(d), na)
        if i == 1:
            o_ref, lse_ref = oracle_full(inp)
            assert_close(na[0].astype(np.float64), na[1].astype(np.float64), o_ref, lse_ref, "noalloc")


def test_noalloc_rejects_oversized_problem():
    """A workspace larger than the fixed array is refused before anything runs."""
    need = mla.workspace_size(4096, 2, 1)
    assert need > mla.NOALLOC_SCRATCH_BYTES
    d = to_device(W.make_inputs(W.custom([2] * 4096, s_q=2, seed=73)))
    with pytest.raises(mla.MLAError) as e:
        mla.decode_noalloc(d["q_latent"], d["q_rope"], d["kv_cache"], d["block_table"],
                           d["seq_lens"], s_q=2, scale=d["scale"])
    assert e.value.status == 3
