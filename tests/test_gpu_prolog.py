"""The prolog kernel (absorbed q, RoPE, RMSNorm, paged append) vs the fp64 oracle, on cuda:0.

Tolerances come from the arithmetic: every output is one bf16 rounding
(relative half-ulp 2^-8) of an fp32 result whose own error is far below it
(128-term fp32 sums of exact bf16 products; fp32 sin/cos of an angle reduced
in fp64; an fp32 sum of squares), so each element must satisfy
|gpu - oracle| <= 2^-8 |oracle| + 1e-4.  Cache rows the step does not own
must come back bit-identical.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close
from oracle import prolog as OP

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import mla_decode_attention_02_gb300 as mla  # noqa: E402

REL = 2.0 ** -8
ABS = 1e-4
BASE = 10000.0
EPS = 1e-6


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


def _close(gpu, ref, what):
    g = gpu.float().cpu().double().numpy() if isinstance(gpu, torch.Tensor) else gpu
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bound = REL * np.abs(ref) + ABS
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside 2^-8|ref| + 1e-4, "
                           f"worst err {err.max():.3e}")
    return err.max()


def _run(t, c, base=BASE, eps=EPS):
    d = {k: v.cuda() for k, v in {**t, **c}.items()}
    cache = d["kv_cache"]
    ql, qr, st = mla.prolog(d["q_nope"], d["q_pe"], d["kv_latent"], d["k_pe"], d["w_uk"],
                            d["kv_norm_weight"], cache, d["block_table"], d["seq_lens"],
                            rope_base=base, rms_eps=eps)
    torch.cuda.synchronize()
    return ql, qr, cache, int(st.item())


def _check_all(t, c, s_q, base=BASE, eps=EPS):
    ql, qr, cache, st = _run(t, c, base, eps)
    assert st == 0, f"device status {st:#x}"
    ql_ref, qr_ref, cache_ref = OP.prolog(t["q_nope"], t["q_pe"], t["kv_latent"], t["k_pe"], t["w_uk"],
                                          t["kv_norm_weight"], c["kv_cache"], c["block_table"],
                                          c["seq_lens"], rope_base=base, rms_eps=eps)
    _close(ql, ql_ref, "q_latent")
    _close(qr, qr_ref, "q_rope")
    pos = OP.positions(c["seq_lens"].numpy(), s_q)
    owned = np.zeros(c["kv_cache"].shape[:2], dtype=bool)
    bt = c["block_table"].numpy()
    for b in range(pos.shape[0]):
        for j in range(s_q):
            owned[bt[b, pos[b, j] // W.PAGE], pos[b, j] % W.PAGE] = True
    got = cache.cpu()
    np.testing.assert_array_equal(_bits(got)[~owned], _bits(c["kv_cache"])[~owned])
    _close(got.double().numpy()[owned], cache_ref[owned], "appended rows")


@pytest.mark.parametrize("lens,s_q", [
    ([1], 1),                                   # one token at position 0
    ([2, 64, 65], 2),                           # pos 0, a page's last slot, a page boundary between t
    ([5, 130, 4096] * 43 + [77], 1),            # 130 tokens: two token tiles, ragged tail
    ([64 * k + 1 for k in range(1, 65)], 2),    # 128 tokens, one full tile, each straddles a page
    ([1000003, 262144, 524289], 2),             # positions past half a million (angle reduction)
])
def test_prolog_parity(lens, s_q):
    t = W.prolog_tensors(len(lens), s_q, seed=len(lens) * 7 + s_q)
    c = W.sparse_cache(lens, s_q, seed=len(lens) + s_q)
    _check_all(t, c, s_q)


def test_prolog_parity_three_token_tiles_other_constants():
    """300 tokens (three token tiles, last one 44 rows), a different RoPE base and eps."""
    rng = np.random.default_rng(9)
    lens = rng.integers(2, 40000, size=150).tolist()
    t = W.prolog_tensors(150, 2, seed=31)
    c = W.sparse_cache(lens, 2, seed=32)
    _check_all(t, c, 2, base=50000.0, eps=1e-5)


def test_prolog_bad_slots_flagged_and_skipped():
    """seq_len < s_q and a page outside the pool: status bits, NaN q_rope, no cache write."""
    lens = [300, 1, 641]
    t = W.prolog_tensors(3, 2, seed=41)
    c = W.sparse_cache(lens, 2, seed=42)
    pool = c["kv_cache"].shape[0]
    c["block_table"][2, 640 // W.PAGE] = pool + 5          # request 2's second slot: page outside the pool
    before = c["kv_cache"].clone()
    ql, qr, cache, st = _run(t, c)
    assert st & mla.MLA_DEV_BAD_SEQ_LEN and st & mla.MLA_DEV_BAD_PAGE
    qrn = qr.float().cpu().numpy()
    assert np.isnan(qrn[1, 0]).all()                       # request 1, token 0: position -1
    # every token with a position is rotated, the bad-page one included
    pos = OP.positions(np.array(lens), 2)
    for b, j in [(0, 0), (0, 1), (1, 1), (2, 0), (2, 1)]:
        _close(qr[b, j], OP.rope(t["q_pe"][b, j], pos[b, j], BASE), f"q_rope of token ({b}, {j})")
    _close(ql, OP.absorb_q(t["q_nope"].reshape(6, 128, 128), t["w_uk"]).reshape(3, 2, 128, 512),
           "q_latent")
    got = cache.cpu()
    bt = c["block_table"].numpy()
    valid = [(0, 0), (0, 1), (1, 1), (2, 0)]
    owned = np.zeros(got.shape[:2], dtype=bool)
    for b, j in valid:
        owned[bt[b, pos[b, j] // W.PAGE], pos[b, j] % W.PAGE] = True
    np.testing.assert_array_equal(_bits(got)[~owned], _bits(before)[~owned])


@pytest.mark.parametrize("s_q", [1, 2])
def test_prolog_then_decode(s_q):
    """The prolog's outputs feed decode: same result as the oracle's prolog fed to the oracle's decode.

    The oracle side rounds its fp64 prolog outputs to bf16 (the dtype decode reads).
    """
    lens = [1 + s_q, 63, 64, 65, 500, 2049]
    w = W.custom(lens, s_q=s_q, seed=50 + s_q)
    inp = W.make_inputs(w, extra_pages=2)
    t = W.prolog_tensors(len(lens), s_q, seed=60 + s_q)
    c = {k: inp[k] for k in ("kv_cache", "block_table", "seq_lens")}
    ql, qr, cache, st = _run(t, c)
    assert st == 0
    p = mla.plan(c["seq_lens"].cuda(), s_q=s_q, max_pages_per_seq=c["block_table"].shape[1])
    o, lse = mla.decode(p, ql, qr, cache, c["block_table"].cuda(), scale=W.SCALE)
    assert mla.check(p) == 0
    ql_ref, qr_ref, cache_ref = OP.prolog(t["q_nope"], t["q_pe"], t["kv_latent"], t["k_pe"], t["w_uk"],
                                          t["kv_norm_weight"], c["kv_cache"], c["block_table"],
                                          c["seq_lens"], rope_base=BASE, rms_eps=EPS)
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)   # noqa: E731
    o_ref, lse_ref = oracle.decode(bf(ql_ref), bf(qr_ref), bf(cache_ref), c["block_table"],
                                   c["seq_lens"], s_q=s_q, scale=W.SCALE)
    assert_close(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
                 f"prolog+decode s_q={s_q}")


@pytest.mark.parametrize("base", [10000.0, 50000.0, 1e6])
def test_rope_table(base):
    """hi + lo of the device table carries base^(-2i/64) / (2 pi) to about 2^-48 relative."""
    table = mla.rope_table(base).cpu().double().numpy()
    g = table[:32] + table[32:]
    ref = OP.rope_angles(np.array(1), 64, base) / (2 * np.pi)
    np.testing.assert_allclose(g, ref, rtol=2.0 ** -46, atol=0)
    assert np.all(np.abs(table[32:]) <= np.abs(table[:32]) * 2.0 ** -24)


@pytest.mark.parametrize("name", ["uniform", "mtp"])
def test_prolog_parity_bench_configuration(name):
    """The inputs bench.py --stage prolog times (same workload, seeds and table), every element."""
    w = W.workload(name)
    t = W.prolog_tensors(w.batch, w.s_q, w.seed)
    c = W.sparse_cache(w.seq_lens, w.s_q, w.seed)
    _check_all(t, c, w.s_q, base=W.ROPE_BASE, eps=W.RMS_EPS)
