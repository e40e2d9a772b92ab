"""The step after attention (W_UV per head, o_proj) vs the fp64 oracle, on cuda:0; and the whole
absorbed layer (prolog, decode, W_UV) on the GPU against plain unabsorbed multi-head attention.

Element bounds come from the arithmetic: one bf16 rounding of the output (2^-8 relative) plus
the worst-case fp32 summation error of a K-term dot product, K * 2^-24 * sum |a_k b_k|.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import epilog as E
from oracle import prolog as OP

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import mla_decode_attention_02_gb300 as mla  # noqa: E402

REL = 2.0 ** -8


def _np(t):
    return t.float().cpu().double().numpy()


def _within(gpu, ref, absdot, k, what):
    err = np.abs(gpu - ref)
    bound = REL * np.abs(ref) + k * 2.0 ** -24 * absdot + 1e-6
    bad = err > bound
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside the bound, worst err {err.max():.3e}"


@pytest.mark.parametrize("batch,s_q", [(1, 1), (64, 1), (65, 2), (128, 2), (3, 2), (129, 1), (150, 2)])
def test_uv_parity(batch, s_q):
    """Token counts below, at and above one 128-token tile, ragged last tiles included
    (129 tokens: a one-token tile; 300 tokens: three tiles)."""
    T = batch * s_q
    e = W.epilog_tensors(T, seed=T)
    o_lat = e["o_latent"].view(batch, s_q, 128, 512).cuda()
    o_v, st = mla.epilog_uv(o_lat, e["w_uv"].cuda())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = E.uv_project(e["o_latent"], e["w_uv"])
    absdot = E.uv_project(np.abs(_np(e["o_latent"])), np.abs(_np(e["w_uv"])))
    _within(_np(o_v).reshape(T, 128, 128), ref, absdot, 512, f"o_v T={T}")


@pytest.mark.parametrize("tokens,hidden", [(64, 7168), (5, 1024), (256, 7168)])
def test_oproj_parity(tokens, hidden):
    e = W.epilog_tensors(tokens, seed=100 + tokens, hidden=hidden)
    o_v = (e["o_latent"][:, :, :128].contiguous())          # any bf16 [T][128][128] input
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mla.epilog_oproj(o_v.cuda(), e["w_o"].cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = E.o_project(o_v, e["w_o"])
    absdot = E.o_project(np.abs(_np(o_v)), np.abs(_np(e["w_o"])))
    _within(_np(out), ref, absdot, 128 * 128, f"out T={tokens} hidden={hidden}")


@pytest.mark.parametrize("tokens,hidden", [(8, 512), (300, 1000), (129, 136)])
def test_oproj_ragged_shapes(tokens, hidden):
    """Token counts past one 256-token tile and hidden sizes that end inside a 128-output
    tile: the rows past the ends read zeros and are not stored."""
    e = W.epilog_tensors(tokens, seed=7 + tokens, hidden=hidden)
    o_v = e["o_latent"][:, :, :128].contiguous()
    guard = torch.full((tokens + 2, hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = guard[:tokens]
    mla.epilog_oproj(o_v.cuda(), e["w_o"].cuda(), out=out)
    torch.cuda.synchronize()
    assert torch.isnan(guard[tokens:]).all()            # nothing past the last token row
    ref = E.o_project(o_v, e["w_o"])
    absdot = E.o_project(np.abs(_np(o_v)), np.abs(_np(e["w_o"])))
    _within(_np(out), ref, absdot, 128 * 128, f"out T={tokens} hidden={hidden}")


def test_oproj_deterministic():
    e = W.epilog_tensors(256, seed=9, hidden=7168)
    o_v = e["o_latent"][:, :, :128].contiguous().cuda()
    w_o = e["w_o"].cuda()
    a = mla.epilog_oproj(o_v, w_o)
    b = mla.epilog_oproj(o_v, w_o)
    assert torch.equal(a, b)


@pytest.mark.parametrize("s_q", [1, 2])
def test_absorbed_layer_on_gpu_equals_unabsorbed_attention(s_q):
    """GPU prolog -> decode -> W_UV vs fp64 plain multi-head attention with 192-value keys.

    The oracle side gets the raw inputs and the oracle's own rotated q_rope and cache rows; the
    bar is the decode bar (max |err| <= 2e-2, mean <= 2e-3): o_v has o_latent's scale.
    """
    lens = [1 + s_q, 64, 65, 300, 700]
    B = len(lens)
    w = W.custom(lens, s_q=s_q, seed=70 + s_q)
    inp = W.make_inputs(w, extra_pages=1)
    t = W.prolog_tensors(B, s_q, seed=80 + s_q)
    wv = W.epilog_tensors(1, seed=90 + s_q)["w_uv"]
    d = {k: v.cuda() for k, v in {**t, "kv_cache": inp["kv_cache"], "block_table": inp["block_table"],
                                  "seq_lens": inp["seq_lens"], "w_uv": wv}.items()}
    ql, qr, st = mla.prolog(d["q_nope"], d["q_pe"], d["kv_latent"], d["k_pe"], d["w_uk"], d["kv_norm_weight"],
                            d["kv_cache"], d["block_table"], d["seq_lens"])
    p = mla.plan(d["seq_lens"], s_q=s_q, max_pages_per_seq=d["block_table"].shape[1])
    o, _ = mla.decode(p, ql, qr, d["kv_cache"], d["block_table"], scale=W.SCALE)
    o_v, st2 = mla.epilog_uv(o, d["w_uv"])
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0 and mla.check(p) == 0
    _, qr_ref, cache_ref = OP.prolog(t["q_nope"], t["q_pe"], t["kv_latent"], t["k_pe"], t["w_uk"],
                                     t["kv_norm_weight"], inp["kv_cache"], inp["block_table"], inp["seq_lens"])
    bt = inp["block_table"].numpy()
    got = _np(o_v)
    errs = []
    for b, L in enumerate(lens):
        rows = np.stack([cache_ref[bt[b, j // W.PAGE], j % W.PAGE] for j in range(L)])
        for tq in range(s_q):
            vis = L - s_q + 1 + tq
            ref = E.unabsorbed_attention(t["q_nope"][b, tq], qr_ref[b, tq], rows[:vis, :512], rows[:vis, 512:],
                                         t["w_uk"], wv, W.SCALE)
            errs.append(np.abs(got[b, tq] - ref))
    err = np.stack(errs)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())


@pytest.mark.parametrize("name", ["uniform", "mtp"])
def test_epilog_parity_bench_configuration(name):
    """The inputs bench.py --stage epilog times (same workload and seeds), every element of both steps."""
    w = W.workload(name)
    T = w.batch * w.s_q
    e = W.epilog_tensors(T, w.seed)
    o_v, st = mla.epilog_uv(e["o_latent"].view(w.batch, w.s_q, 128, 512).cuda(), e["w_uv"].cuda())
    out = mla.epilog_oproj(o_v, e["w_o"].cuda())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_v = E.uv_project(e["o_latent"], e["w_uv"])
    _within(_np(o_v).reshape(T, 128, 128), ref_v,
            E.uv_project(np.abs(_np(e["o_latent"])), np.abs(_np(e["w_uv"]))), 512, f"o_v {name}")
    # o_proj against the oracle's own chain (its fp64 o_v, never the GPU's): the bound adds to
    # out's rounding and summation terms the GPU o_v's allowed error carried through |W_O|
    absdot_v = E.uv_project(np.abs(_np(e["o_latent"])), np.abs(_np(e["w_uv"])))
    bound_v = REL * np.abs(ref_v) + 512 * 2.0 ** -24 * absdot_v + 1e-6
    w_abs = np.abs(_np(e["w_o"]))
    ref_o = E.o_project(ref_v, e["w_o"])
    bound_o = (REL * np.abs(ref_o) + 128 * 128 * 2.0 ** -24 * E.o_project(np.abs(ref_v) + bound_v, w_abs)
               + E.o_project(bound_v, w_abs) + 1e-6)
    err = np.abs(_np(out) - ref_o)
    assert np.isfinite(_np(out)).all() and not (err > bound_o).any(), \
        f"out {name}: {(err > bound_o).sum()} outside the bound, worst err {err.max():.3e}"
