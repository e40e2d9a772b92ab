"""Pins for the fp8 (e4m3) cache oracle: torch's own float8_e4m3fn conversion, the code table,
round trips and the row layout."""

import numpy as np
import pytest
import torch

from oracle import fp8 as F


def test_code_table():
    codes = np.arange(256, dtype=np.uint8)
    v = F.e4m3_value(codes)
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6 and v[0x38] == 1.0
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                      # codes 0..126 increase strictly
    np.testing.assert_array_equal(v[0x80:0xFF], -pos[:0x7F])
    # every finite code is its own nearest value
    fin = codes[~np.isnan(v)]
    np.testing.assert_array_equal(F.e4m3_encode(F.e4m3_value(fin).astype(np.float32)) & 0x7F, fin & 0x7F)


def test_encode_matches_torch_float8_e4m3fn():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(200000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = np.clip(x, -448, 448).astype(np.float32)
    # ties and binade edges: exact midpoints between neighbouring codes, and the codes themselves
    vals = F.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, vals.astype(np.float32), np.float32([0.0, 2.0 ** -10, 3 * 2.0 ** -10])])
    ours = F.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    zero = x == 0
    np.testing.assert_array_equal(ours[~zero], ref[~zero])
    np.testing.assert_array_equal(ours[zero] & 0x7F, ref[zero] & 0x7F)


def test_round_trip_error_is_half_a_step():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(100000) * 60).clip(-448, 448).astype(np.float32)
    back = F.e4m3_value(F.e4m3_encode(x))
    a = np.abs(x.astype(np.float64))
    step = np.exp2(np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6) - 3)
    assert np.all(np.abs(back - x) <= step / 2 + 1e-30)


def test_quantize_cache_layout_and_scale():
    g = torch.Generator().manual_seed(3)
    kv = torch.randn(3, 64, 576, generator=g).to(torch.bfloat16)
    kv[1, 5, :512] = 0                                   # an all-zero latent: scale 1, codes 0
    q = F.quantize_cache(kv)
    assert q.shape == (3, 64, 656) and np.all(q[..., 644:] == 0)
    rows = q.reshape(-1, 656)
    s = rows[:, 640:644].copy().view("<f4").reshape(-1)
    lat = kv.reshape(-1, 576)[:, :512].float().numpy()
    amax = np.abs(lat).max(1)
    np.testing.assert_array_equal(s[amax > 0], (amax[amax > 0] / np.float32(448)).astype(np.float32))
    assert s[1 * 64 + 5] == 1.0 and np.all(rows[1 * 64 + 5, :512] == 0)
    # the largest value of each row lands on the largest code; k_rope is stored divided by s
    # (correctly rounded fp32 quotient, then bf16 round to nearest even: checked bit by bit
    # against an integer rounding of the fp32 bits)
    top = np.abs(lat).argmax(1)
    assert np.all(rows[np.arange(rows.shape[0]), top][amax > 0] & 0x7F == 0x7E)
    rope = kv.reshape(-1, 576)[:, 512:].float().numpy()
    qbits = (rope / s[:, None]).astype(np.float32).view(np.uint32).astype(np.uint64)
    rne = ((qbits + 0x7FFF + ((qbits >> 16) & 1)) >> 16).astype(np.uint16)
    np.testing.assert_array_equal(rows[:, 512:640].copy().view("<u2"), rne)
    deq = F.dequantize_cache(q)
    ropeq = (rne.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(deq.reshape(-1, 576)[:, 512:], ropeq * s[:, None].astype(np.float64))
    assert np.all(deq.reshape(-1, 576)[1 * 64 + 5, 512:] == rope[1 * 64 + 5])   # s = 1: k_rope unchanged
    rrel = np.abs(deq.reshape(-1, 576)[:, 512:] - rope) / np.maximum(np.abs(rope), 1e-30)
    assert rrel[rope != 0].max() <= 2.0 ** -8 * (1 + 1e-6)  # bf16 rounding of the quotient and fp32 division
    ref = kv[..., :512].double().numpy()
    err = np.abs(deq[..., :512] - ref)
    assert np.all(err[1, 5] == 0)
    rng_ = np.abs(ref).max(-1, keepdims=True)
    rel = err / np.where(rng_ > 0, rng_, 1.0)
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)             # at most half an e4m3 step: 2^-4 of the row's max


def test_decode_over_exact_fp8_cache_equals_bf16_decode():
    """A cache whose latent values are e4m3 values times a power-of-two scale survives
    quantisation unchanged, so the fp8 decode must equal the bf16 decode exactly."""
    import oracle
    import workloads as W
    w = W.custom([5, 64, 130], s_q=2, seed=9)
    inp = W.make_inputs(w)
    g = np.random.default_rng(9)
    codes = g.integers(0, 0x7F, size=inp["kv_cache"].shape[:-1] + (512,), dtype=np.int64)   # finite codes
    vals = F.e4m3_value(codes.astype(np.uint8)) * np.where(g.random(codes.shape) < 0.5, -1, 1)
    # each row's largest magnitude must be 448 so that its scale is exactly 1 (then every value is kept)
    vals[..., 0] = 448.0
    kv = inp["kv_cache"].clone()
    kv[..., :512] = torch.from_numpy(vals).to(torch.bfloat16)       # e4m3 values are exact in bf16
    assert np.array_equal(kv[..., :512].double().numpy(), vals)
    q8 = F.quantize_cache(kv)
    o8, l8 = F.decode(inp["q_latent"], inp["q_rope"], q8, inp["block_table"], inp["seq_lens"], s_q=2,
                      scale=inp["scale"])
    ob, lb = oracle.decode(inp["q_latent"], inp["q_rope"], kv, inp["block_table"], inp["seq_lens"], s_q=2,
                           scale=inp["scale"])
    np.testing.assert_array_equal(o8, ob)
    np.testing.assert_array_equal(l8, lb)
