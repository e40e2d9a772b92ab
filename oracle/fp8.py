"""fp64/fp32 oracle of an fp8 (e4m3) latent cache (test infrastructure only).

Only the test suite and ``bench.py``'s CPU legs may import this module.

What it computes: the low-bit KV cache the Ascend best-practice page lists as
next work ("Huawei Ascend servers: DeepSeek V3/R1 inference best practice",
section 8: KV-cache-only quantisation of the attention and MLAProlog
operators), in the form this hardware has native arithmetic for: each cached
row's 512 c_kv values stored as e4m3 codes of c_kv / s with one fp32 scale per
token, s = max |c_kv| / 448 (448 is e4m3's largest finite value; s = 1 for an
all-zero row), and the 64 k_rope values divided by the same s and kept in
bf16, so that the whole row dequantises by one factor.

Row layout (656 bytes, a multiple of 16): bytes [0, 512) the codes,
[512, 640) k_rope / s (bf16: the correctly rounded fp32 quotient rounded to
nearest even), [640, 644) s (fp32, little-endian), [644, 656) zero.

The codes are decided in fp32, the precision the GPU decides them in: s is the
correctly rounded fp32 quotient of fp32(max |c_kv|) by 448, each value's
quotient by s is the correctly rounded fp32 division, and that fp32 value is
rounded to the nearest e4m3 value (ties to even; e4m3: 1 sign, 4 exponent
bits biased by 7, 3 mantissa bits, subnormal step 2^-9, no infinities).

Pins: ``tests/test_fp8_pins.py`` (torch's own float8_e4m3fn conversion, the
code table, round trips).
"""

from __future__ import annotations

import numpy as np

ROW_BYTES = 656
E4M3_MAX = 448.0


def e4m3_value(code) -> np.ndarray:
    """The value of each e4m3 code (uint8); 0x7F / 0xFF are NaN."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3 code of each fp32 value (ties to even), finite values only, |x| <= 464."""
    v = np.asarray(x, dtype=np.float32).astype(np.float64)   # exact
    if np.any(~np.isfinite(v)) or np.any(np.abs(v) >= 464.0):
        raise ValueError("e4m3_encode: value outside the finite e4m3 range")
    sign = (np.signbit(v)).astype(np.int64) << 7
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0))).astype(np.int64)
    e = np.maximum(e, -6)                                     # below 2^-6: subnormal spacing
    step = np.exp2(e - 3.0)
    k = np.rint(a / step).astype(np.int64)                    # a / step is exact; rint: ties to even
    # k counts steps of 2^(e-3): 8..16 in a normal binade (16 carries into the next one),
    # 0..8 below 2^-6 (8 is the smallest normal)
    out = np.empty(a.shape, dtype=np.int64)
    sub = (e == -6) & (k < 8)
    out[sub] = k[sub]                                         # subnormal: exponent field 0
    norm = ~sub
    kk = k[norm]
    ee = e[norm] + (kk == 16)                                 # rounding up to the next power of two
    mm = np.where(kk == 16, 0, kk - 8)
    out[norm] = ((ee + 7) << 3) | mm
    out[a == 0] = 0
    return (out | sign).astype(np.uint8)


def quantize_rows(kv_bf16):
    """Codes [R][512] uint8 and scales [R] fp32 of bf16 cache rows [..][576] (see the module notes)."""
    import torch
    x = kv_bf16.detach().cpu().reshape(-1, kv_bf16.shape[-1])[:, :512].to(torch.float32).numpy()
    amax = np.max(np.abs(x), axis=1).astype(np.float32)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (x / s[:, None]).astype(np.float32)                   # correctly rounded fp32 quotients
    return e4m3_encode(y), s


def quantize_cache(kv_bf16) -> np.ndarray:
    """The fp8 cache, uint8 [..][656], of a bf16 cache [..][576]."""
    import torch
    lead = tuple(kv_bf16.shape[:-1])
    codes, s = quantize_rows(kv_bf16)
    R = codes.shape[0]
    out = np.zeros((R, ROW_BYTES), dtype=np.uint8)
    out[:, :512] = codes
    rope = kv_bf16.detach().cpu().reshape(R, -1)[:, 512:].to(torch.float32).numpy()
    rope_s = (rope / s[:, None]).astype(np.float32)           # correctly rounded fp32 quotients
    rope_b = torch.from_numpy(rope_s).to(torch.bfloat16)      # round to nearest even
    out[:, 512:640] = rope_b.contiguous().view(torch.int16).numpy().view(np.uint8).reshape(R, 128)
    out[:, 640:644] = s.astype("<f4").view(np.uint8).reshape(R, 4)
    return out.reshape(lead + (ROW_BYTES,))


def dequantize_cache(fp8_cache) -> np.ndarray:
    """fp64 [..][576] rows of an fp8 cache: (codes, then the bf16 k_rope / s) x scale."""
    c = np.asarray(fp8_cache, dtype=np.uint8)
    lead = c.shape[:-1]
    c = c.reshape(-1, ROW_BYTES)
    s = c[:, 640:644].copy().view("<f4").reshape(-1).astype(np.float64)
    lat = e4m3_value(c[:, :512]) * s[:, None]
    rope_bits = c[:, 512:640].copy().view("<u2").astype(np.uint32) << 16
    rope = rope_bits.view(np.float32).astype(np.float64) * s[:, None]
    return np.concatenate([lat, rope], axis=1).reshape(lead + (576,))


def decode(q_latent, q_rope, fp8_cache, block_table, seq_lens, *, s_q: int, scale: float, rows=None,
           threads=None):
    """fp64 decode over an fp8 cache: the attention of ``oracle.decode`` on the dequantised rows.

    This is what a kernel reading the fp8 cache computes up to its own rounding; the gap to the
    bf16 cache's result is the quantisation error, reported separately.
    """
    import torch

    import oracle
    rows64 = torch.from_numpy(dequantize_cache(fp8_cache))
    qd = lambda x: x.double() if isinstance(x, torch.Tensor) else torch.from_numpy(np.asarray(x, np.float64))  # noqa: E731
    return oracle.decode(qd(q_latent), qd(q_rope), rows64, block_table, seq_lens, s_q=s_q, scale=scale,
                         rows=rows, threads=threads)
