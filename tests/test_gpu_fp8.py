"""The fp8 cache quantiser on cuda:0 vs the oracle: every byte identical (codes are integers decided
in fp32 on both sides; the scale and k_rope / s are correctly rounded fp32 quotients, the latter then
rounded to bf16 to nearest even on both sides)."""

import numpy as np
import pytest
import torch

from oracle import fp8 as F

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import mla_decode_attention_02_gb300 as mla  # noqa: E402


def _cache(pages, seed):
    g = torch.Generator().manual_seed(seed)
    kv = torch.randn(pages, 64, 576, generator=g)
    rows = kv.view(-1, 576)
    # rows across magnitudes (subnormal codes, large values), an all-zero latent, a one-hot row
    rows[:16] *= 1e-4
    rows[16:32] *= 300.0
    rows[40, :512] = 0.0
    rows[41, :512] = 0.0
    rows[41, 77] = -5.0
    return kv.to(torch.bfloat16)


@pytest.mark.parametrize("pages,seed", [(1, 1), (7, 2), (300, 3)])
def test_quantize_bit_exact(pages, seed):
    kv = _cache(pages, seed)
    got = mla.quantize_cache_fp8(kv.cuda()).cpu().numpy()
    ref = F.quantize_cache(kv)
    diff = got != ref
    assert not diff.any(), f"{diff.sum()} bytes differ, first at {np.argwhere(diff)[:3].tolist()}"


def test_quantize_ragged_row_count():
    """A row count that is not a multiple of the kernel's rows per CTA."""
    kv = _cache(1, 4).reshape(64, 576)[:13].contiguous()
    got = mla.quantize_cache_fp8(kv.cuda()).cpu().numpy()
    np.testing.assert_array_equal(got, F.quantize_cache(kv))
