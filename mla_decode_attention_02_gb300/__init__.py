"""GB300 (sm_103a) weight-absorbed MLA decode over a paged 576-d latent cache.

The computation runs in hand-written CUDA kernels behind the C ABI in
``include/mla_decode.h`` (``libmla_decode.so``); this package is a thin
ctypes binding with the same names:

    p = plan(seq_lens, s_q=1, max_pages_per_seq=maxp)       # mla_decode_plan
    o_latent, lse = decode(p, q_latent, q_rope, kv_cache, block_table)   # mla_decode
    status = check(p)                                         # mla_decode_check

The step before attention (``include/mla_prolog.h``) produces q_latent and
q_rope and appends the step's rows to the cache:

    q_latent, q_rope, st = prolog(q_nope, q_pe, kv_latent, k_pe, w_uk, gamma,
                                  kv_cache, block_table, seq_lens)   # mla_prolog

and the step after it (``include/mla_epilog.h``) projects the heads back out:

    o_v, st = epilog_uv(o_latent, w_uv)                      # mla_epilog_uv
    out = epilog_oproj(o_v, w_o)                             # mla_epilog_oproj

An fp8 (e4m3) cache (``include/mla_fp8.h``) holds half the bytes per token:

    kv8 = quantize_cache_fp8(kv_cache)                       # mla_cache_quantize_fp8
    o_latent, lse = decode_fp8(p, q_latent, q_rope, kv8, block_table)   # mla_decode_fp8
"""

from ._binding import (D_V, HIDDEN, DEFAULT_ROPE_BASE, DEFAULT_RMS_EPS, DEFAULT_SCALE, D_LATENT, D_NOPE, D_ROPE, LIB_PATH, NUM_HEADS, PAGE_SIZE,
                       MLA_DEV_BAD_PAGE, MLA_DEV_BAD_PLAN, MLA_DEV_BAD_SEQ_LEN, MLA_DEV_TIMEOUT,
                       MLAError, MLA_FLAG_POW2_MAX, MLA_INJECT_WITHHOLD_K_LOAD, NOALLOC_SCRATCH_BYTES, Plan, check, decode,
                       decode_diag, decode_fp8, decode_noalloc, epilog_oproj, epilog_uv, quantize_cache_fp8,
                       load_library, num_units, parse_plan, plan, prolog, rope_table,
                       plan_device_bytes, plan_host, plan_layout, workspace_size)

__all__ = ["D_V", "HIDDEN", "epilog_oproj", "epilog_uv",
           "quantize_cache_fp8",
           "DEFAULT_ROPE_BASE", "DEFAULT_RMS_EPS", "DEFAULT_SCALE", "D_LATENT", "D_NOPE", "D_ROPE", "LIB_PATH", "NUM_HEADS", "PAGE_SIZE",
           "MLA_DEV_BAD_PAGE", "MLA_DEV_BAD_PLAN", "MLA_DEV_BAD_SEQ_LEN", "MLA_DEV_TIMEOUT",
           "MLAError", "MLA_FLAG_POW2_MAX", "MLA_INJECT_WITHHOLD_K_LOAD", "NOALLOC_SCRATCH_BYTES", "Plan", "check", "decode",
           "decode_diag", "decode_fp8", "decode_noalloc",
           "load_library", "num_units", "parse_plan",
           "plan", "plan_device_bytes", "prolog", "rope_table", "plan_host", "plan_layout", "workspace_size"]
