"""GB300 (sm_103a) weight-absorbed MLA decode over a paged 576-d latent cache.

The computation runs in hand-written CUDA kernels behind the C ABI in
``include/mla_decode.h`` (``libmla_decode.so``); this package is a thin
ctypes binding with the same names:

    p = plan(seq_lens, s_q=1, max_pages_per_seq=maxp)       # mla_decode_plan
    o_latent, lse = decode(p, q_latent, q_rope, kv_cache, block_table)   # mla_decode
    status = check(p)                                         # mla_decode_check
"""

from ._binding import (DEFAULT_SCALE, D_LATENT, D_ROPE, LIB_PATH, NUM_HEADS, PAGE_SIZE,
                       MLA_DEV_BAD_PAGE, MLA_DEV_BAD_PLAN, MLA_DEV_BAD_SEQ_LEN, MLA_DEV_TIMEOUT,
                       MLAError, NOALLOC_SCRATCH_BYTES, Plan, check, decode, decode_noalloc,
                       load_library, num_units, parse_plan, plan,
                       plan_device_bytes, plan_host, plan_layout, workspace_size)

__all__ = ["DEFAULT_SCALE", "D_LATENT", "D_ROPE", "LIB_PATH", "NUM_HEADS", "PAGE_SIZE",
           "MLA_DEV_BAD_PAGE", "MLA_DEV_BAD_PLAN", "MLA_DEV_BAD_SEQ_LEN", "MLA_DEV_TIMEOUT",
           "MLAError", "NOALLOC_SCRATCH_BYTES", "Plan", "check", "decode", "decode_noalloc",
           "load_library", "num_units", "parse_plan",
           "plan", "plan_device_bytes", "plan_host", "plan_layout", "workspace_size"]
