/*
 * mla_fp8.h - C ABI for the fp8 (e4m3) latent cache format.
 *
 * The low-bit KV cache the Ascend best-practice page lists as next work
 * ("Huawei Ascend servers: DeepSeek V3/R1 inference best practice", section
 * 8: KV-cache-only quantisation of the attention operators), in the form this
 * GPU has native arithmetic for.  One row (token) of the fp8 cache is
 * MLA_FP8_ROW_BYTES = 656 bytes:
 *
 *   [0, 512)    e4m3 codes of c_kv[i] / s, i < 512 (round to nearest even,
 *               saturating at +-448)
 *   [512, 640)  k_rope[i] / s, i < 64, as bf16 (round to nearest even)
 *   [640, 644)  s = max_i |c_kv[i]| / 448 as fp32 (1 for an all-zero c_kv)
 *   [644, 656)  zero
 *
 * s and every quotient (c_kv[i] / s, k_rope[i] / s) are correctly rounded
 * fp32 values, so the row is a function of the bf16 row alone.  The whole
 * 576-value row dequantises by the one factor s: c_kv as value(code) * s,
 * within half an e4m3 step (2^-4 of the row's largest magnitude), k_rope as
 * value(bf16) * s, within half a bf16 step.  One factor for the whole row
 * lets a kernel form a score with one contraction over all 576 values and
 * scale it once.  Rows must be finite.
 *
 * Conventions (as in mla_decode.h): device pointers, caller-owned buffers,
 * work enqueued on `stream`, nothing synchronises; host argument errors
 * return a status and enqueue nothing.
 */
#ifndef MLA_FP8_H
#define MLA_FP8_H

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_FP8_ROW_BYTES 656

/*
 * Quantise num_rows rows of a bf16 cache (kv_cache: [num_rows][576] bf16, e.g.
 * num_pages * 64 rows of a paged cache) into kv_cache_fp8 ([num_rows][656]
 * bytes).  Both pointers 16-byte aligned; num_rows >= 1.
 */
mla_status mla_cache_quantize_fp8(const void *kv_cache, int64_t num_rows, void *kv_cache_fp8,
                                  mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_FP8_H */
