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

/*
 * mla_decode over a paged fp8 cache (kv_cache_fp8: [num_pages][64][656] bytes in
 * the row format above): the attention of mla_decode on the dequantised rows.
 * Same problem, schedule (mla_decode_plan), workspace, outputs, scale rule,
 * flags and error contract as mla_decode; num_pages bounds the block table's
 * entries as there.  q stays bf16; the kernel turns each page's e4m3 codes into
 * bf16 operands on the SM (exactly: every e4m3 value is a bf16 value), contracts
 * q with [codes | k_rope / s] in fp32, multiplies each score by its token's s,
 * and folds s into each attention weight before the weight is rounded to bf16
 * for the contraction with the codes.  The roundings are thus those of
 * mla_decode (bf16 weights, fp32 accumulation, bf16 o_latent), moved by the
 * factor s, and the result is the dequantised cache's attention to that
 * accuracy.  Half the cache bytes per token (656 against 1152).  The cache
 * pointer must be 16-byte aligned.  events: NULL, or 3 cudaEvent_t handles
 * recorded as mla_decode_timed records them (before the main kernel, before
 * the merge, after the merge; NULL entries skipped).
 */
mla_status mla_decode_fp8(const mla_problem *prob, const void *q_latent, const void *q_rope,
                          const void *kv_cache_fp8, int64_t num_pages, const int32_t *block_table,
                          float scale, void *o_latent, float *lse, void *workspace,
                          size_t workspace_bytes, mla_stream_t stream, void *const *events);

#ifdef __cplusplus
}
#endif

#endif /* MLA_FP8_H */
