/*
 * mla_prolog.h - C ABI of the MLA prolog slice: the step of a decode layer
 * that produces the attention inputs of mla_decode (include/mla_decode.h).
 *
 * What it computes (sources are the pages this project follows):
 *
 *   "Huawei Ascend servers: DeepSeek V3/R1 inference best practice",
 *   section 3.2.1 (Multi-head Latent Attention): decode absorbs the key
 *   up-projection into the query, so each head's 128-value no-position query
 *   becomes a 512-value query against the shared compressed cache.  Section
 *   6.1 names the fused operator that does this ahead of attention
 *   (MLAProlog); the CloudMatrix384 digest, section 3.2 (MLA optimisation),
 *   lists what it fuses: RMSNorm, the Q/K/V projections and RoPE.  This entry
 *   point is the part of that operator after the projections:
 *
 *   For request b, new token t < s_q, head h, with
 *   pos = seq_lens[b] - s_q + t (seq_lens count this step's tokens, as in
 *   mla_decode), and tok = b * s_q + t:
 *
 *     q_latent[tok][h][n] = sum_k q_nope[tok][h][k] * w_uk[h][k][n]     k < 128, n < 512
 *     q_rope[tok][h]      = RoPE(q_pe[tok][h], pos)
 *     cache row pos of b  = RMSNorm(kv_latent[tok]) || RoPE(k_pe[tok], pos)
 *
 *   RoPE rotates the pairs (2i, 2i+1) of the 64 position dims by the angle
 *   pos * rope_base^(-2i/64) (rope_base enters through the table of
 *   mla_prolog_rope_table); RMSNorm is x / sqrt(mean(x^2) + rms_eps) *
 *   kv_norm_weight over the 512 latent values.  The pages give neither
 *   formula; these are the standard definitions of both (DeepSeek V3/R1 uses
 *   rope_base 10000 and rms_eps 1e-6).  The cache row of position pos is
 *   kv_cache[block_table[b][pos / 64]][pos % 64].
 *
 * Conventions (as in mla_decode.h): device pointers; caller-owned buffers;
 * work enqueued on `stream`, nothing synchronises; host-side argument
 * errors return a status and enqueue nothing.  Dense row-major layouts,
 * every base pointer 16-byte aligned:
 *      q_nope         [batch][s_q][num_heads][128]    bf16
 *      q_pe           [batch][s_q][num_heads][64]     bf16 (before RoPE)
 *      kv_latent      [batch][s_q][512]               bf16 (before RMSNorm)
 *      k_pe           [batch][s_q][64]                bf16 (before RoPE)
 *      w_uk           [num_heads][128][512]           bf16 (row k of head h: the
 *                                                     512 latent weights of dim k)
 *      kv_norm_weight [512]                           bf16
 *      kv_cache       [num_pages][64][576]            bf16, updated in place
 *      block_table    [batch][max_pages_per_seq]      int32
 *      seq_lens       [batch]                         int32
 *      q_latent       [batch][s_q][num_heads][512]    bf16 (output)
 *      q_rope         [batch][s_q][num_heads][64]     bf16 (output)
 *
 * Device-detected errors are OR-ed into *device_status (a device int32 the
 * caller clears; MLA_DEV_* bits of mla_decode.h): MLA_DEV_BAD_SEQ_LEN when
 * pos < 0 or pos / 64 >= max_pages_per_seq, MLA_DEV_BAD_PAGE when the block
 * table entry is outside [0, num_pages), MLA_DEV_TIMEOUT when a bounded
 * wait inside the kernel ran out.  A token whose position is out of range
 * (MLA_DEV_BAD_SEQ_LEN) gets NaN in its q_rope; a token with a bad slot of
 * either kind writes nothing to the cache; every other output is computed.
 */
#ifndef MLA_PROLOG_H
#define MLA_PROLOG_H

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_D_NOPE 128
#define MLA_ROPE_TABLE_FLOATS 64

/*
 * The rotary table of a model: for each pair i < 32 the turns per position
 * g_i = rope_base^(-2i/64) / (2 pi), computed in fp64 on the device (one
 * 32-thread kernel on `stream`) and stored as an unevaluated sum of two
 * floats, table[i] = hi and table[32 + i] = lo (hi + lo carries g_i to about
 * 2^-48 relative).  It depends on rope_base alone: build it once per model,
 * like the rotary cache of a serving engine, and pass it to every
 * mla_prolog.  table: device memory of MLA_ROPE_TABLE_FLOATS floats, 4-byte
 * aligned, owned by the caller.  rope_base must be finite and > 0.
 */
mla_status mla_prolog_rope_table(double rope_base, float *table, mla_stream_t stream);

/*
 * One launch on `stream`.  prob: the same problem description as
 * mla_decode (batch >= 1, s_q in {1, 2}, num_heads 128, page_size 64).
 * rope_table: a table written by mla_prolog_rope_table (device memory);
 * rms_eps finite and >= 0; num_pages >= 1.  kv_cache rows other than the
 * new tokens' are neither read nor written.
 */
mla_status mla_prolog(const mla_problem *prob, const void *q_nope, const void *q_pe,
                      const void *kv_latent, const void *k_pe, const void *w_uk,
                      const void *kv_norm_weight, float rms_eps, const float *rope_table,
                      void *kv_cache, int64_t num_pages, const int32_t *block_table,
                      const int32_t *seq_lens, void *q_latent, void *q_rope, int32_t *device_status,
                      mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PROLOG_H */
