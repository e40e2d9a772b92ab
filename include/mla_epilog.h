/*
 * mla_epilog.h - C ABI of the step after decode attention: the value
 * up-projection of every head and the output projection.
 *
 * What it computes (sources are the pages this project follows):
 *
 *   "Huawei Ascend servers: DeepSeek V3/R1 inference best practice",
 *   section 3.2.1 (Multi-head Latent Attention): with the weights absorbed,
 *   mla_decode returns each head's output in the 512-value latent space
 *   (o_latent); the head's value up-projection brings it to its 128 value
 *   dims.  Sections 3.2-3.3 (figures 5-9) place the output projection
 *   ("O Proj") after attention; the pages print no shape for it, DeepSeek
 *   V3/R1 maps the 128 x 128 = 16384 head values to a hidden size of 7168.
 *
 *   For token tok = b * s_q + t, head h < 128, value dim v < 128, n < hidden:
 *
 *     o_v[tok][h][v] = sum_c w_uv[h][v][c] * o_latent[tok][h][c]      c < 512
 *     out[tok][n]    = sum_k w_o[n][k] * o_v[tok][k / 128][k % 128]    k < 16384
 *
 * Conventions (as in mla_decode.h): device pointers; caller-owned buffers;
 * work enqueued on `stream`, nothing synchronises; host-side argument errors
 * return a status and enqueue nothing.  Dense row-major layouts, every base
 * pointer 16-byte aligned:
 *      o_latent [batch][s_q][num_heads][512]   bf16 (mla_decode's output)
 *      w_uv     [num_heads][128][512]          bf16 (row v of head h: the 512
 *                                              latent weights of value dim v)
 *      o_v      [batch][s_q][num_heads][128]   bf16
 *      w_o      [hidden][16384]                bf16 (row n: the weights of output n)
 *      out      [tokens][hidden]               bf16
 */
#ifndef MLA_EPILOG_H
#define MLA_EPILOG_H

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_D_V 128
#define MLA_HIDDEN 7168

/*
 * The value up-projection: one tensor-core kernel on `stream`.  prob: the
 * problem description of the mla_decode that produced o_latent (batch >= 1,
 * s_q in {1, 2}, num_heads 128).  device_status: a device int32 the caller
 * clears; MLA_DEV_TIMEOUT is OR-ed in if a bounded wait inside the kernel
 * ran out (o_v is then not written for that tile).
 */
mla_status mla_epilog_uv(const mla_problem *prob, const void *o_latent, const void *w_uv,
                         void *o_v, int32_t *device_status, mla_stream_t stream);

/*
 * The output projection: out = o_v . w_o^T, bf16 in and out, fp32
 * accumulation, for `tokens` rows of o_v (viewed as [tokens][16384]): one
 * tensor-core kernel on `stream` (each SM pair holds 128 outputs and splits
 * the 16384-term sums in two halves that it adds in a fixed way, so the
 * result is the same on every run).  tokens >= 1; hidden >= 8 and a multiple
 * of 8.  device_status: a device int32 the caller clears; MLA_DEV_TIMEOUT is
 * OR-ed in if a bounded wait inside the kernel ran out (that tile of out is
 * then not written).
 */
mla_status mla_epilog_oproj(int32_t tokens, int32_t hidden, const void *o_v, const void *w_o,
                            void *out, int32_t *device_status, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_EPILOG_H */
