/*
 * mla_decode.h - C ABI of a GB300 (sm_103a) library for decode-phase
 * Multi-head Latent Attention in its weight-absorbed form over a paged,
 * compressed KV cache.
 *
 * What the library computes (sources are the pages this project follows):
 *
 *   "Huawei Ascend servers: DeepSeek V3/R1 inference best practice",
 *   section 3.2.1 (Multi-head Latent Attention): the heads of MLA share one
 *   compressed KV cache, and decode runs with weight absorption, so every
 *   head attends over the same cached rows.  Section 7.2 (CloudMatrix 384
 *   performance analysis) fixes the sizes through its cost formula
 *   BS x 3072 x (576 + 512) x 128 x 2 x 2: scores contract over 576 values,
 *   outputs over 512, and there are 128 heads.  Section 6.1 (MLA operator
 *   optimisation) computes it as tiled exact softmax attention after
 *   FlashAttention.
 *
 *   For request b, query token t < s_q and head h < 128, with
 *   L_vis = seq_lens[b] - s_q + 1 + t visible keys and cached row
 *   r_j = kv_cache[block_table[b][j / 64]][j % 64] (512 c_kv values, then 64
 *   k_rope values):
 *
 *     s_j  = scale * (q_latent[b][t][h] . r_j[0:512] + q_rope[b][t][h] . r_j[512:576])
 *     o    = sum_{j < L_vis} softmax(s)_j * r_j[0:512]      -> o_latent[b][t][h][0:512], bf16
 *     lse  = ln sum_{j < L_vis} exp(s_j)                     -> lse[b][t][h], fp32
 *
 *   Long rows are split across the GPU and merged by log-sum-exp, as the
 *   FlashDecoding optimisation does (Atlas 800I A3 TPOT-jitter
 *   troubleshooting post, "MLAKernel performance root cause"); the split
 *   schedule is length-aware so that a mix of long and short requests keeps
 *   every SM busy (the same post, and section 8 of the Ascend report on
 *   sequence load balancing).
 *
 * Conventions for every entry point:
 *  - All array arguments are DEVICE pointers unless the name ends in _host.
 *    The caller owns every buffer (the workspace included); the library
 *    allocates no device memory and only borrows pointers for the duration
 *    of the stream-ordered work it enqueues.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and nothing synchronises, except mla_decode_check.
 *  - Host-side argument errors return a status and enqueue nothing.
 *    Errors found on the device (a block_table entry outside the page pool,
 *    seq_len < s_q, a row longer than max_pages_per_seq pages) set a status
 *    word in the workspace, which mla_decode_check reads; the affected rows
 *    are written as NaN and no memory outside the caller's buffers is
 *    touched.
 *  - Layouts are dense row-major (C order), no padding:
 *      q_latent    [batch][s_q][num_heads][512]       bf16
 *      q_rope      [batch][s_q][num_heads][64]        bf16
 *      kv_cache    [num_pages][page_size][576]        bf16
 *      block_table [batch][max_pages_per_seq]         int32
 *      seq_lens    [batch]                            int32 (keys cached, this step's included)
 *      o_latent    [batch][s_q][num_heads][512]       bf16
 *      lse         [batch][s_q][num_heads]            fp32 (natural log)
 *    Every base pointer must be 16-byte aligned.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *mla_stream_t;

#define MLA_NUM_HEADS 128
#define MLA_D_LATENT 512
#define MLA_D_ROPE 64
#define MLA_PAGE_SIZE 64

typedef enum mla_status {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad scale */
    MLA_ERR_UNSUPPORTED = 2,  /* a shape outside the supported set (see mla_problem) */
    MLA_ERR_WORKSPACE = 3,    /* workspace smaller than mla_decode_workspace_size() */
    MLA_ERR_CUDA = 4,         /* a CUDA runtime or driver call failed */
    MLA_ERR_DEVICE_CHECK = 5, /* mla_decode_check: the device recorded an input error */
    MLA_ERR_TIMEOUT = 6       /* mla_decode_check: a bounded device wait gave up */
} mla_status;

/* Device status bits (mla_decode_check's device_status). */
#define MLA_DEV_BAD_PAGE 0x1     /* block_table entry < 0 or >= num_pages */
#define MLA_DEV_BAD_SEQ_LEN 0x2  /* seq_len < s_q, or more pages than max_pages_per_seq */
#define MLA_DEV_BAD_PLAN 0x4     /* workspace plan does not match the problem */
#define MLA_DEV_TIMEOUT 0x8      /* a bounded wait inside a kernel ran out */

/*
 * Problem description.  Supported set: batch >= 1, s_q in {1, 2},
 * num_heads == 128, page_size == 64, max_pages_per_seq >= 1,
 * batch * max_pages_per_seq < 2^31, flags == 0 or MLA_FLAG_POW2_MAX
 * (decode entry points only; the prolog and epilog require 0).
 */
typedef struct mla_problem {
    int32_t batch;
    int32_t s_q;
    int32_t num_heads;
    int32_t page_size;
    int32_t max_pages_per_seq; /* row stride of block_table; bounds every seq_len */
    int32_t flags;
} mla_problem;

/*
 * Power-of-two running maxima (the AMLA-style rescale of "Huawei Ascend
 * servers: DeepSeek V3/R1 inference best practice", section 6.1): the online
 * softmax keeps each running max as an integer in log2 units (a raised max is
 * rounded up), so every rescale of P and of the output accumulator is by an
 * exact power of two.  The result is the same attention (within the usual
 * tolerance); only the rounding path differs.  The planner ignores the flag.
 */
#define MLA_FLAG_POW2_MAX 0x1

/*
 * Bytes of device workspace that mla_decode_plan / mla_decode need for this
 * problem on the current device.  The workspace holds the split schedule,
 * the fp32 partial outputs of split rows and the device status word.
 * Returns MLA_OK and writes *bytes, or an argument/CUDA error.
 */
mla_status mla_decode_workspace_size(const mla_problem *prob, size_t *bytes);

/*
 * Number of work units (SM groups) the main kernel runs on the current
 * device; the schedule splits the work across exactly this many.
 */
mla_status mla_decode_num_units(int32_t *units);

/*
 * Build the length-aware split-KV schedule from seq_lens (device, [batch]
 * int32) into the workspace, on `stream`.  One single-CTA kernel: it reads
 * seq_lens on the device, so no host synchronisation is needed.  The
 * schedule stays valid for every later mla_decode with the same problem and
 * seq_lens (e.g. every layer of a decode step).  Also clears the status word.
 */
mla_status mla_decode_plan(const mla_problem *prob, const int32_t *seq_lens, void *workspace,
                           size_t workspace_bytes, mla_stream_t stream);

/*
 * Run the attention for the schedule in `workspace` (built by
 * mla_decode_plan for the same problem): the main kernel, then the LSE
 * merge of split rows.  kv_cache holds num_pages pages; scale multiplies
 * the 576-value dot product (1/sqrt(192) for DeepSeek V3/R1) and must be
 * finite and > 0 (MLA_ERR_INVALID_ARG otherwise).  Writes o_latent (bf16)
 * and lse (fp32) for every (b, t, h).  Argument errors (null or unaligned
 * pointers, num_pages < 1, a bad scale, a workspace below the size any
 * device could need) are found before any CUDA call.
 */
mla_status mla_decode(const mla_problem *prob, const void *q_latent, const void *q_rope,
                      const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                      float scale, void *o_latent, float *lse, void *workspace,
                      size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_decode with phase timing for profiling tools: records events[0] on
 * `stream` before the main kernel, events[1] after it (before the merge)
 * and events[2] after the merge.  events points to 3 cudaEvent_t handles
 * created by the caller; NULL entries are skipped.  Under stream capture the
 * records are external event nodes (cudaEventRecordExternal), so the
 * timestamps can be read after the graph is launched.  Same contract as
 * mla_decode otherwise.
 */
mla_status mla_decode_timed(const mla_problem *prob, const void *q_latent, const void *q_rope,
                            const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                            float scale, void *o_latent, float *lse, void *workspace,
                            size_t workspace_bytes, mla_stream_t stream, void *const *events);

/*
 * mla_decode with a caller-chosen limit for the bounded waits inside the
 * main kernel, and an optional injected stall, for testing the time-out path
 * without a GPU fault.  The pages have no counterpart of this entry point.
 *  - wait_limit_ns: how long any one wait of the main kernel may last before
 *    the kernel records MLA_DEV_TIMEOUT and winds down (mla_decode uses 2 s).
 *    Must lie in [1000, 60e9]; MLA_ERR_INVALID_ARG otherwise.
 *  - inject: 0, or MLA_INJECT_WITHHOLD_K_LOAD: the first CTA of the work
 *    unit that runs the schedule's first item never issues the K-stage load
 *    of its second page, so the waits for it run out (the unit must own two
 *    pages or more, else nothing is withheld).  The kernel then records MLA_DEV_TIMEOUT, lets every copy
 *    already in flight land, frees its tensor memory and returns; the rows of
 *    that unit are left unspecified, the stream and context stay usable, and
 *    the next call (which rewrites the status word in mla_decode_plan) runs
 *    normally.  Other bits: MLA_ERR_INVALID_ARG.
 * With inject == 0 the results are those of mla_decode, bit for bit.
 */
#define MLA_INJECT_WITHHOLD_K_LOAD 0x1u
mla_status mla_decode_diag(const mla_problem *prob, const void *q_latent, const void *q_rope,
                           const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                           float scale, void *o_latent, float *lse, void *workspace,
                           size_t workspace_bytes, mla_stream_t stream, uint64_t wait_limit_ns,
                           uint32_t inject);

/*
 * Synchronise `stream`, read the device status word from the workspace into
 * *device_status (MLA_DEV_* bits) and return MLA_OK if it is zero,
 * MLA_ERR_TIMEOUT if MLA_DEV_TIMEOUT is set, else MLA_ERR_DEVICE_CHECK.
 */
mla_status mla_decode_check(const void *workspace, int32_t *device_status, mla_stream_t stream);

/* Static English text for a status code (never NULL). */
const char *mla_status_string(mla_status status);

/*
 * The planner's algorithm run on the host, for tests and tooling: writes
 * the same schedule bytes that mla_decode_plan writes at the start of the
 * workspace, for `num_units` units, into plan_host (host memory of
 * plan_bytes >= mla_decode_plan_bytes(prob, num_units)).  seq_lens_host is
 * host memory.
 */
size_t mla_decode_plan_bytes(const mla_problem *prob, int32_t num_units);
mla_status mla_decode_plan_host(const mla_problem *prob, const int32_t *seq_lens_host,
                                int32_t num_units, void *plan_host, size_t plan_bytes);

/*
 * Allocation-free variant of plan + decode.  The pages have no counterpart
 * of this entry point: it exists for callers that cannot call cudaMalloc on
 * their decode path, such as serving loops and plugin hosts that own every
 * byte of device memory, or latency-critical code where an allocation (which
 * may synchronise the device and has unbounded latency) is forbidden.
 *
 * It runs mla_decode_plan and mla_decode with the workspace placed in a
 * file-scope static device array of MLA_NOALLOC_SCRATCH_BYTES bytes inside
 * the library, so the caller passes only inputs and outputs (same layouts
 * and meanings as mla_decode; seq_lens is a device pointer).  Every GPU on
 * which this entry point runs holds that array until the process exits.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make
 *    that first call before any stream capture.
 *  - Problems whose workspace (mla_decode_workspace_size) exceeds
 *    MLA_NOALLOC_SCRATCH_BYTES are rejected with MLA_ERR_WORKSPACE before
 *    anything is enqueued.
 *  - It allocates nothing: no cudaMalloc, cudaFree or allocating library
 *    routine is called.
 *  - All calls share the one array and it keeps the last call's contents;
 *    every call rewrites the schedule and status word before reading them.
 *    Calls that overlap on the GPU (e.g. on two streams, or from two host
 *    threads without ordering) race on the array and give wrong results:
 *    order them on one stream.
 *  - The device status word is not readable through mla_decode_check here;
 *    rows with device-detected input errors are still written as NaN.
 */
#define MLA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
mla_status mla_decode_noalloc(const mla_problem *prob, const void *q_latent, const void *q_rope,
                              const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                              const int32_t *seq_lens, float scale, void *o_latent, float *lse,
                              mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
