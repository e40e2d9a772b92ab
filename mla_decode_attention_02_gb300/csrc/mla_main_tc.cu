// Main attention kernel: weight-absorbed MLA decode on the 5th-generation
// tensor cores (tcgen05 + TMEM), pages streamed by TMA.
//
// What it computes is the attention of "Huawei Ascend servers: DeepSeek
// V3/R1 inference best practice" section 3.2.1 (128 heads share one
// 576-value cached row per token, weights absorbed) as tiled exact softmax
// attention (section 6.1, after FlashAttention), over the key ranges the
// split-KV schedule hands each work unit (FlashDecoding, Atlas 800I A3
// troubleshooting post).
//
// GB300 design.  The fp32 output of one row (128 heads x 512 values =
// 256 KB) alone fills one SM's tensor memory, so a work unit is a cluster of
// two CTAs on two SMs: CTA c owns output columns [256c, 256c + 256) and the
// tokens [32c, 32c + 32) of every 64-token page.
//
//   S_c = q . k_c^T     tcgen05 M=128 (heads) N=32 (own tokens) K=576, fp32
//                       in TMEM (two buffers: page parity); q dims 0-383
//                       are the A operand in TMEM, 384-575 in shared memory
//   P_c = exp2(S_c*scale*log2e - m)   fp32, rounded to bf16, into this CTA's
//                       P slot and, by asynchronous remote stores, into the
//                       peer's (9 KB per page)
//   merge: the pair agrees on the running max per head (each side's max
//          travels with its P half; the lower half is scaled) and rescales
//          O when the max grows; each half's running row sum rides along
//   O_c += [P_0 | P_1] . V_c   tcgen05 M=128 N=256 K=64, V_c = the page's
//                       latent dims [256c, 256c + 256) of all 64 tokens
//
// Three rings, so that no stage waits for a later one: the K ring (this
// CTA's 32 tokens of a page, all 576 dims, 36 KB) is freed by the score
// MMAs; the V ring (the page's 64 tokens of this CTA's 256 output dims,
// 32 KB; own tokens loaded a second time, from L2) and the P ring (the two
// halves' P tiles and messages, 18 KB, two slots) are freed by PV.  Each
// K and V stage is one TMA box of a blocked view of the cache (one SM takes
// in a few large TMA copies from L2 far faster than many 4 KB ones: about
// 117 ns per copy plus 5 ns per KB, measured on this part).
//
// Each softmax thread stores its head's P row and (max, row sum) twice: into
// this CTA's P slot and, with st.async, into the peer's, whose mbarrier
// counts the bytes (one phase per page, armed by a merge warp of the
// receiver).  The P slot lives from the softmax of a page to the PV of both
// CTAs, and only a few fit in shared memory, so the exchange latency bounds the
// page rate: a bulk copy of the half through the TMA engine queued behind the
// page loads and took about 2 us; the remote stores take about 0.5 us, so two
// slots suffice and the space of a third holds the second score buffer's q
// dims instead.  With one score buffer the next page's score MMAs waited for
// the softmax to read the scores, and that loop (about 1.3 us) set the page
// rate.
// The sender's own half stays its own: the merge may rescale it in place.
//
// TMEM (512 columns): O half [0,256), S [256,320), q [320,512).  Warp roles
// per CTA: warp 0 loads the K ring and q, warp 2 the V ring; warp 1 issues
// the score MMAs and warp 3 the PV MMAs (each a whole warp that waits
// together and issues from one elected lane: about 15 ns per tcgen05.mma,
// against 35 ns from a lane-0 branch); warps 4-7 (one per TMEM lane quarter,
// one thread per head) load q into TMEM, compute P and send it to the peer;
// warps 8-11 merge the two halves and run the epilogue.  The score buffer is released
// right after the softmax's TMEM load, so the next page's score MMAs wait
// only for that.  Every wait is bounded: on time-out the kernel records
// MLA_DEV_TIMEOUT and winds down instead of hanging.
//
// fp8 cache (the same kernel, kFp8 = true, 512 threads): the K load brings the
// 32 tokens' e4m3 codes (16 KB) into the upper half of the stage's latent
// blocks, k_rope / s (bf16) into its place, and the tokens' scales into a
// four-slot ring; the V load brings the codes of the CTA's 256 dims (16 KB)
// into the upper half of the V stage.  Warps 12-13 expand each K stage and
// warps 14-15 each V stage in place into the bf16 layout above (exact: every
// e4m3 value is a bf16 value), then release it to the MMAs.  The softmax
// multiplies each score by its token's s and folds s into the token's weight
// before rounding it to bf16, so both contractions see the codes themselves.
// The expansion lengthens each stage's load-to-MMA chain on the two-stage
// rings, which sets this variant's page rate (about twice the bf16 cache's
// time per page, measured): the fp8 cache halves the bytes held per token,
// not the time.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mla_fp8.h"
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kQkWarp = 1;          // score MMAs (and TMEM allocation)
constexpr int kVWarp = 2;           // V ring loads
constexpr int kPvWarp = 3;
constexpr int kSoftmaxWarp0 = 4;    // warps 4-7
constexpr int kMergeWarp0 = 8;      // warps 8-11
constexpr int kKStages = 2;         // K ring (page parity)
constexpr int kVStages = 2;         // V ring (page parity)
constexpr int kPSlots = 2;          // P ring (page parity)
constexpr int kPrefetch = 3;        // L2 prefetch distance in pages
constexpr int kClusterSize = 2;
constexpr int kHalfTok = 32;                      // tokens of a page per CTA
constexpr uint32_t kBox = kHalfTok * 128;         // 32 tokens x 64 dims, 128-byte swizzle
constexpr uint32_t kKStageBytes = 9 * kBox;       // own tokens, dim blocks 0-8 (one TMA box)
constexpr uint32_t kVBlk = kPage * 128;           // 64 tokens x 64 dims, 128-byte swizzle
constexpr uint32_t kVStageBytes = 4 * kVBlk;      // the page's tokens x output dims (one TMA box)
constexpr uint32_t kPHalf = 128 * 64;             // one token half: 128 heads x 32 tokens, bf16,
                                                  // 64-byte rows, 64-byte swizzle
constexpr uint32_t kPPart = kPHalf + 1024;        // a CTA's part of a P slot: its half, then
                                                  // (max, row sum) per head; one copy to the peer
constexpr uint32_t kPSlotBytes = 2 * kPPart;
static_assert(kPPart % 512 == 0, "64-byte-swizzle tiles start on 512-byte boundaries");
constexpr uint32_t kQBlk = 128 * 128;             // q block: 128 heads x 64 dims
constexpr int kQTDims = 384;                      // q dims 0-383 live in TMEM
constexpr int kQSBlocks = (kDl + kDr - kQTDims) / 64;   // q dims 384-575: 64-dim blocks in shared memory
constexpr uint32_t kQSBytes = kQSBlocks * kQBlk;
constexpr int kRefLag = 4;          // the softmax of page g starts from the agreed max of page g - 4
constexpr uint32_t kOffQS = 0;
constexpr uint32_t kOffK = kQSBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kKStageBytes;
constexpr uint32_t kOffP = kOffV + kVStages * kVStageBytes;
constexpr uint32_t kOffRef = kOffP + kPSlots * kPSlotBytes;   // agreed max, kRefLag x 128 floats
constexpr uint32_t kOffBar = kOffRef + kRefLag * 512;
constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;  // + barriers, + alignment slack
// fp8 cache (variant of the same kernel): four more warps convert each landed K
// and V stage from e4m3 codes to the bf16 layout above, and each K load brings
// this CTA's 32 tokens' scales (16 bytes per token) into a ring after the barriers
constexpr int kThreadsFp8 = 512;
constexpr int kConvWarp0 = 12;                      // warps 12-15 (fp8 only)
constexpr uint32_t kScaleStage = kHalfTok * 16;     // 512 bytes per page
constexpr int kScaleSlots = 4;                      // page mod 4, freed by the softmax
constexpr uint32_t kOffScale = kOffBar + 512;
constexpr uint32_t kSmemBytesFp8 = kOffScale + kScaleSlots * kScaleStage + 1024;
static_assert(kSmemBytesFp8 <= 232448, "shared memory budget (fp8)");
static_assert(kOffScale % 128 == 0, "scale ring alignment");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0 &&
                  kKStageBytes % 1024 == 0 && kVStageBytes % 1024 == 0 && kPSlotBytes % 1024 == 0,
              "TMA/UMMA tile alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kMsgBytes = kPPart;            // per page: P half tile + (max, row sum) per head

// TMEM columns
constexpr uint32_t kColO = 0;       // 256 fp32 output columns of this CTA's half
constexpr uint32_t kColS = 256;     // 2 x 32 fp32 scores (page parity)
constexpr uint32_t kColQ = 320;     // 192 columns of packed bf16 q (dims 0-383)
constexpr uint32_t kTmemCols = 512;
static_assert(kColQ + kQTDims / 2 == kTmemCols, "TMEM budget");

constexpr float kRescaleThreshold = 8.0f;  // log2 units: raise the max only when it grows by > 2^8

// barrier slots (8 bytes each) in the barrier area
enum : uint32_t {
    B_Q_FULL = 0,                        // softmax warps: q dims 0-383 in TMEM
    B_Q_EMPTY = 1,                       // this CTA's score MMAs done with the item's q
    B_KFULL = 2,                         // + page parity: K stage landed (+tx)
    B_KEMPTY = B_KFULL + 2,              // + page parity: score MMAs done with the K stage
    B_VFULL = B_KEMPTY + 2,              // + page parity: V stage landed (+tx)
    B_VEMPTY = B_VFULL + 2,              // + page parity: PV done with the V stage
    B_PEMPTY = B_VEMPTY + 2,             // + slot: this CTA's PV done with the P slot
    B_PEMPTY_PEER = B_PEMPTY + kPSlots,  // + slot: the peer's PV done with its P slot
    B_SFULL = B_PEMPTY_PEER + kPSlots,   // + page parity: scores in TMEM
    B_SEMPTY = B_SFULL + 2,              // + page parity: scores read into registers
    B_SDONE = B_SEMPTY + 2,              // + slot: own P half written
    B_PMSG = B_SDONE + kPSlots,          // + slot: the peer's P half arrived (+tx, remote stores)
    B_PREADY = B_PMSG + kPSlots,         // + slot: P tile final, PV may run
    B_RESDONE = B_PREADY + kPSlots,      // + page mod kRefLag: agreed max published
    B_PVDONE = B_RESDONE + kRefLag,      // + page parity: PV done
    B_PVLAST = B_PVDONE + 2,             // an item's last PV done (one phase per item)
    B_OFREE = B_PVLAST + 1,              // epilogue done reading O
    B_EPI = B_OFREE + 1,                 // merge warps done with the staged epilogue
    B_DRAIN = B_EPI + 1,                 // + issuer (0: score, 1: PV)
    B_QSTAGE = B_DRAIN + 2,              // item start: q dims 0-319 staged (+tx)
    B_QCOPIED = B_QSTAGE + 1,            // item start: softmax warps moved the staged q to TMEM
    B_QTILE = B_QCOPIED + 1,             // q dims 384-575 landed in the shared-memory q tile (+tx)
    B_KCONV = B_QTILE + 1,               // fp8: + page parity: K stage converted to bf16
    B_VCONV = B_KCONV + 2,               // fp8: + page parity: V stage converted to bf16
    B_SCEMPTY = B_VCONV + 2,             // fp8: + page mod 4: the softmax is done with the scales
    B_COUNT = B_SCEMPTY + kScaleSlots,
};
static_assert(B_COUNT * 8 <= 512, "barrier area");

struct Params {
    CUtensorMap tm_q_lat;   // q_latent as [rows*128][512], box 64 x 128, SW128
    CUtensorMap tm_q_rope;  // q_rope   as [rows*128][64],  box 64 x 128, SW128
    // kv_cache [pages][64][576] seen as (64 dims, 64 tokens, 9 dim blocks, pages) with
    // the block stride 128 bytes: one box lands as stacked 128-byte-swizzled tiles
    // [block][token][64 dims], the layout the MMAs read
    CUtensorMap tm_k;       // box 64 x 32 x 9 x 1: a token half, all 576 dims
    CUtensorMap tm_v;       // box 64 x 64 x 4 x 1: all 64 tokens, one CTA's 256 output dims
    // fp8 cache: tm_k / tm_v are views of the e4m3 codes (128 codes, 64 tokens, 4 blocks,
    // pages; box 128 x 32 x 4 x 1 and 128 x 64 x 2 x 1), and
    CUtensorMap tm_kr;      // k_rope / s: (64 values, 64 tokens, pages), box 64 x 32 x 1, bf16
    CUtensorMap tm_ks;      // s: (4 floats, 64 tokens, pages), box 4 x 32 x 1
    const __nv_bfloat16 *q_latent;
    const int32_t *block_table;
    uint8_t *ws;
    __nv_bfloat16 *o_latent;
    float *lse;
    int64_t num_pages;
    uint64_t wait_limit_ns;
    float scale_log2;
    int32_t batch, s_q, max_pages, num_units;
    uint32_t test_flags;
    uint32_t flags;          // mla_problem.flags (MLA_FLAG_POW2_MAX)
};

struct Ctl {
    uint32_t bar0;       // shared address of barrier 0
    volatile int *abort; // shared abort flag
    int *status;         // device status word
    uint64_t limit_ns;   // a wait gives up after this long
};

__device__ __forceinline__ uint32_t bar(const Ctl &c, uint32_t i) { return c.bar0 + 8u * i; }

__device__ __forceinline__ void fail(const Ctl &c) {
    if (!*c.abort) {
        *c.abort = 1;
        atomicOr(c.status, MLA_DEV_TIMEOUT);
    }
}

// How a wait acquires: CTA scope; cluster scope, for phases that the peer
// CTA completes with data (its remote stores, its MMAs'
// commits); or not at all, for pure progress signals from the peer.
enum Scope : int { kCta = 0, kCluster = 1, kSignal = 2 };

__device__ __forceinline__ bool try_wait(uint32_t b, uint32_t parity, int scope) {
    return scope == kCta       ? mbar_try_wait(b, parity)
           : scope == kCluster ? mbar_try_wait_cluster(b, parity)
                               : mbar_try_wait_relaxed_cluster(b, parity);
}

// Bounded wait for the completion of the phase with the given parity: gives
// up (and flags the time-out) after the limit, or at once if another thread
// of the CTA already gave up.  The first probe is inline; the polling loop is
// out of line, so that the many wait sites of the page loop stay small in the
// instruction cache.
__device__ __noinline__ bool wait_slow(const Ctl c, uint32_t b, uint32_t parity, int scope) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (try_wait(b, parity, scope)) return true;
        if ((i & 255) == 255) {
            if (*c.abort) return false;
            const uint64_t t = globaltimer_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > c.limit_ns) {
                fail(c);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait(const Ctl &c, uint32_t b, uint32_t parity,
                                     int scope = kCta) {
    return try_wait(b, parity, scope) || wait_slow(c, b, parity, scope);
}

// Teardown wait that ignores the abort flag (for copies already in flight,
// which always land): bounded by the limit.
__device__ __noinline__ void wait_landed(const Ctl c, uint32_t b, uint32_t parity, int scope = kCta) {
    const uint64_t t0 = globaltimer_ns();
    while (!try_wait(b, parity, scope)) {
        if (globaltimer_ns() - t0 > c.limit_ns) {
            fail(c);
            return;
        }
    }
}

// Warp-uniform version: every lane waits (and acquires), and the warp agrees
// on the outcome, so no lane leaves a .sync.aligned sequence early.
__device__ __forceinline__ bool wait_warp(const Ctl &c, uint32_t b, uint32_t parity,
                                          int scope = kCta) {
    return __all_sync(0xffffffffu, wait(c, b, parity, scope));
}

// Zero the latent rows of tokens [valid, 64) of a landed V stage (the four
// 64-dim blocks of this CTA's output dims, 128-byte rows), one warp, then
// make the stores visible to the tensor cores.  Out of line: the PV issue
// loop stays small.
__device__ __noinline__ void zero_v_tail(uint8_t *vst, int valid, int lane) {
    const int per_blk = (kPage - valid) * 8;   // 16-byte chunks per dim block
    for (int idx = lane; idx < 4 * per_blk; idx += 32) {
        const int blk = idx / per_blk, rem = idx % per_blk;
        *reinterpret_cast<uint4 *>(vst + blk * kVBlk + (valid + rem / 8) * 128 + (rem % 8) * 16) =
            make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 2^k for an integer k <= 0, exactly (0 below the normal range).
__device__ __forceinline__ float pow2i(int k) {
    return k < -126 ? 0.f : __int_as_float((k + 127) << 23);
}

// The factor 2^d that moves values from one reference max to a higher one
// (d <= 0).  With power-of-two maxima (MLA_FLAG_POW2_MAX) every reference is an
// integer in log2 units, d is an integer and the factor is built exactly from
// its exponent bits, so rescaling a bf16 P row or the fp32 O accumulator is
// exact; otherwise it is ex2.approx.
__device__ __forceinline__ float fast_exp2(float x);
__device__ __forceinline__ float rescale(float d, bool pow2) {
    return pow2 ? pow2i((int)d) : fast_exp2(d);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of 16-byte chunk cc (8 tokens) of head h's row in a P half
// tile (64-byte rows, 64-byte swizzle: chunk cc of row h sits at
// cc ^ ((h >> 1) & 3)).
__device__ __forceinline__ uint32_t p_chunk(int h, int cc) {
    return (uint32_t)(h * 64 + ((cc ^ ((h >> 1) & 3)) << 4));
}

// Scale head h's 32 bf16 values in one P half tile by f.
__device__ __noinline__ void scale_p_row(uint8_t *tile, int h, float f) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        uint4 *p = reinterpret_cast<uint4 *>(tile + p_chunk(h, cc));
        uint4 v = *p;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&w[e]);
            const float2 fx = __bfloat1622float2(x);
            w[e] = pack_bf16(fx.x * f, fx.y * f);
        }
        *p = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// At an item's start q dims 0-319 (five 64-dim blocks, 128 heads each, 128-byte
// swizzle) come in by TMA through buffers that are free then: blocks 0-1 in the
// K stage that the item's second page will use (its first page loads into the
// other one meanwhile), 2-4 in the shared-memory q tile (free once this CTA's
// score MMAs of the previous item are done).  Loading q through registers costs
// one L1 wavefront per head row per instruction, and those loads delay the
// shared-memory reads of the copy into TMEM queued behind them (measured: the
// copy of four staged blocks took 2.1 us behind two register chunks, 0.4 us
// without), so only dims 320-383 take that path, overlapped.
constexpr int kQStaged = 5;
__device__ __forceinline__ uint32_t q_stage_off(int b, uint32_t kstage) {
    return b < 2 ? kOffK + kstage * kKStageBytes + b * kQBlk : kOffQS + (b - 2) * kQBlk;
}
static_assert(2 * kQBlk <= kKStageBytes && (kQStaged - 2) * kQBlk <= kQSBytes && kQStaged * 64 < kQTDims,
              "q staging");

// Head h's row of staged q block b -> TMEM columns [32 b, 32 b + 32): chunk c
// (8 dims) of row h sits at c ^ (h & 7); eight consecutive heads read eight
// different chunk positions, so the loads are free of bank conflicts.
__device__ __forceinline__ void q_stage_to_tmem(const uint8_t *smem, int b, uint32_t kstage, int h,
                                                uint32_t tq) {
    const uint8_t *row = smem + q_stage_off(b, kstage) + h * 128;
    uint32_t q[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 x = *reinterpret_cast<const uint4 *>(row + ((c ^ (h & 7)) << 4));
        q[4 * c] = x.x;
        q[4 * c + 1] = x.y;
        q[4 * c + 2] = x.z;
        q[4 * c + 3] = x.w;
    }
    tmem_st32(tq + b * 32, q);
}

// Item epilogue, one merge warp (32 heads): normalise this CTA's output half
// (the last PV is done), store it as bf16 output rows or fp32 partial rows
// and the lse, and arrive on OFREE (TMEM read) and EPI (staging done).  The
// rows go through the last page's V stage (free now: its MMAs are done and it
// is only refilled after the epilogue releases it), so that every global
// store writes 256 contiguous bytes of one row.  Out of line: once per item.
__device__ __noinline__ void item_epilogue(const Ctl ctl, __nv_bfloat16 *o_latent, float *lse_out, float *o_part,
                                           float *lse_part, PlanHeader *hdr, uint32_t lstage, uint32_t tO,
                                           const WorkItem it, bool bad, float l_run, float m_ref, int quarter,
                                           int lane, uint32_t rank) {
    const int h = quarter * 32 + lane;
    const float nan = __int_as_float(0x7fc00000);
    const float inv = bad ? nan : 1.f / l_run;
    const float lse = bad ? nan : (m_ref + log2f(l_run)) * 0.69314718055994531f;
    const uint32_t stg = lstage + quarter * 8192;   // 32 rows x 256 B (shared address)
    const uint32_t my_stg = stg + lane * 256;
    const bool final_out = it.part < 0;
    const int passes = final_out ? 2 : 4;     // 256 B of a row per pass
#pragma unroll 1
    for (int pass = 0; pass < passes; ++pass) {
        // TMEM -> normalised values -> swizzled staging row (chunk c at c ^ lane)
        if (final_out) {
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t o[32];
                tmem_ld32(tO + (pass * 4 + ch) * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 v;
                    v.x = pack_bf16(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                    v.y = pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                    v.z = pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                    v.w = pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                    const int c = ch * 4 + q;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(my_stg + ((c ^ (lane & 15)) << 4)),
                                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
                }
            }
        } else {
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t o[32];
                tmem_ld32(tO + (pass * 2 + ch) * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = ch * 8 + q;
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(my_stg + ((c ^ (lane & 15)) << 4)),
                                 "f"(__uint_as_float(o[4 * q]) * inv), "f"(__uint_as_float(o[4 * q + 1]) * inv),
                                 "f"(__uint_as_float(o[4 * q + 2]) * inv), "f"(__uint_as_float(o[4 * q + 3]) * inv)
                                 : "memory");
                }
            }
        }
        if (pass == passes - 1) {  // O fully read: the next item's PV may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ctl, B_OFREE));
        }
        __syncwarp();
        // staging -> global: two rows per step, 16 lanes x 16 B contiguous per row
        const int j = lane & 15;
#pragma unroll 4
        for (int st = 0; st < 16; ++st) {
            const int r = 2 * st + (lane >> 4);
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(stg + r * 256 + ((j ^ (r & 15)) << 4)) : "memory");
            const size_t hr = (size_t)it.row * kHeads + quarter * 32 + r;
            if (final_out) {
                reinterpret_cast<uint4 *>(o_latent + hr * kDl + rank * 256 + pass * 128)[j] = v;
            } else {
                const size_t slot = (size_t)it.part * kHeads + quarter * 32 + r;
                reinterpret_cast<uint4 *>(o_part + slot * kDl + rank * 256 + pass * 64)[j] = v;
            }
        }
        __syncwarp();
    }
    if (rank == 0) {
        if (final_out) lse_out[(size_t)it.row * kHeads + h] = lse;
        else lse_part[(size_t)it.part * kHeads + h] = lse;
    }
    if (bad && lane == 0 && rank == 0) atomicOr(&hdr->status, MLA_DEV_BAD_PAGE);
    // once every merge warp is done with the stage, release it
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(ctl, B_EPI));
}

// One converter thread's share of a stage (64 threads per stage): the stage's
// first 16 KB of latent space receives 16 KB of e4m3 codes in its upper half as
// [16 KB / (rows * 128) code blocks of 128 codes][rows tokens][128 bytes], and
// becomes [2 x that many bf16 blocks of 64 dims][rows tokens][128 bytes]; both
// are 128-byte swizzled (16-byte chunk c of a row at c ^ (row & 7)).  Thread t
// reads code rows t and t + 64 into registers, meets the other converter warp
// at named barrier `bar_id`, then writes its four bf16 rows.  rows = 2^rows_log2
// (32 for a K stage, 64 for a V stage).  One out-of-line copy serves both: the
// unrolled body inlined once per ring had pushed the kernel's instruction-cache
// hit rate to 60% (98% for the bf16 cache) and made the fp8 page loop 1.2-1.4x
// slower (measured: 4K-uniform 190 -> 150 us, long 680 -> 491 us).
__device__ __noinline__ void convert_codes(uint8_t *stage, int t, int bar_id, int rows_log2) {
    const int rows_mask = (1 << rows_log2) - 1;
    const uint8_t *codes = stage + 16384;
    uint4 x[2][8];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int R = t + 64 * rr;            // code row: block R / rows, token R % rows
        const int tok = R & rows_mask;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            x[rr][c] = *reinterpret_cast<const uint4 *>(codes + R * 128 + ((c ^ (tok & 7)) << 4));
    }
    asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int R = t + 64 * rr;
        const int b8 = R >> rows_log2, tok = R & rows_mask;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            // 16 codes = dims 16c .. 16c + 15 of code block b8 -> bf16 block 2 b8 + c / 4,
            // chunks 2 (c % 4) and 2 (c % 4) + 1 of its row
            const uint32_t w[4] = {x[rr][c].x, x[rr][c].y, x[rr][c].z, x[rr][c].w};
            uint32_t o[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // e4m3 -> f16 -> f32 -> bf16: each step exact (an e4m3 value has at
                // most 4 significant bits and lies within both formats' normal range)
                const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] & 0xFFFFu), __NV_E4M3);
                const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[q] >> 16), __NV_E4M3);
                const float2 flo = __half22float2(__half2(lo));
                const float2 fhi = __half22float2(__half2(hi));
                o[2 * q] = pack_bf16(flo.x, flo.y);
                o[2 * q + 1] = pack_bf16(fhi.x, fhi.y);
            }
            uint8_t *row = stage + ((2 * b8 + c / 4) << (rows_log2 + 7)) + tok * 128;
            const int cb = 2 * (c % 4);
            *reinterpret_cast<uint4 *>(row + ((cb ^ (tok & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(row + (((cb + 1) ^ (tok & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
    }
}

template <bool kFp8>
__global__ void __launch_bounds__(kFp8 ? kThreadsFp8 : kThreads, 1)
mla_main_tc_kernel(const __grid_constant__ Params P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_qs = s_base + kOffQS;
    const uint32_t s_k = s_base + kOffK;
    const uint32_t s_v = s_base + kOffV;
    const uint32_t s_p = s_base + kOffP;
    float *oref = reinterpret_cast<float *>(smem + kOffRef);  // [page mod kRefLag][head]
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const uint16_t peer_mask = (uint16_t)(1u << peer);
    const uint32_t unit = cluster_id_x();

    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(P.ws);
    Ctl ctl;
    ctl.bar0 = s_base + kOffBar;
    ctl.abort = &abort_flag;
    ctl.status = &hdr->status;
    ctl.limit_ns = P.wait_limit_ns;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(ctl, B_Q_FULL), 4);
        mbar_init(bar(ctl, B_QTILE), 1);
        for (int p = 0; p < 2; ++p) {
            mbar_init(bar(ctl, B_KCONV + p), 2);   // its two converter warps
            mbar_init(bar(ctl, B_VCONV + p), 2);
        }
        for (int q = 0; q < kScaleSlots; ++q) mbar_init(bar(ctl, B_SCEMPTY + q), 4);
        mbar_init(bar(ctl, B_QSTAGE), 1);
        mbar_init(bar(ctl, B_QCOPIED), 4);
        mbar_init(bar(ctl, B_Q_EMPTY), 1);
        for (int p = 0; p < 2; ++p) {
            mbar_init(bar(ctl, B_KFULL + p), 1);
            mbar_init(bar(ctl, B_KEMPTY + p), 1);
            mbar_init(bar(ctl, B_VFULL + p), 1);
            mbar_init(bar(ctl, B_VEMPTY + p), 1);
            mbar_init(bar(ctl, B_PVDONE + p), 1);
        }
        for (int s = 0; s < kPSlots; ++s) {
            mbar_init(bar(ctl, B_PEMPTY + s), 1);
            mbar_init(bar(ctl, B_PEMPTY_PEER + s), 1);
            mbar_init(bar(ctl, B_SDONE + s), 4);
            mbar_init(bar(ctl, B_PMSG + s), 1);
            mbar_init(bar(ctl, B_PREADY + s), 4);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(bar(ctl, B_SFULL + p), 1);
            mbar_init(bar(ctl, B_SEMPTY + p), 4);
        }
        for (int r = 0; r < kRefLag; ++r) mbar_init(bar(ctl, B_RESDONE + r), 4);
        mbar_init(bar(ctl, B_PVLAST), 1);
        mbar_init(bar(ctl, B_OFREE), 4);
        mbar_init(bar(ctl, B_EPI), 4);
        for (int d = 0; d < 2; ++d) mbar_init(bar(ctl, B_DRAIN + d), 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&P.tm_q_lat);
        prefetch_tmap(&P.tm_q_rope);
        prefetch_tmap(&P.tm_k);
        prefetch_tmap(&P.tm_v);
    }
    if (warp == kQkWarp) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before any multicast targets them
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // Launched as a programmatic dependent of the planner: everything above
    // overlaps its tail; the schedule and every input are read only after it.
    pdl_wait_prior();
    pdl_launch_dependents();

    const PlanLayout L = plan_layout(P.batch, P.s_q, P.num_units);
    const WorkItem *items = reinterpret_cast<const WorkItem *>(P.ws + L.items);
    const int32_t *unit_begin = reinterpret_cast<const int32_t *>(P.ws + L.unit_begin);
    float *lse_part = reinterpret_cast<float *>(P.ws + L.lse_part);
    float *o_part = reinterpret_cast<float *>(P.ws + L.o_part);
    const bool plan_ok = hdr->magic == kPlanMagic && hdr->batch == P.batch &&
                         hdr->s_q == P.s_q && hdr->num_units == P.num_units &&
                         hdr->max_pages == P.max_pages && (int)unit < P.num_units;
    int i_begin = 0, i_end = 0;
    if (plan_ok) {
        i_begin = unit_begin[unit];
        i_end = unit_begin[unit + 1];
    } else if (threadIdx.x == 0 && rank == 0) {
        atomicOr(&hdr->status, MLA_DEV_BAD_PLAN);
    }
    const int tok_own = kHalfTok * (int)rank;
    const bool pow2 = (P.flags & MLA_FLAG_POW2_MAX) != 0;   // power-of-two running maxima

    if (warp == 0 || warp == kVWarp) {
        // ------------------------------------------------------------ TMA producers
        // Warp 0: K ring (this CTA's tokens, all dims) and q; warp 2: V ring
        // (both token halves of this CTA's output dims).  Out-of-pool page
        // indices read zeros (TMA bounds fill); the merge warps flag the row.
        const bool kring = warp == 0;
        // injected stall (mla_decode_diag): rank 0 of the unit that runs the schedule's
        // first item never loads its second K stage
        const bool withhold = kring && (P.test_flags & MLA_INJECT_WITHHOLD_K_LOAD) && i_begin == 0 &&
                              i_end > 0 && rank == 0;
        uint32_t g = 0, issued = 0;
        int q_stage_par = -1, q_tile_par = -1;   // parity of the last q copies issued
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const WorkItem it = items[i];
            const int b = it.row / P.s_q;
            const int p0 = it.kv_begin / kPage;
            const int n = (it.kv_end - it.kv_begin + kPage - 1) / kPage;
            const uint32_t ii = (uint32_t)(i - i_begin);
            const int32_t *bt = P.block_table + (size_t)b * P.max_pages + p0;
            for (int k0 = 0; k0 < n && ok; k0 += 32) {
                const int mine = k0 + lane < n ? bt[k0 + lane] : 0;
                const int ahead = k0 + lane + kPrefetch < n ? bt[k0 + lane + kPrefetch] : 0;
                const int cnt = min(32, n - k0);
                for (int kk = 0; kk < cnt; ++kk, ++g) {
                    const int page = __shfl_sync(0xffffffffu, mine, kk);
                    const int page_ahead = __shfl_sync(0xffffffffu, ahead, kk);
                    const uint32_t p = g & 1;
                    if (kring) {
                        if (k0 + kk == 0) {
                            // Item start: this CTA's score MMAs of the previous item are
                            // done, so the K stage of this item's second page and the
                            // shared-memory q tile are free.  Stage q dims 0-319 there
                            // (see q_stage_off) beside this page's K load; this item's
                            // q dims 384-575 follow once the softmax warps moved the
                            // staged blocks into TMEM.
                            if (ii > 0 && !wait_warp(ctl, bar(ctl, B_Q_EMPTY), (ii - 1) & 1)) {
                                ok = false;
                                break;
                            }
                            if (lane == 0) {
                                const uint32_t fq = bar(ctl, B_QSTAGE);
                                mbar_arrive_expect_tx(fq, kQStaged * kQBlk);
                                for (int b = 0; b < kQStaged; ++b)
                                    tma_load_2d(s_base + q_stage_off(b, p ^ 1), &P.tm_q_lat, 64 * b,
                                                it.row * kHeads, fq);
                            }
                            q_stage_par = (int)(ii & 1);
                        }
                        if (g >= 2 && !wait_warp(ctl, bar(ctl, B_KEMPTY + p), ((g >> 1) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        if (kFp8 && g >= (uint32_t)kScaleSlots &&
                            !wait_warp(ctl, bar(ctl, B_SCEMPTY + g % kScaleSlots), ((g / kScaleSlots) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0 && !(withhold && g == 1)) {
                            // one 36 KB box: an SM ingests a few large TMA copies much
                            // faster than many 4 KB ones
                            const uint32_t fa = bar(ctl, B_KFULL + p);
                            if constexpr (kFp8) {
                                // the codes (16 KB) into the upper half of the stage's latent
                                // blocks, k_rope / s (4 KB) into its place (the converter
                                // warps expand the codes downward), the tokens' scales into
                                // the ring (its slot was freed above)
                                mbar_arrive_expect_tx(fa, 4 * kBox + kBox + kScaleStage);
                                tma_load_4d(s_k + p * kKStageBytes + 4 * kBox, &P.tm_k, 0, tok_own, 0, page, fa);
                                tma_load_3d(s_k + p * kKStageBytes + 8 * kBox, &P.tm_kr, 0, tok_own, page, fa);
                                tma_load_3d(s_base + kOffScale + (g % kScaleSlots) * kScaleStage, &P.tm_ks, 0,
                                            tok_own, page, fa);
                            } else {
                                mbar_arrive_expect_tx(fa, kKStageBytes);
                                tma_load_4d(s_k + p * kKStageBytes, &P.tm_k, 0, tok_own, 0, page, fa);
                            }
                        }
                        issued = g + 1;
                        if (k0 + kk == 0) {
                            if (!wait_warp(ctl, bar(ctl, B_QCOPIED), ii & 1)) {
                                ok = false;
                                break;
                            }
                            if (lane == 0) {
                                const uint32_t fb = bar(ctl, B_QTILE);
                                mbar_arrive_expect_tx(fb, kQSBytes);
                                const int y = it.row * kHeads;
                                for (int b = 0; b < kQSBlocks; ++b) {
                                    const int dim = kQTDims + 64 * b;
                                    if (dim < kDl) tma_load_2d(s_qs + b * kQBlk, &P.tm_q_lat, dim, y, fb);
                                    else tma_load_2d(s_qs + b * kQBlk, &P.tm_q_rope, dim - kDl, y, fb);
                                }
                                q_tile_par = (int)(ii & 1);
                                // warm L2 for the next item's q
                                if (i + 1 < i_end) {
                                    for (int b = 0; b < kDl / 64; ++b)
                                        tma_prefetch_2d(&P.tm_q_lat, 64 * b, items[i + 1].row * kHeads);
                                    tma_prefetch_2d(&P.tm_q_rope, 0, items[i + 1].row * kHeads);
                                }
                            }
                        }
                        // warm L2 for a page beyond the ones in flight (each CTA warms
                        // its own token half, which the peer's V ring reads as well)
                        if (lane == 0 && k0 + kk + kPrefetch < n)
                            tma_prefetch_4d(&P.tm_k, 0, tok_own, 0, page_ahead);
                    } else {
                        if (g >= 2 && !wait_warp(ctl, bar(ctl, B_VEMPTY + p), ((g >> 1) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            const uint32_t fv = bar(ctl, B_VFULL + p);
                            if constexpr (kFp8) {
                                // the codes of this CTA's 256 output dims (16 KB) into the upper
                                // half of the stage (the scales came with the page's K load)
                                mbar_arrive_expect_tx(fv, kVStageBytes / 2);
                                tma_load_4d(s_v + p * kVStageBytes + kVStageBytes / 2, &P.tm_v, 0, 0, 2 * (int)rank,
                                            page, fv);
                            } else {
                                mbar_arrive_expect_tx(fv, kVStageBytes);
                                tma_load_4d(s_v + p * kVStageBytes, &P.tm_v, 0, 0, 4 * (int)rank, page, fv);
                            }
                        }
                        issued = g + 1;
                    }
                    __syncwarp();
                }
            }
        }
        // on a time-out, the copies in flight land before the CTA may exit (each stage's
        // last load; a load always completes)
        if (__any_sync(0xffffffffu, *ctl.abort != 0)) {
            if (lane == 0) {
                const uint32_t full = kring ? B_KFULL : B_VFULL;
                for (uint32_t q = issued > 2 ? issued - 2 : 0; q < issued; ++q)
                    if (!(withhold && q == 1)) wait_landed(ctl, bar(ctl, full + (q & 1)), (q >> 1) & 1);
                if (q_stage_par >= 0) wait_landed(ctl, bar(ctl, B_QSTAGE), (uint32_t)q_stage_par);
                if (q_tile_par >= 0) wait_landed(ctl, bar(ctl, B_QTILE), (uint32_t)q_tile_par);
            }
            __syncwarp();
        }
    } else if (warp == kQkWarp || warp == kPvWarp) {
        // ------------------------------------------------------------ MMA issuers
        // The whole warp runs the schedule and waits; one elected lane issues.
        const bool qk = warp == kQkWarp;
        // Descriptor bases; every MMA below adds a byte offset (>> 4).
        const uint64_t d_qs = smem_desc(s_qs, 16, 1024, 2);
        const uint64_t d_k = smem_desc(s_k, 16, 1024, 2);
        const uint64_t d_p = smem_desc(s_p, 16, 512, 4);   // P halves: 64-byte swizzle
        const uint64_t d_v = smem_desc(s_v, kVBlk, 1024, 2);  // MN-major: dim blocks kVBlk apart
        constexpr uint32_t id_qk = idesc_bf16(128, kHalfTok, 0, 0);
        constexpr uint32_t id_pv = idesc_bf16(128, 256, 0, 1);
        const uint32_t tQ = tmem + kColQ, tO = tmem + kColO, tS = tmem + kColS;
        uint32_t g = 0;
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const WorkItem it = items[i];
            const int n = (it.kv_end - it.kv_begin + kPage - 1) / kPage;
            const uint32_t ii = (uint32_t)(i - i_begin);
            if (qk && (!wait_warp(ctl, bar(ctl, B_Q_FULL), ii & 1) || !wait_warp(ctl, bar(ctl, B_QTILE), ii & 1)))
                break;
            for (int k = 0; k < n && ok; ++k, ++g) {
                const uint32_t p = g & 1;
                if (qk) {
                    // S = q . k_own^T into the score buffer of the page's parity, once
                    // the softmax has read the scores of page g - 2 from it
                    const uint32_t ko = p * kKStageBytes;
                    const uint32_t tSp = tS + kHalfTok * p;
                    // (fp8: the stage is read once the converter warps turned its codes into bf16)
                    if (!wait_warp(ctl, bar(ctl, (kFp8 ? B_KCONV : B_KFULL) + p), (g >> 1) & 1)) { ok = false; break; }
                    if (g >= 2 && !wait_warp(ctl, bar(ctl, B_SEMPTY + p), ((g >> 1) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (elect_one()) {
                        constexpr int kTs = kQTDims / 16;   // k-steps with q in TMEM
#pragma unroll
                        for (int ks = 0; ks < kTs; ++ks)
                            mma_ts(tSp, tQ + 8 * ks,
                                   d_k + (uint64_t)((ko + (ks >> 2) * kBox + (ks & 3) * 32) >> 4),
                                   id_qk, ks > 0 ? 1u : 0u);
#pragma unroll
                        for (int ks = kTs; ks < 36; ++ks)
                            mma_ss(tSp, d_qs + (uint64_t)((((ks - kTs) >> 2) * kQBlk + (ks & 3) * 32) >> 4),
                                   d_k + (uint64_t)((ko + (ks >> 2) * kBox + (ks & 3) * 32) >> 4),
                                   id_qk, 1u);
                        mma_commit(bar(ctl, B_SFULL + p));
                        mma_commit(bar(ctl, B_KEMPTY + p));
                    }
                    __syncwarp();
                } else {
                    // O_c (+)= [P_0 | P_1] . V_c once the V stage landed and the merge
                    // warps released the P slot
                    const uint32_t ps = g % kPSlots, pu = g / kPSlots;
                    const uint32_t vo = p * kVStageBytes, po = ps * kPSlotBytes;
                    if (!wait_warp(ctl, bar(ctl, (kFp8 ? B_VCONV : B_VFULL) + p), (g >> 1) & 1) ||
                        !wait_warp(ctl, bar(ctl, B_PREADY + ps), pu & 1)) {
                        ok = false;
                        break;
                    }
                    if (k == 0 && ii > 0 && !wait_warp(ctl, bar(ctl, B_OFREE), (ii - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    // the masked tail's latent rows in the V stage become zeros, so that
                    // 0 * garbage stays 0 in PV (the stage has landed: waited above)
                    if (k == n - 1) {
                        const int valid_last = it.kv_end - (it.kv_begin + (n - 1) * kPage);
                        if (valid_last < kPage) zero_v_tail(smem + kOffV + p * kVStageBytes, valid_last, lane);
                    }
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ss(tO, d_p + (uint64_t)((po + (ks >> 1) * kPPart + (ks & 1) * 32) >> 4),
                                   d_v + (uint64_t)((vo + ks * 2048) >> 4), id_pv,
                                   (k == 0 && ks == 0) ? 0u : 1u);
                        mma_commit(bar(ctl, B_PVDONE + p));
                        mma_commit(bar(ctl, B_PEMPTY + ps));
                        mma_commit_to(bar(ctl, B_PEMPTY_PEER + ps), peer_mask);
                        // the last page's V stage is released by the epilogue, which
                        // stages the output through it
                        if (k != n - 1)
                            mma_commit(bar(ctl, B_VEMPTY + p));
                        else
                            mma_commit(bar(ctl, B_PVLAST));
                    }
                    __syncwarp();
                }
            }
            // the score issuer is done with the item's q
            if (ok && qk) {
                if (elect_one()) mma_commit(bar(ctl, B_Q_EMPTY));
                __syncwarp();
            }
        }
        // wind down: every MMA this warp issued completes before TMEM is freed
        if (elect_one()) {
            const uint32_t drain = bar(ctl, B_DRAIN + (qk ? 0 : 1));
            mma_commit(drain);
            wait_landed(ctl, drain, 0);
        }
        __syncwarp();
    } else if (warp >= kSoftmaxWarp0 && warp < kMergeWarp0) {
        // ------------------------------------------------------------ softmax warps
        // One thread per head (TMEM lane); this CTA's 32 tokens of each page.
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tQ = tmem + lane_off + kColQ;
        const float NEG_INF = -INFINITY;
        uint32_t g = 0;
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const WorkItem it = items[i];
            const int n = (it.kv_end - it.kv_begin + kPage - 1) / kPage;
            const int valid_last = it.kv_end - (it.kv_begin + (n - 1) * kPage);
            const uint32_t ii = (uint32_t)(i - i_begin);

            // q of this head -> TMEM: dims 0-319 from the staged blocks (the
            // staging was issued after the previous item's score MMAs were done, into
            // the K stage of the item's second page and the q tile), dims 320-383
            // through registers
            {
                constexpr int kRegChunks = kQTDims / 64 - kQStaged;
                const uint4 *src = reinterpret_cast<const uint4 *>(P.q_latent + ((size_t)it.row * kHeads + h) * kDl) +
                                   kQStaged * 8;
                uint4 x[8 * kRegChunks];
#pragma unroll
                for (int v = 0; v < 8 * kRegChunks; ++v) x[v] = src[v];
                if (!wait_warp(ctl, bar(ctl, B_QSTAGE), ii & 1)) break;
                tc_fence_after();
#pragma unroll 1
                for (int b = 0; b < kQStaged; ++b) q_stage_to_tmem(smem, b, (g & 1) ^ 1u, h, tQ);
                // the staging buffers may be refilled: every read above has returned
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ctl, B_QCOPIED));
#pragma unroll
                for (int c = 0; c < kRegChunks; ++c) {
                    uint32_t q[32];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        q[4 * v] = x[c * 8 + v].x;
                        q[4 * v + 1] = x[c * 8 + v].y;
                        q[4 * v + 2] = x[c * 8 + v].z;
                        q[4 * v + 3] = x[c * 8 + v].w;
                    }
                    tmem_st32(tQ + (kQStaged + c) * 32, q);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ctl, B_Q_FULL));
            float m_prev = NEG_INF;   // max used for this half's previous page
            float l_own = 0.f;        // row sum of this half's tokens so far, relative to m_prev
            for (int k = 0; k < n; ++k, ++g) {
                const uint32_t ps = g % kPSlots;
                // Start from the pair's agreed max of kRefLag pages back (a fixed
                // point in the schedule, so the result does not depend on timing;
                // far enough back that the merge chain never stalls this loop).  The
                // wait is taken on every page so that no phase of the barrier is
                // skipped.
                float base = m_prev;
                if (g >= (uint32_t)kRefLag) {
                    const uint32_t slot = g % kRefLag;
                    if (!wait_warp(ctl, bar(ctl, B_RESDONE + slot), ((g / kRefLag) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    if (k >= kRefLag) base = fmaxf(base, oref[slot * 128 + h]);
                }
                const uint32_t sp = g & 1;
                if (!wait_warp(ctl, bar(ctl, B_SFULL + sp), (g >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + kColS + kHalfTok * sp, r);
                tmem_wait_ld();
                // the scores are in registers: the score MMAs of page g + 2 may start
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ctl, B_SEMPTY + sp));

                const int valid = (k == n - 1) ? valid_last : kPage;
                const int v_own = min(max(valid - tok_own, 0), kHalfTok);
                // fp8 cache: the score MMAs contracted q with the codes and k_rope / s, so
                // each token's raw score is multiplied by its scale s (> 0)
                const float *tsc = reinterpret_cast<const float *>(smem + kOffScale + (g % kScaleSlots) * kScaleStage);
                if constexpr (kFp8) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * tsc[4 * j]);
                }
                // scores in log2 units are r * scale_log2 (scale > 0, so the max of
                // the raw scores gives the max); masked tokens (ragged last page)
                // are -inf
                const float sc = P.scale_log2;
                float rmax = NEG_INF;
                if (v_own == kHalfTok) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) rmax = fmaxf(rmax, __uint_as_float(r[j]));
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j >= v_own) r[j] = __float_as_uint(NEG_INF);
                        rmax = fmaxf(rmax, __uint_as_float(r[j]));
                    }
                }
                const float lm = rmax * sc;
                // raise the max only when this half's page exceeds it by > 2^8
                // (with power-of-two maxima a raised max is rounded up to an integer, so
                // that every later rescale is by an exact power of two)
                const float m_used = (lm - base > kRescaleThreshold) ? (pow2 ? ceilf(lm) : lm) : base;
                const float l_scale = m_prev == NEG_INF ? 0.f : (m_used == m_prev ? 1.f : rescale(m_prev - m_used, pow2));
                m_prev = m_used;
                const float mu = m_used == NEG_INF ? 0.f : m_used;
                uint32_t pk[16];
                float rsum = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float e0 = fast_exp2(fmaf(__uint_as_float(r[2 * j]), sc, -mu));
                    const float e1 = fast_exp2(fmaf(__uint_as_float(r[2 * j + 1]), sc, -mu));
                    rsum += e0 + e1;
                    if constexpr (kFp8) {
                        // PV contracts with the codes: each weight carries its token's
                        // scale (masked tokens stay 0 whatever their scale slot holds)
                        pk[j] = pack_bf16(2 * j < v_own ? e0 * tsc[8 * j] : 0.f,
                                          2 * j + 1 < v_own ? e1 * tsc[8 * j + 4] : 0.f);
                    } else {
                        pk[j] = pack_bf16(e0, e1);
                    }
                }
                // the scales of this page are no longer needed
                if constexpr (kFp8) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(ctl, B_SCEMPTY + g % kScaleSlots));
                }
                l_own = l_own * l_scale + rsum;
                // the P slot is free in both CTAs once PV of page g - kPSlots is done
                if (g >= (uint32_t)kPSlots &&
                    (!wait_warp(ctl, bar(ctl, B_PEMPTY + ps), ((g / kPSlots) - 1) & 1) ||
                     !wait_warp(ctl, bar(ctl, B_PEMPTY_PEER + ps), ((g / kPSlots) - 1) & 1, kSignal))) {
                    ok = false;
                    break;
                }
                // this half's P row and (max, row sum) -> this CTA's P slot, and the
                // same bytes into the peer's (its P slot is free: waited above)
                uint8_t *pst = smem + kOffP + ps * kPSlotBytes;
                const uint32_t part = ps * kPSlotBytes + rank * kPPart;
                const uint32_t peer_part = mapa(s_p + part, peer);
                const uint32_t peer_msg = mapa(bar(ctl, B_PMSG + ps), peer);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const uint4 v = make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                    *reinterpret_cast<uint4 *>(pst + rank * kPPart + p_chunk(h, cc)) = v;
                    st_async_v4(peer_part + p_chunk(h, cc), v, peer_msg);
                }
                *reinterpret_cast<float2 *>(pst + rank * kPPart + kPHalf + h * 8) = make_float2(m_used, l_own);
                st_async_v2f(peer_part + kPHalf + h * 8, m_used, l_own, peer_msg);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ctl, B_SDONE + ps));
            }
        }
    } else if (warp < kMergeWarp0 + 4) {
        // ------------------------------------------------------------ merge + epilogue warps
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + kColO;
        const float NEG_INF = -INFINITY;
        uint32_t g = 0;
        bool ok = true;
        // warp 8 arms the receive barrier of each page (armed: pages armed so far;
        // merged: pages merged so far)
        uint32_t armed = 0, merged = 0, total_pages = 0;
        for (int i = i_begin; i < i_end; ++i)
            total_pages += (uint32_t)((items[i].kv_end - items[i].kv_begin + kPage - 1) / kPage);
        for (int i = i_begin; i < i_end && ok; ++i) {
            const WorkItem it = items[i];
            const int b = it.row / P.s_q;
            const int p0 = it.kv_begin / kPage;
            const int n = (it.kv_end - it.kv_begin + kPage - 1) / kPage;
            const uint32_t ii = (uint32_t)(i - i_begin);
            // every page of the item must lie in the pool
            bool bad = false;
            for (int k0 = 0; k0 < n; k0 += 32) {
                int pg = k0 + lane < n ? P.block_table[(size_t)b * P.max_pages + p0 + k0 + lane] : 0;
                bad |= __any_sync(0xffffffffu, pg < 0 || (int64_t)pg >= P.num_pages);
            }
            // Per page, once both halves are in the slot, merge them: agree on the
            // max per head (a half computed against a lower
            // one is scaled; O is rescaled when the agreed max grows), publish it
            // for the softmax kRefLag pages on and release the P slot to the PV
            // warp.  Each half's message carries its running row sum, so the sums
            // are combined once, at the last page.
            float m_ref = NEG_INF, l_run = 0.f;
            for (int k = 0; k < n; ++k) {
                const uint32_t gp = g + k, par = gp & 1, ps = gp % kPSlots, pu = gp / kPSlots;
                if (warp == kMergeWarp0) {
                    // this page's receive phase: its previous phase (page gp - kPSlots)
                    // completed before this warp merged that page; bytes that land
                    // before the arming are counted against it
                    if (elect_one()) mbar_arrive_expect_tx(bar(ctl, B_PMSG + ps), kMsgBytes);
                    __syncwarp();
                    armed = gp + 1;
                }
                if (!wait_warp(ctl, bar(ctl, B_SDONE + ps), pu & 1) ||
                    !wait_warp(ctl, bar(ctl, B_PMSG + ps), pu & 1, kCluster)) {
                    ok = false;
                    break;
                }
                uint8_t *pst = smem + kOffP + ps * kPSlotBytes;
                const float2 h0 = *reinterpret_cast<const float2 *>(pst + kPHalf + h * 8);
                const float2 h1 = *reinterpret_cast<const float2 *>(pst + kPPart + kPHalf + h * 8);
                const float nref = fmaxf(m_ref, fmaxf(h0.x, h1.x));   // finite: token 0 is valid
                if (h0.x != NEG_INF && h0.x < nref) scale_p_row(pst, h, rescale(h0.x - nref, pow2));
                if (h1.x != NEG_INF && h1.x < nref) scale_p_row(pst + kPPart, h, rescale(h1.x - nref, pow2));
                // O is rescaled (rarely) once the previous PV is done
                const bool need = k > 0 && nref > m_ref;
                if (__any_sync(0xffffffffu, need)) {
                    if (!wait_warp(ctl, bar(ctl, B_PVDONE + (par ^ 1)), ((gp - 1) >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float a = need ? rescale(m_ref - nref, pow2) : 1.f;
#pragma unroll 1
                    for (int ch = 0; ch < 8; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + ch * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * a);
                        tmem_st32(tO + ch * 32, o);
                    }
                    tmem_wait_st();
                }
                m_ref = nref;
                oref[(gp % kRefLag) * 128 + h] = m_ref;
                if (k == n - 1) {
                    // both halves' row sums, relative to the final max (same order in both CTAs)
                    const float f0 = h0.x == NEG_INF ? 0.f : (h0.x == nref ? 1.f : rescale(h0.x - nref, pow2));
                    const float f1 = h1.x == NEG_INF ? 0.f : (h1.x == nref ? 1.f : rescale(h1.x - nref, pow2));
                    l_run = h0.y * f0 + h1.y * f1;
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(ctl, B_RESDONE + gp % kRefLag));
                    mbar_arrive(bar(ctl, B_PREADY + ps));
                }
                merged = gp + 1;
            }
            g += n;
            if (!ok) break;

            // epilogue: wait for the last PV, normalise, store this CTA's half.  The
            // rows go through the last page's V stage (free now: its MMAs are done
            // and it is only refilled after this epilogue releases it) so that every
            // global store writes 256 contiguous bytes of one row.
            if (!wait_warp(ctl, bar(ctl, B_PVLAST), ii & 1)) break;
            tc_fence_after();
            const uint32_t p_last = (g - 1) & 1;
            item_epilogue(ctl, P.o_latent, P.lse, o_part, lse_part, hdr, s_base + kOffV + p_last * kVStageBytes, tO,
                          it, bad, l_run, m_ref, quarter, lane, rank);
            if (warp == kMergeWarp0) {
                if (!wait_warp(ctl, bar(ctl, B_EPI), ii & 1)) break;
                if (lane == 0) mbar_arrive(bar(ctl, B_VEMPTY + p_last));
            }
        }
        // After a time-out, the peer may have stored halves of up to kPSlots pages
        // past the last one merged here (its softmax waits for this CTA's PV of
        // page g - kPSlots before it stores page g): wait (bounded) until those
        // that were sent have landed, so that no remote store reaches this CTA's
        // shared memory after it exits.
        if (warp == kMergeWarp0 && __any_sync(0xffffffffu, *ctl.abort != 0)) {
            if (lane == 0) {
                for (uint32_t q = merged; q < merged + kPSlots && q < total_pages; ++q) {
                    const uint32_t b = bar(ctl, B_PMSG + q % kPSlots);
                    if (q >= armed) mbar_arrive_expect_tx(b, kMsgBytes);
                    wait_landed(ctl, b, (q / kPSlots) & 1, kCluster);
                }
            }
            __syncwarp();
        }
    } else if constexpr (kFp8) {
        // ------------------------------------------------------------ fp8 -> bf16 converters
        // Warps 12-13 expand each landed K stage, warps 14-15 each V stage, in place:
        // the codes sit in the upper half of the stage's latent blocks; every thread
        // reads its two 128-byte code rows, the pair of warps meets at a named barrier,
        // then writes the bf16 rows over the whole stage.  e4m3 values are exact in bf16.
        const bool kside = warp < kConvWarp0 + 2;
        const int ct = (warp - (kside ? kConvWarp0 : kConvWarp0 + 2)) * 32 + lane;   // 0..63
        uint32_t g = 0;
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const int n = (items[i].kv_end - items[i].kv_begin + kPage - 1) / kPage;
            for (int k = 0; k < n; ++k, ++g) {
                const uint32_t p = g & 1;
                if (!wait_warp(ctl, bar(ctl, (kside ? B_KFULL : B_VFULL) + p), (g >> 1) & 1)) {
                    ok = false;
                    break;
                }
                static_assert(kHalfTok == 32 && kPage == 64, "converter row counts");
                if (kside) convert_codes(smem + kOffK + p * kKStageBytes, ct, 1, 5);
                else convert_codes(smem + kOffV + p * kVStageBytes, ct, 2, 6);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ctl, (kside ? B_KCONV : B_VCONV) + p));
            }
        }
    }

    // teardown: both CTAs finish (every remote store landed, no remote arrive in
    // flight) before shared memory and TMEM are released
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == kQkWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle swz,
            CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, type, rank, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int units = 0;
    bool attr_set = false;
    int fp8 = 0;   // the fp8 variant: 0 not checked, 1 runs on the same units, -1 does not
};
std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

cudaError_t prepare(int dev, int *units) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.attr_set) {
        cudaError_t e = cudaFuncSetAttribute(mla_main_tc_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kClusterSize * (sms / kClusterSize));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = kClusterSize;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, mla_main_tc_kernel<false>, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        d.units = n;
        d.attr_set = true;
    }
    *units = d.units;
    return cudaSuccess;
}

// The fp8 variant runs the same schedule, so it must fit as many units.
cudaError_t prepare_fp8(int dev, int units) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (d.fp8 == 0) {
        cudaError_t e = cudaFuncSetAttribute(mla_main_tc_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytesFp8);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kClusterSize * units);
        cfg.blockDim = dim3(kThreadsFp8);
        cfg.dynamicSmemBytes = kSmemBytesFp8;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = kClusterSize;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, mla_main_tc_kernel<true>, &cfg);
        if (e != cudaSuccess) return e;
        d.fp8 = n >= units ? 1 : -1;
    }
    return d.fp8 == 1 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

}  // namespace

cudaError_t main_units(int32_t *units) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int u = 0;
    e = prepare(dev, &u);
    if (e != cudaSuccess) return e;
    *units = u;
    return cudaSuccess;
}

cudaError_t launch_main(const void *q_latent, const void *q_rope, const void *kv,
                        int64_t num_pages, const int32_t *block_table, float scale, void *ws,
                        void *o_latent, float *lse, int32_t batch, int32_t s_q, int32_t max_pages,
                        int32_t num_units, uint64_t wait_limit_ns, uint32_t test_flags, uint32_t flags,
                        bool fp8, cudaStream_t stream) {
    if (fp8) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = prepare_fp8(dev, num_units);
        if (e != cudaSuccess) return e;
    }
    Params p;
    const cuuint64_t qrows = (cuuint64_t)batch * s_q * kHeads;
    {
        cuuint64_t dims[2] = {(cuuint64_t)kDl, qrows};
        cuuint64_t strides[1] = {(cuuint64_t)kDl * 2};
        cuuint32_t box[2] = {64, 128};
        if (!encode(&p.tm_q_lat, q_latent, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)kDr, qrows};
        cuuint64_t strides[1] = {(cuuint64_t)kDr * 2};
        cuuint32_t box[2] = {64, 128};
        if (!encode(&p.tm_q_rope, q_rope, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (fp8) {
        // 656-byte rows: the codes as (128 codes, token, 128-code block, page), the
        // block stride (128 bytes) below the row stride; k_rope / s (bf16) at byte 512
        // and the scale (fp32) at byte 640 of each row
        const uint8_t *kv8 = static_cast<const uint8_t *>(kv);
        const cuuint64_t row = MLA_FP8_ROW_BYTES, pg = row * kPage;
        cuuint64_t dims[4] = {128, (cuuint64_t)kPage, 4, (cuuint64_t)num_pages};
        cuuint64_t strides[3] = {row, 128, pg};
        cuuint32_t box_k[4] = {128, (cuuint32_t)kHalfTok, 4, 1};
        cuuint32_t box_v[4] = {128, (cuuint32_t)kPage, 2, 1};
        cuuint64_t rdims[3] = {64, (cuuint64_t)kPage, (cuuint64_t)num_pages};
        cuuint64_t rstrides[2] = {row, pg};
        cuuint32_t rbox[3] = {64, (cuuint32_t)kHalfTok, 1};
        cuuint64_t sdims[3] = {4, (cuuint64_t)kPage, (cuuint64_t)num_pages};
        cuuint32_t sbox[3] = {4, (cuuint32_t)kHalfTok, 1};
        if (!encode(&p.tm_k, kv8, 4, dims, strides, box_k, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
            !encode(&p.tm_v, kv8, 4, dims, strides, box_v, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
            !encode(&p.tm_kr, kv8 + kDl, 3, rdims, rstrides, rbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode(&p.tm_ks, kv8 + kDl + 2 * kDr, 3, sdims, rstrides, sbox, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
            return cudaErrorInvalidValue;
    } else {
        // (dim within block, token, dim block, page); the block stride (128 bytes) is
        // below the token stride, so a box lands block-major in shared memory
        cuuint64_t dims[4] = {64, (cuuint64_t)kPage, (cuuint64_t)(kDrow / 64), (cuuint64_t)num_pages};
        cuuint64_t strides[3] = {(cuuint64_t)kDrow * 2, 128, (cuuint64_t)kDrow * 2 * kPage};
        cuuint32_t box_k[4] = {64, (cuuint32_t)kHalfTok, (cuuint32_t)(kDrow / 64), 1};
        cuuint32_t box_v[4] = {64, (cuuint32_t)kPage, 4, 1};
        if (!encode(&p.tm_k, kv, 4, dims, strides, box_k, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode(&p.tm_v, kv, 4, dims, strides, box_v, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    p.q_latent = static_cast<const __nv_bfloat16 *>(q_latent);
    p.block_table = block_table;
    p.ws = static_cast<uint8_t *>(ws);
    p.o_latent = static_cast<__nv_bfloat16 *>(o_latent);
    p.lse = lse;
    p.num_pages = num_pages;
    p.wait_limit_ns = wait_limit_ns;
    p.test_flags = test_flags;
    p.flags = flags;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.batch = batch;
    p.s_q = s_q;
    p.max_pages = max_pages;
    p.num_units = num_units;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterSize * num_units);
    cfg.blockDim = dim3(fp8 ? kThreadsFp8 : kThreads);
    cfg.dynamicSmemBytes = fp8 ? kSmemBytesFp8 : kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterSize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return fp8 ? cudaLaunchKernelEx(&cfg, mla_main_tc_kernel<true>, p)
               : cudaLaunchKernelEx(&cfg, mla_main_tc_kernel<false>, p);
}

}  // namespace mla
