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
// two CTAs on two SMs, and CTA c owns output columns [256c, 256c + 256).
// Cross-SM traffic through distributed shared memory measures only
// 10-20 GB/s per SM on this part, far too slow to exchange per-page score
// partials, so nothing is exchanged per page: each CTA computes the full
// score tile itself and the pair shares only the page loads.
//
//   page g (64 tokens x 576) -> TMA multicast: CTA 0 loads dim blocks 0-4,
//                               CTA 1 blocks 5-8, each into both CTAs
//   S   = q . k^T            tcgen05 M=128 (heads) N=64 (tokens) K=576, fp32
//                            in TMEM, as two partial sums (dims 0-287 and
//                            288-575) from two issuing warps; q dims 0-255
//                            are the A operand in TMEM, 256-575 in shared memory
//   P   = exp2(S*scale*log2e - m)    fp32 online softmax with a lazily
//                            raised running max, rounded to bf16 into two
//                            blocks of the page's stage that this CTA's PV
//                            does not read
//   O_c += P . V_c           tcgen05 M=128 N=256 K=64,
//                            B = the page's latent dims [256c, 256c + 256)
//
// TMEM (512 columns): O half [0,256), S partials [256,384), q [384,512).
// Warp roles per CTA: warp 0 issues TMA; warps 1 and 6 issue the two QK
// partial sums and warp 7 the PV product (one thread issues a tcgen05.mma
// about every 27 ns, so each chain gets its own issuer); warp 1 also owns
// TMEM; warps 2-5 and 8-11 (two per TMEM lane quarter, one thread per head
// and half of the columns) load q into TMEM and run the softmax and the
// epilogue.  Every wait is bounded: on time-out the kernel
// records MLA_DEV_TIMEOUT and winds down instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 384;       // warp 0 TMA, warps 1/6 QK MMA, 7 PV MMA, 2-5 + 8-11 softmax
constexpr int kSoftmaxWarps = 8;    // two per TMEM lane quarter, 32 score columns each
constexpr int kQkbWarp = 6;
constexpr int kPvWarp = 7;
constexpr int kStages = 2;          // KV page ring (a full page per stage)
constexpr int kPrefetch = 2;        // L2 prefetch distance in pages (one beyond the stages)
constexpr int kClusterSize = 2;
constexpr uint16_t kBoth = 0x3;     // multicast mask: both CTAs of the pair
constexpr uint32_t kBlk = 64 * 128;               // page block: 64 tokens x 64 dims (SW128)
constexpr uint32_t kStageBytes = 9 * kBlk;        // dims 0-511 latent + 512-575 rope
constexpr uint32_t kQBlk = 128 * 128;             // q block: 128 heads x 64 dims (SW128)
constexpr uint32_t kQSBytes = 5 * kQBlk;          // q dims 256-575 in shared memory
constexpr int kQTDims = 256;                      // q dims 0-255 live in TMEM
constexpr uint32_t kOffQS = 0;
constexpr uint32_t kOffStage = kQSBytes;
constexpr uint32_t kOffBar = kOffStage + kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + barriers, + alignment slack
static_assert(kOffStage % 1024 == 0 && kStageBytes % 1024 == 0, "TMA/UMMA tile alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM columns
constexpr uint32_t kColO = 0;       // 256 fp32 output columns of this CTA's half
constexpr uint32_t kColS = 256;     // 2 x 64 fp32 partial scores (dims 0-287, 288-575)
constexpr uint32_t kColQ = 384;     // 128 columns of packed bf16 q (dims 0-255)
constexpr uint32_t kTmemCols = 512;
static_assert(kColQ + kQTDims / 2 == kTmemCols, "TMEM budget");

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a wait gives up after 2 s

// barrier slots (8 bytes each) in the barrier area
enum : uint32_t {
    B_Q_FULL = 0,                   // producer (+tx) and the softmax warps (q in TMEM)
    B_Q_EMPTY = 1,                  // last QK of an item done, in both CTAs
    B_KV_FULL = 2,                  // + stage
    B_KV_EMPTY = B_KV_FULL + kStages,  // + stage; both CTAs' PVs done
    B_S_FULL = B_KV_EMPTY + kStages,
    B_S_EMPTY = B_S_FULL + 1,
    B_P_FULL = B_S_EMPTY + 1,
    B_PV_DONE = B_P_FULL + 1,
    B_O_FREE = B_PV_DONE + 1,
    B_EPI = B_O_FREE + 1,           // softmax warps done with the staged epilogue
    B_PAIR = B_EPI + 1,             // + lane quarter: both halves posted their row max
    B_PAIRL = B_PAIR + 4,           // + lane quarter: both halves posted their row sum
    B_DRAIN = B_PAIRL + 4,          // + issuer (0: QK a, 1: QK b, 2: PV)
    B_COUNT = B_DRAIN + 3,
};
static_assert(B_COUNT * 8 + 16 <= 256, "barrier area");

struct Params {
    CUtensorMap tm_q_lat;   // q_latent as [rows*128][512], box 64 x 128, SW128
    CUtensorMap tm_q_rope;  // q_rope   as [rows*128][64],  box 64 x 128, SW128
    CUtensorMap tm_kv;      // kv_cache as [pages][64][576], box 64 x 64 x 1, SW128
    const __nv_bfloat16 *q_latent;
    const int32_t *block_table;
    uint8_t *ws;
    __nv_bfloat16 *o_latent;
    float *lse;
    int64_t num_pages;
    float scale_log2;
    int32_t batch, s_q, max_pages, num_units;
};

struct Ctl {
    uint32_t bar0;       // shared address of barrier 0
    volatile int *abort; // shared abort flag
    int *status;         // device status word
};

__device__ __forceinline__ uint32_t bar(const Ctl &c, uint32_t i) { return c.bar0 + 8u * i; }

__device__ __forceinline__ void fail(const Ctl &c) {
    if (!*c.abort) {
        *c.abort = 1;
        atomicOr(c.status, MLA_DEV_TIMEOUT);
    }
}

// Bounded wait for the completion of the phase with the given parity: gives
// up (and flags the time-out) after kWaitLimitNs, or at once if another
// thread of the CTA already gave up.
__device__ __forceinline__ bool wait(const Ctl &c, uint32_t b, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(b, parity)) return true;
        if ((i & 255) == 255) {
            if (*c.abort) return false;
            const uint64_t t = globaltimer_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > kWaitLimitNs) {
                fail(c);
                return false;
            }
        }
    }
}

// Warp-uniform version: every lane waits (and acquires), and the warp agrees
// on the outcome, so no lane leaves a .sync.aligned sequence early.
__device__ __forceinline__ bool wait_warp(const Ctl &c, uint32_t b, uint32_t parity) {
    return __all_sync(0xffffffffu, wait(c, b, parity));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kThreads, 1)
mla_main_tc_kernel(const __grid_constant__ Params P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_qs = s_base + kOffQS;
    const uint32_t s_stage = s_base + kOffStage;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t unit = cluster_id_x();

    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(P.ws);
    Ctl ctl;
    ctl.bar0 = s_base + kOffBar;
    ctl.abort = &abort_flag;
    ctl.status = &hdr->status;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(ctl, B_Q_FULL), 1 + kSoftmaxWarps);
        mbar_init(bar(ctl, B_Q_EMPTY), 2 * kClusterSize);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(ctl, B_KV_FULL + s), 1);
            mbar_init(bar(ctl, B_KV_EMPTY + s), kClusterSize);
        }
        mbar_init(bar(ctl, B_S_FULL), 2);
        mbar_init(bar(ctl, B_S_EMPTY), kSoftmaxWarps);
        mbar_init(bar(ctl, B_P_FULL), kSoftmaxWarps);
        mbar_init(bar(ctl, B_PV_DONE), 1);
        mbar_init(bar(ctl, B_O_FREE), kSoftmaxWarps);
        mbar_init(bar(ctl, B_EPI), kSoftmaxWarps);
        for (int q = 0; q < 4; ++q) {
            mbar_init(bar(ctl, B_PAIR + q), 2);
            mbar_init(bar(ctl, B_PAIRL + q), 2);
        }
        for (int d = 0; d < 3; ++d) mbar_init(bar(ctl, B_DRAIN + d), 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&P.tm_q_lat);
        prefetch_tmap(&P.tm_q_rope);
        prefetch_tmap(&P.tm_kv);
    }
    if (warp == 1) {
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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        uint32_t g = 0;
        for (int i = i_begin; i < i_end && !abort_flag; ++i) {
            const WorkItem it = items[i];
            const int b = it.row / P.s_q;
            const int p0 = it.kv_begin / kPage;
            const int n = (it.kv_end - it.kv_begin + kPage - 1) / kPage;
            const uint32_t ii = (uint32_t)(i - i_begin);
            bool ok = true;
            const int kb0 = rank == 0 ? 0 : 5, kb1 = rank == 0 ? 5 : 9;  // this CTA's page blocks
            const int32_t *bt = P.block_table + (size_t)b * P.max_pages + p0;
            for (int k0 = 0; k0 < n && ok; k0 += 32) {
                const int mine = k0 + lane < n ? bt[k0 + lane] : 0;
                const int ahead = k0 + lane + kPrefetch < n ? bt[k0 + lane + kPrefetch] : 0;
                const int cnt = min(32, n - k0);
                for (int kk = 0; kk < cnt; ++kk, ++g) {
                    const int page = __shfl_sync(0xffffffffu, mine, kk);
                    const int page_ahead = __shfl_sync(0xffffffffu, ahead, kk);
                    const uint32_t s = g % kStages;
                    // the stage is free in both CTAs (our loads write into both)
                    if (g >= kStages &&
                        !wait_warp(ctl, bar(ctl, B_KV_EMPTY + s), ((g / kStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const uint32_t fb = bar(ctl, B_KV_FULL + s);
                        const uint32_t dst = s_stage + s * kStageBytes;
                        mbar_arrive_expect_tx(fb, kStageBytes);
                        // An out-of-pool page index reads zeros (TMA bounds fill);
                        // the softmax warps flag the row.
                        for (int kb = kb0; kb < kb1; ++kb)
                            tma_load_3d_mc(dst + kb * kBlk, &P.tm_kv, 64 * kb, 0, page, fb, kBoth);
                    }
                    if (k0 + kk == 0) {
                        // q dims 256-575, once the first page is on its way: both CTAs'
                        // copies must be free (last QKs of the previous item done)
                        if (ii > 0 && !wait_warp(ctl, bar(ctl, B_Q_EMPTY), (ii - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            const uint32_t fb = bar(ctl, B_Q_FULL);
                            mbar_arrive_expect_tx(fb, kQSBytes);
                            const int y = it.row * kHeads;
                            for (int j = rank == 0 ? 0 : 3; j < (rank == 0 ? 3 : 5); ++j) {
                                if (j < 4)
                                    tma_load_2d_mc(s_qs + j * kQBlk, &P.tm_q_lat, kQTDims + 64 * j, y,
                                                   fb, kBoth);
                                else
                                    tma_load_2d_mc(s_qs + j * kQBlk, &P.tm_q_rope, 0, y, fb, kBoth);
                            }
                        }
                    }
                    // warm L2 for a page beyond the two stages in flight
                    if (lane == 0 && k0 + kk + kPrefetch < n)
                        for (int kb = kb0; kb < kb1; ++kb)
                            tma_prefetch_3d(&P.tm_kv, 64 * kb, 0, page_ahead);
                    __syncwarp();
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 || warp == kQkbWarp || warp == kPvWarp) {
        // ------------------------------------------------------------ MMA issuers
        // One thread issues a tcgen05.mma about every 27 ns, so the score
        // contraction is split over two issuers with separate accumulators
        // (dims 0-287 and 288-575, summed by the softmax in a fixed order)
        // and the PV product gets a third.
        if (lane == 0) {
            const int role = warp == 1 ? 0 : (warp == kQkbWarp ? 1 : 2);
            // Descriptor bases; every MMA below adds a compile-time byte offset (>> 4).
            const uint64_t d_qs = smem_desc(s_qs, 16, 1024, 2);
            const uint64_t d_kv0 = smem_desc(s_stage, 16, 1024, 2);
            const uint64_t d_v0 = smem_desc(s_stage + 4 * rank * kBlk, 8192, 1024, 2);
            const uint64_t d_p0 = smem_desc(s_stage + (rank == 0 ? 7 : 0) * kBlk, 16, 1024, 2);
            constexpr uint32_t id_qk = idesc_bf16(128, 64, 0, 0);
            constexpr uint32_t id_pv = idesc_bf16(128, 256, 0, 1);
            const uint32_t tSa = tmem + kColS, tSb = tmem + kColS + 64, tQ = tmem + kColQ;
            const uint32_t tO = tmem + kColO;
            uint32_t g = 0;
            bool ok = true;
            for (int i = i_begin; i < i_end && ok; ++i) {
                const WorkItem it = items[i];
                const int n = (it.kv_end - it.kv_begin + kPage - 1) / kPage;
                const uint32_t ii = (uint32_t)(i - i_begin);
                if (role < 2 && !wait(ctl, bar(ctl, B_Q_FULL), ii & 1)) break;
                for (int k = 0; k < n && ok; ++k, ++g) {
                    const uint32_t s = g % kStages;
                    const uint64_t stage_off = (uint64_t)((s * kStageBytes) >> 4);
                    if (role < 2) {
                        if (!wait(ctl, bar(ctl, B_KV_FULL + s), (g / kStages) & 1)) { ok = false; break; }
                        if (g >= 1 && !wait(ctl, bar(ctl, B_S_EMPTY), (g - 1) & 1)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t kv = d_kv0 + stage_off;
                        if (role == 0) {
                            // S_a: dims 0-255 (q from TMEM) and 256-287 (q block 0, k-steps 0-1)
#pragma unroll
                            for (int ks = 0; ks < 16; ++ks)
                                mma_ts(tSa, tQ + 8 * ks,
                                       kv + (uint64_t)(((ks >> 2) * kBlk + (ks & 3) * 32) >> 4),
                                       id_qk, ks > 0 ? 1u : 0u);
#pragma unroll
                            for (int ks = 0; ks < 2; ++ks)
                                mma_ss(tSa, d_qs + (uint64_t)((ks * 32) >> 4),
                                       kv + (uint64_t)((4 * kBlk + ks * 32) >> 4), id_qk, 1u);
                        } else {
                            // S_b: dims 288-319 (q block 0, k-steps 2-3) and 320-575 (q blocks 1-4)
#pragma unroll
                            for (int ks = 2; ks < 4; ++ks)
                                mma_ss(tSb, d_qs + (uint64_t)((ks * 32) >> 4),
                                       kv + (uint64_t)((4 * kBlk + ks * 32) >> 4), id_qk,
                                       ks > 2 ? 1u : 0u);
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                mma_ss(tSb,
                                       d_qs + (uint64_t)(((1 + (j >> 2)) * kQBlk + (j & 3) * 32) >> 4),
                                       kv + (uint64_t)(((5 + (j >> 2)) * kBlk + (j & 3) * 32) >> 4),
                                       id_qk, 1u);
                        }
                        mma_commit(bar(ctl, B_S_FULL));
                        if (k == n - 1) mma_commit_mc(bar(ctl, B_Q_EMPTY), kBoth);
                    } else {
                        // O_c (+)= P . V_c, P (bf16) in two spare blocks of the page's stage
                        if (!wait(ctl, bar(ctl, B_P_FULL), g & 1)) { ok = false; break; }
                        if (k == 0 && ii > 0 && !wait(ctl, bar(ctl, B_O_FREE), (ii - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t v = d_v0 + stage_off;
                        const uint64_t pa = d_p0 + stage_off;
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ss(tO, pa + (uint64_t)((ks * 32) >> 4), v + (uint64_t)((ks * 2048) >> 4),
                                   id_pv, (k == 0 && ks == 0) ? 0u : 1u);
                        mma_commit(bar(ctl, B_PV_DONE));
                        // the last page's stage is released by the epilogue, which stages
                        // the output through it
                        if (k != n - 1) mma_commit_mc(bar(ctl, B_KV_EMPTY + s), kBoth);
                    }
                }
            }
            // wind down: every MMA this thread issued completes before TMEM is freed
            const uint32_t drain = bar(ctl, B_DRAIN + role);
            mma_commit(drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps
        // Two warps per TMEM lane quarter: `half` selects the 32 score columns
        // (tokens) and the 128 output columns a warp owns.  The two halves of
        // a row agree on the running max through a page block that is free
        // once the scores are computed.
        const int quarter = warp & 3;              // TMEM lane quarter this warp may access
        const int half = warp >= 8 ? 1 : 0;
        const int sidx = warp >= 8 ? warp - 4 : warp - 2;   // 0..7 among the softmax warps
        const int h = quarter * 32 + lane;         // head = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + kColS + 32 * half;
        const uint32_t tO = tmem + lane_off + kColO + 128 * half;
        const uint32_t tQ = tmem + lane_off + kColQ + 64 * half;
        const float NEG_INF = -INFINITY;
        uint32_t g = 0;
        bool ok = true;
        for (int i = i_begin; i < i_end && ok; ++i) {
            const WorkItem it = items[i];
            const int b = it.row / P.s_q;
            const int p0 = it.kv_begin / kPage;
            const int n = (it.kv_end - it.kv_begin + kPage - 1) / kPage;
            const int valid_last = it.kv_end - (it.kv_begin + (n - 1) * kPage);
            const uint32_t ii = (uint32_t)(i - i_begin);

            // q dims [128 half, 128 half + 128) of this head -> TMEM
            if (ii > 0 && !wait_warp(ctl, bar(ctl, B_Q_EMPTY), (ii - 1) & 1)) break;
            {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    P.q_latent + ((size_t)it.row * kHeads + h) * kDl + 128 * half);
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    uint32_t q[32];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const uint4 x = src[c * 8 + v];
                        q[4 * v] = x.x;
                        q[4 * v + 1] = x.y;
                        q[4 * v + 2] = x.z;
                        q[4 * v + 3] = x.w;
                    }
                    tmem_st32(tQ + c * 32, q);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ctl, B_Q_FULL));
            }
            // every page of the item must lie in the pool
            bool bad = false;
            for (int k0 = 0; k0 < n; k0 += 32) {
                int pg = k0 + lane < n ? P.block_table[(size_t)b * P.max_pages + p0 + k0 + lane] : 0;
                bad |= __any_sync(0xffffffffu, pg < 0 || (int64_t)pg >= P.num_pages);
            }
            float m_run = NEG_INF, l_half = 0.f;
            for (int k = 0; k < n; ++k, ++g) {
                if (!wait_warp(ctl, bar(ctl, B_S_FULL), g & 1)) { ok = false; break; }
                tc_fence_after();
                uint32_t r[32];
                {   // this half's columns of both partial sums (dims 0-287, 288-575)
                    uint32_t t[32];
                    tmem_ld32(tS, r);
                    tmem_ld32(tS + 64, t);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(t[j]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ctl, B_S_EMPTY));

                const int valid = (k == n - 1) ? valid_last : kPage;
                uint8_t *stage = smem + kOffStage + (g % kStages) * kStageBytes;
                float s[32];
                float m_half = NEG_INF;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float a = __uint_as_float(r[j]) * P.scale_log2;
                    a = 32 * half + j < valid ? a : NEG_INF;
                    s[j] = a;
                    m_half = fmaxf(m_half, a);
                }
                // row max over both halves (a block of this page the PV never reads)
                float *pm = reinterpret_cast<float *>(stage + (rank == 0 ? 4 : 2) * kBlk);
                pm[half * 128 + h] = m_half;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ctl, B_PAIR + quarter));
                if (!wait_warp(ctl, bar(ctl, B_PAIR + quarter), g & 1)) { ok = false; break; }
                const float m_loc = fmaxf(m_half, pm[(1 - half) * 128 + h]);
                // lazy rescale of the running output (the same decision in both halves)
                float alpha = 1.f;
                bool need = false;
                if (k == 0) {
                    m_run = m_loc;
                } else if (m_loc > m_run + kRescaleThreshold) {
                    alpha = fast_exp2(m_run - m_loc);
                    m_run = m_loc;
                    need = true;
                }
                // probabilities -> bf16 (registers)
                uint32_t pk[16];
                float lsum = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float e0 = fast_exp2(s[2 * j] - m_run);
                    const float e1 = fast_exp2(s[2 * j + 1] - m_run);
                    lsum += e0 + e1;
                    pk[j] = pack_bf16(e0, e1);
                }
                // PV(g-1) must be done before O is rescaled
                if (g >= 1 && !wait_warp(ctl, bar(ctl, B_PV_DONE), (g - 1) & 1)) { ok = false; break; }
                if (__any_sync(0xffffffffu, need)) {
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + ch * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        tmem_st32(tO + ch * 32, o);
                    }
                    tmem_wait_st();
                }
                l_half = l_half * alpha + lsum;
                {   // this half's 32 tokens of the P row, K-major with the 128-byte swizzle
                    uint8_t *prow = stage + (rank == 0 ? 7 : 0) * kBlk + h * 128;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int c = 4 * half + cc;
                        *reinterpret_cast<uint4 *>(prow + ((c ^ (h & 7)) << 4)) =
                            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                    }
                }
                if (valid < kPage) {
                    // zero this CTA's latent rows of the masked tail so that 0 * garbage stays 0
                    uint8_t *vbase = stage + 4 * rank * kBlk;
                    const int per_blk = (kPage - valid) * 8;  // 16-byte chunks per block
                    for (int idx = sidx * 32 + lane; idx < 4 * per_blk; idx += 32 * kSoftmaxWarps) {
                        const int blk = idx / per_blk, rem = idx % per_blk;
                        const int tok = valid + rem / 8;
                        *reinterpret_cast<uint4 *>(vbase + blk * kBlk + tok * 128 + (rem % 8) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(ctl, B_P_FULL));
            }
            if (!ok) break;

            // epilogue: wait for the last PV, normalise, store this CTA's half.  The
            // rows go through the last page's stage (free now: its QK and PV are done
            // and it is only refilled after this epilogue releases it) so that every
            // global store writes 256 contiguous bytes of one row.
            if (!wait_warp(ctl, bar(ctl, B_PV_DONE), (g - 1) & 1)) break;
            tc_fence_after();
            const uint32_t s_last = (g - 1) % kStages;
            uint8_t *lstage = smem + kOffStage + s_last * kStageBytes;
            float *pl = reinterpret_cast<float *>(lstage + 8 * kBlk);  // row sums of both halves
            pl[half * 128 + h] = l_half;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ctl, B_PAIRL + quarter));
            if (!wait_warp(ctl, bar(ctl, B_PAIRL + quarter), ii & 1)) break;
            const float l_run = pl[h] + pl[128 + h];   // the same order in both halves
            const float nan = __int_as_float(0x7fc00000);
            const float inv = bad ? nan : 1.f / l_run;
            const float lse = bad ? nan : (m_run + log2f(l_run)) * 0.69314718055994531f;
            uint8_t *stg = lstage + sidx * 8192;     // 32 rows x 256 B
            uint8_t *my_stg = stg + lane * 256;
            const bool final_out = it.part < 0;
            const int passes = final_out ? 1 : 2;    // 256 B of a row per pass
#pragma unroll 1
            for (int pass = 0; pass < passes; ++pass) {
                // TMEM -> normalised values -> swizzled staging row (chunk c at c ^ lane)
                if (final_out) {
#pragma unroll 1
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + ch * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 v;
                            v.x = pack_bf16(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                            v.y = pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                            v.z = pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                            v.w = pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                            const int c = ch * 4 + q;
                            *reinterpret_cast<uint4 *>(my_stg + ((c ^ (lane & 15)) << 4)) = v;
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
                            *reinterpret_cast<float4 *>(my_stg + ((c ^ (lane & 15)) << 4)) =
                                make_float4(__uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                                            __uint_as_float(o[4 * q + 2]) * inv, __uint_as_float(o[4 * q + 3]) * inv);
                        }
                    }
                }
                if (pass == passes - 1) {  // O fully read: the next item's PV may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(ctl, B_O_FREE));
                }
                __syncwarp();
                // staging -> global: two rows per step, 16 lanes x 16 B contiguous per row
                const int j = lane & 15;
#pragma unroll 4
                for (int st = 0; st < 16; ++st) {
                    const int r = 2 * st + (lane >> 4);
                    const uint4 v = *reinterpret_cast<const uint4 *>(stg + r * 256 + ((j ^ (r & 15)) << 4));
                    const size_t hr = (size_t)it.row * kHeads + quarter * 32 + r;
                    if (final_out) {
                        reinterpret_cast<uint4 *>(P.o_latent + hr * kDl + rank * 256 + half * 128)[j] = v;
                    } else {
                        const size_t slot = (size_t)it.part * kHeads + quarter * 32 + r;
                        reinterpret_cast<uint4 *>(o_part + slot * kDl + rank * 256 + half * 128 +
                                                  pass * 64)[j] = v;
                    }
                }
                __syncwarp();
            }
            if (rank == 0 && half == 0) {
                if (final_out) P.lse[(size_t)it.row * kHeads + h] = lse;
                else lse_part[(size_t)it.part * kHeads + h] = lse;
            }
            if (bad && lane == 0) atomicOr(&hdr->status, MLA_DEV_BAD_PAGE);
            // once every softmax warp is done with the stage, release it in both CTAs
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ctl, B_EPI));
            if (warp == 2 && !wait_warp(ctl, bar(ctl, B_EPI), ii & 1)) break;
            if (warp == 2 && lane == 0) {
                mbar_arrive(bar(ctl, B_KV_EMPTY + s_last));
                mbar_arrive_cluster(mapa(bar(ctl, B_KV_EMPTY + s_last), rank ^ 1u));
            }
        }
    }

    // teardown: both CTAs finish (no multicast or remote arrive in flight) before TMEM is freed
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
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
            const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle swz) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int units = 0;
    bool attr_set = false;
};
std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

cudaError_t prepare(int dev, int *units) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.attr_set) {
        cudaError_t e = cudaFuncSetAttribute(mla_main_tc_kernel,
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
        e = cudaOccupancyMaxActiveClusters(&n, mla_main_tc_kernel, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        d.units = n;
        d.attr_set = true;
    }
    *units = d.units;
    return cudaSuccess;
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
                        int32_t num_units, cudaStream_t stream) {
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
    {
        cuuint64_t dims[3] = {(cuuint64_t)kDrow, (cuuint64_t)kPage, (cuuint64_t)num_pages};
        cuuint64_t strides[2] = {(cuuint64_t)kDrow * 2, (cuuint64_t)kDrow * 2 * kPage};
        cuuint32_t box[3] = {64, 64, 1};
        if (!encode(&p.tm_kv, kv, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    p.q_latent = static_cast<const __nv_bfloat16 *>(q_latent);
    p.block_table = block_table;
    p.ws = static_cast<uint8_t *>(ws);
    p.o_latent = static_cast<__nv_bfloat16 *>(o_latent);
    p.lse = lse;
    p.num_pages = num_pages;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.batch = batch;
    p.s_q = s_q;
    p.max_pages = max_pages;
    p.num_units = num_units;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterSize * num_units);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
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
    return cudaLaunchKernelEx(&cfg, mla_main_tc_kernel, p);
}

}  // namespace mla
