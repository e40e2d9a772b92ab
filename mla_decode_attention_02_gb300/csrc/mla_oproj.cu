// The output projection on the tensor cores: out = o_v . W_O^T.
//
// What it computes ("Huawei Ascend servers: DeepSeek V3/R1 inference best
// practice", sections 3.2-3.3 and figures 5-9: "O Proj" follows attention;
// the 128 heads x 128 value dims = 16384 values of a token map to the hidden
// size):
//
//   out[t][n] = sum_k w_o[n][k] * o_v[t][k]        k < 16384, n < hidden
//
// GB300 design.  The weights (hidden x 16384 bf16, 235 MB at hidden 7168)
// are read once per call and dominate the bytes, so the kernel is a weight
// stream: every SM pair holds 128 output features, and its two CTAs (a
// cluster) take one half of K each.
//  - Per CTA: D[n][t] = W[n0 .. n0+127][k half] . o_v[t][k half]^T, M=128
//    features, N = the token tile (a multiple of 64, up to 256; rows past the
//    last token read zeros), K = 8192 in 128 blocks of 64 values.  Warp 0
//    streams the weight blocks (16 KB each) and the token blocks through a
//    ring of TMA stages of one to four K blocks (two copies per stage: an SM
//    takes in a few large TMA copies much faster than many small ones; each
//    copy lands as one 128-byte-swizzled tile per K block, both operands
//    K-major); warp 1 issues four tcgen05.mma (K=16) per K block into TMEM
//    and frees each stage with tcgen05.commit.
//  - The two halves of the sum meet in shared memory: each CTA owns half of
//    the token columns, sends its partial of the other half to the peer with
//    st.async (completing on the peer's mbarrier), adds the peer's partial to
//    its own, rounds to bf16 and stores its rows of `out` (32 consecutive
//    features of one token per warp instruction).  fp32 addition commutes, so
//    the result does not depend on which CTA adds.
// Every wait is bounded: on time-out the kernel ORs MLA_DEV_TIMEOUT into the
// caller's status word and leaves its tile unwritten.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "mla_epilog.h"
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
bool encode_bf16_kblocks(CUtensorMap *m, const void *base, cuuint64_t cols, cuuint64_t rows,
                         cuuint32_t box_rows, cuuint32_t box_blocks);
namespace {
using namespace ptx;

constexpr int kOpK = MLA_NUM_HEADS * MLA_D_V;   // 16384 values per token
constexpr int kOpKHalf = kOpK / 2;              // per CTA of the pair
constexpr int kOpKBlocks = kOpKHalf / 64;       // 64-value K blocks per CTA
constexpr int kOpThreads = 128;
constexpr int kOpTileN = 128;                   // output features per pair (MMA M)
constexpr int kOpMaxTok = 256;                  // tokens per tile (MMA N)
constexpr uint32_t kOpWBlock = kOpTileN * 128;  // one K block of the weight tile: 128 rows x 128 B
constexpr int kOpMaxStages = 8;
constexpr uint32_t kOpSmemMax = 232448 - 2048;  // dynamic budget, less static shared memory
constexpr uint64_t kOpWaitLimitNs = 2000000000ull;
static_assert(kOpK % 128 == 0, "two K halves of whole 64-value blocks");

struct OprojParams {
    CUtensorMap tm_w;    // w_o as (64 values, hidden, 256 K blocks), box 64 x 128 x kb
    CUtensorMap tm_x;    // o_v as (64 values, tokens, 256 K blocks), box 64 x npad x kb
    __nv_bfloat16 *out;  // [tokens][hidden]
    int32_t *status;
    int32_t tokens, hidden, npad, stages, kb;   // kb: K blocks per stage (1, 2 or 4)
};

__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// Bounded wait; cluster scope where the peer completes the phase.
__device__ __noinline__ bool op_wait(uint32_t bar, uint32_t parity, bool cluster, int32_t *status) {
    const uint64_t t0 = globaltimer_ns();
    while (!(cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))) {
        if (globaltimer_ns() - t0 > kOpWaitLimitNs) {
            atomicOr(status, MLA_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ uint32_t bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kOpThreads, 1)
mla_epilog_oproj_kernel(const __grid_constant__ OprojParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kOpMaxStages + 4];   // full[s], empty[s], done, ready, recv, drain
    __shared__ uint32_t tmem_slot;
    __shared__ int32_t abort_tile;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int n0 = (int)(blockIdx.x / 2) * kOpTileN;
    const int t0 = (int)blockIdx.y * kOpMaxTok;
    const int S = P.stages, npad = P.npad, half = npad / 2, KB = P.kb, nst = kOpKBlocks / KB;
    const uint32_t x_block = (uint32_t)npad * 128;                 // one K block of the token tile
    const uint32_t w_bytes = KB * kOpWBlock;
    const uint32_t stage_bytes = KB * (kOpWBlock + x_block);
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    // the peer's partial of this CTA's token half, after the ring is drained:
    // [128 features][half fp32 + 4 of padding] (the padding spreads the rows over the banks)
    const uint32_t recv_stride = (uint32_t)(half + 4) * 4;
    auto full = [&](int s) { return smem_u32(&bars[s]); };
    auto empty = [&](int s) { return smem_u32(&bars[kOpMaxStages + s]); };
    const uint32_t b_done = smem_u32(&bars[2 * kOpMaxStages]);
    const uint32_t b_ready = smem_u32(&bars[2 * kOpMaxStages + 1]);   // the peer may send (its ring is drained)
    const uint32_t b_recv = smem_u32(&bars[2 * kOpMaxStages + 2]);    // the peer's partial landed (+tx)
    const uint32_t b_drain = smem_u32(&bars[2 * kOpMaxStages + 3]);
    const uint32_t tmem_cols = npad <= 64 ? 64u : npad <= 128 ? 128u : 256u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(b_done, 1);
        mbar_init(b_ready, 1);
        mbar_init(b_recv, 1);
        mbar_init(b_drain, 1);
        fence_mbar_init();
        abort_tile = 0;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // the peer's barriers are initialised before any remote arrive or store
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_wait_prior();
    pdl_launch_dependents();

    const int kb0 = (int)rank * kOpKBlocks;   // this CTA's first K block
    if (warp == 0) {
        if (elect_one()) {   // producer: the weight block and the token block of each K block
            prefetch_tmap(&P.tm_w);
            prefetch_tmap(&P.tm_x);
            int issued = 0;
            for (int st = 0; st < nst; ++st) {
                const int s = st % S;
                if (st >= S && !op_wait(empty(s), ((st / S) - 1) & 1, false, P.status)) {
                    abort_tile = 1;
                    break;
                }
                const uint32_t sa = base + s * stage_bytes;
                mbar_arrive_expect_tx(full(s), stage_bytes);
                tma_load_3d(sa, &P.tm_w, 0, n0, kb0 + st * KB, full(s));
                tma_load_3d(sa + w_bytes, &P.tm_x, 0, t0, kb0 + st * KB, full(s));
                issued = st + 1;
            }
            // after a time-out, the loads in flight land before the CTA may exit
            if (issued < nst)
                for (int st = issued > S ? issued - S : 0; st < issued; ++st)
                    op_wait(full(st % S), (st / S) & 1, false, P.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (elect_one()) {   // MMA issuer
            const uint32_t idesc = idesc_bf16(kOpTileN, (uint32_t)npad, 0, 0);
            bool ok = true;
            for (int st = 0; st < nst && ok; ++st) {
                const int s = st % S;
                if (!op_wait(full(s), (st / S) & 1, false, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = base + s * stage_bytes;
                for (int j = 0; j < KB; ++j) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss(tmem, smem_desc(sa + j * kOpWBlock + k * 32, 16, 1024, 2),
                               smem_desc(sa + w_bytes + j * x_block + k * 32, 16, 1024, 2), idesc,
                               (st | j | k) ? 1u : 0u);
                }
                mma_commit(empty(s));
            }
            if (ok) {
                mma_commit(b_done);
            } else {
                abort_tile = 1;
                mma_commit(b_drain);   // the MMAs issued complete before TMEM is freed
                op_wait(b_drain, 0, false, P.status);
                mbar_arrive(b_done);
            }
        }
        __syncwarp();
    }

    // every warp: the MMAs are done (the ring is drained); arm the receive barrier and
    // tell the peer it may send
    bool ok = op_wait(b_done, 0, false, P.status);
    tc_fence_after();
    ok = __all_sync(0xffffffffu, ok && *(volatile int32_t *)&abort_tile == 0);
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(b_recv, (uint32_t)kOpTileN * half * 4);
        mbar_arrive_remote(mapa(b_ready, peer));
    }
    const int row = warp * 32 + lane;                       // this thread's feature in the tile
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    // send: the partial of the peer's token half
    if (ok) ok = __all_sync(0xffffffffu, op_wait(b_ready, 0, true, P.status));
    if (ok) {
        const uint32_t dst = mapa(base + (uint32_t)row * recv_stride, peer);
        const uint32_t rbar = mapa(b_recv, peer);
        for (int c = 0; c < half / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + peer * half + c * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_async_v4(dst + c * 128 + q * 16, make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]), rbar);
        }
    }
    // receive, add, store this CTA's token half
    if (ok) ok = __all_sync(0xffffffffu, op_wait(b_recv, 0, true, P.status));
    if (ok) {
        const uint8_t *recv = smem_raw + (base - smem_u32(smem_raw)) + (size_t)row * recv_stride;
        const int n = n0 + row;
        for (int c = 0; c < half / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + rank * half + c * 32, r);
            tmem_wait_ld();
            float v[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = *reinterpret_cast<const float4 *>(recv + c * 128 + q * 16);
                v[4 * q] = __uint_as_float(r[4 * q]) + x.x;
                v[4 * q + 1] = __uint_as_float(r[4 * q + 1]) + x.y;
                v[4 * q + 2] = __uint_as_float(r[4 * q + 2]) + x.z;
                v[4 * q + 3] = __uint_as_float(r[4 * q + 3]) + x.w;
            }
            const int tb = t0 + (int)rank * half + c * 32;
            if (n < P.hidden) {
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    // two tokens per step; each warp instruction writes 32 consecutive features
                    const uint32_t pr = bf16x2(v[j], v[j + 1]);
                    if (tb + j < P.tokens)
                        P.out[(size_t)(tb + j) * P.hidden + n] = __ushort_as_bfloat16((unsigned short)(pr & 0xFFFFu));
                    if (tb + j + 1 < P.tokens)
                        P.out[(size_t)(tb + j + 1) * P.hidden + n] = __ushort_as_bfloat16((unsigned short)(pr >> 16));
                }
            }
        }
    } else if (threadIdx.x == 0) {
        // the peer may still be sending: wait (bounded) for its bytes before exiting
        op_wait(b_recv, 0, true, P.status);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // neither CTA frees shared memory the other still writes
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

std::mutex g_mutex;
bool g_attr[64];

}  // namespace
}  // namespace mla

extern "C" mla_status mla_epilog_oproj(int32_t tokens, int32_t hidden, const void *o_v, const void *w_o,
                                       void *out, int32_t *device_status, mla_stream_t stream) {
    mla::NvtxRange nvtx_range("mla_epilog_oproj");
    using namespace mla;
    auto aligned16 = [](const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (tokens < 1 || hidden < 8 || hidden % 8 != 0 || !aligned16(o_v) || !aligned16(w_o) || !aligned16(out) ||
        !device_status || (reinterpret_cast<uintptr_t>(device_status) & 3u) != 0)
        return MLA_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
    OprojParams p = {};
    p.tokens = tokens;
    p.hidden = hidden;
    p.npad = ((tokens < kOpMaxTok ? tokens : kOpMaxTok) + 63) / 64 * 64;
    // K blocks per stage: the most (up to 4) that still leave a ring of three stages
    const uint32_t per_kb = kOpWBlock + (uint32_t)p.npad * 128;
    p.kb = 1;
    for (int kb = 4; kb > 1; kb /= 2)
        if ((kOpSmemMax - 1024) / (kb * per_kb) >= 3) {
            p.kb = kb;
            break;
        }
    const uint32_t stage = p.kb * per_kb;
    const uint32_t recv = (uint32_t)kOpTileN * (p.npad / 2 + 4) * 4;
    p.stages = (int)((kOpSmemMax - 1024) / stage);
    if (p.stages > kOpMaxStages) p.stages = kOpMaxStages;
    if (p.stages < 2 || (uint32_t)p.stages * stage < recv) return MLA_ERR_UNSUPPORTED;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.status = device_status;
    if (!encode_bf16_kblocks(&p.tm_w, w_o, kOpK, (cuuint64_t)hidden, kOpTileN, (cuuint32_t)p.kb) ||
        !encode_bf16_kblocks(&p.tm_x, o_v, kOpK, (cuuint64_t)tokens, (cuuint32_t)p.npad, (cuuint32_t)p.kb))
        return MLA_ERR_INVALID_ARG;
    const uint32_t smem = (uint32_t)p.stages * stage + 1024;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!g_attr[dev]) {
            if (cudaFuncSetAttribute(mla_epilog_oproj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kOpSmemMax)) != cudaSuccess)
                return MLA_ERR_CUDA;
            g_attr[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ((hidden + kOpTileN - 1) / kOpTileN), (tokens + kOpMaxTok - 1) / kOpMaxTok);
    cfg.blockDim = dim3(kOpThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_epilog_oproj_kernel, p) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
