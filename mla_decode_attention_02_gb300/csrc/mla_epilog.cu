// MLA epilog: the step after decode attention.
//
// What it computes ("Huawei Ascend servers: DeepSeek V3/R1 inference best
// practice" section 3.2.1: with absorbed weights the attention output of each
// head lives in the 512-value latent space; sections 3.2-3.3 and figures 5-9
// place the output projection "O Proj" after attention):
//
//   o_v[t][h][v] = sum_c W_UV[h][v][c] * o_latent[t][h][c]      512 -> 128 per head
//   out[t][n]    = sum_k W_O[n][k] * o_v[t][k]                   16384 -> hidden
//
// GB300 design.
//  - W_UV step (mla_epilog_uv_kernel): one CTA per (head, 128-token tile),
//    M=128 tokens, N=128 value dims, K=512 latent values in eight 64-value
//    blocks (the tile's block of o_latent and W_UV[h]'s block, both K-major,
//    128-byte swizzle).  With up to 64 tokens all eight blocks fit in shared
//    memory and are loaded at once (one CTA per SM, every byte in flight);
//    with more, they pass through a three-stage ring (two CTAs per SM).
//    Warp 0 loads, warp 1 issues
//    four tcgen05.mma (K=16) per block into 128 TMEM columns and frees the
//    stage with tcgen05.commit; all four warps then read TMEM back (a row
//    per thread), round to bf16, stage the tile conflict-free in shared
//    memory and store each token's 256-byte row contiguously.  With fewer
//    than 128 tokens the A box holds only round_up(tokens, 8) rows.
//  - o_proj: its own tensor-core kernel, in mla_oproj.cu.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "mla_epilog.h"
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
bool encode_bf16_4d(CUtensorMap *m, const void *base, cuuint64_t d1, cuuint64_t d2, cuuint64_t d3,
                    cuuint64_t s1, cuuint64_t s2, cuuint64_t s3, cuuint32_t rows, cuuint32_t blocks);
namespace {
using namespace ptx;

constexpr int kDv = MLA_D_V;              // value dims per head
constexpr int kKBlocks = kDl / 64;        // 64-value K blocks of the latent
constexpr int kMaxStagesE = kDl / 64;    // the whole K extent in flight
constexpr int kRingStagesE = 3;          // when it does not fit: a three-stage ring, two CTAs per SM
constexpr int kThreadsE = 128;
constexpr uint32_t kBBlkE = kDv * 128;    // one K block of W_UV[h]: 128 rows x 128 B
constexpr uint32_t kOBlkE = 128 * 128;    // one 64-column block of the staged output tile
constexpr uint32_t kTmemColsE = kDv;
constexpr uint32_t kSmemMinE = 48 * 1024; // never five CTAs on an SM (four fill its TMEM)
constexpr uint64_t kWaitLimitNsE = 2000000000ull;
static_assert(kDv == 128 && kDl % 64 == 0, "M=128 x N=128 tiles over 64-value K blocks");
// dynamic shared memory budget: 227 KB per block, less room for the static barriers
constexpr uint32_t kSmemMaxE = 232448 - 2048;

struct EpilogParams {
    CUtensorMap tm_a;   // o_latent viewed as (64 values, tokens, 8 K blocks, heads)
    CUtensorMap tm_b;   // W_UV viewed as (64 values, 128 rows, 8 K blocks, heads)
    __nv_bfloat16 *o_v;
    int32_t *status;
    int32_t tokens, a_rows, stages;
};

__device__ __forceinline__ bool bounded_wait_e(uint32_t bar, uint32_t parity, int32_t *status) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNsE) {
            atomicOr(status, MLA_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(kThreadsE, 2) mla_epilog_uv_kernel(const __grid_constant__ EpilogParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStagesE + 1];   // full[s], empty[s], done
    __shared__ uint32_t tmem_slot;
    __shared__ int32_t abort_tile;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int h = blockIdx.x % kHeads;
    const int mt = blockIdx.x / kHeads;
    const uint32_t a_bytes = (uint32_t)P.a_rows * 128;
    const uint32_t a_span = (a_bytes + 1023u) & ~1023u;
    const uint32_t stage_bytes = a_span + kBBlkE;
    const uint32_t base = (smem_u32(smem) + 1023u) & ~1023u;
    const int S = P.stages;
    const uint32_t b_done = smem_u32(&bars[2 * kMaxStagesE]);
    auto full = [&](int s) { return smem_u32(&bars[s]); };
    auto empty = [&](int s) { return smem_u32(&bars[kMaxStagesE + s]); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(b_done, 1);
        fence_mbar_init();
        abort_tile = 0;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemColsE);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_wait_prior();
    pdl_launch_dependents();

    if (warp == 0) {
        if (elect_one()) {   // producer: the tile's A block and W_UV[h]'s block per stage
            prefetch_tmap(&P.tm_a);
            prefetch_tmap(&P.tm_b);
            for (int kb = 0; kb < kKBlocks; ++kb) {
                const int s = kb % S;
                if (kb >= S && !bounded_wait_e(empty(s), ((kb / S) - 1) & 1, P.status)) {
                    abort_tile = 1;
                    break;
                }
                const uint32_t sa = base + s * stage_bytes;
                mbar_arrive_expect_tx(full(s), a_bytes + kBBlkE);
                tma_load_4d(sa, &P.tm_a, 0, mt * 128, kb, h, full(s));
                tma_load_4d(sa + a_span, &P.tm_b, 0, 0, kb, h, full(s));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (elect_one()) {   // MMA issuer
            constexpr uint32_t idesc = idesc_bf16(128, kDv, 0, 0);
            bool ok = true;
            for (int kb = 0; kb < kKBlocks && ok; ++kb) {
                const int s = kb % S;
                if (!bounded_wait_e(full(s), (kb / S) & 1, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = base + s * stage_bytes;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // both operands K-major, 128-byte swizzle: a K step of 16 values is 32 bytes.
                    // With a_rows < 128 the rows past it read other bytes of this stage; their
                    // results fall on tokens that are never stored.
                    const uint64_t da = smem_desc(sa + k * 32, 16, 1024, 2);
                    const uint64_t db = smem_desc(sa + a_span + k * 32, 16, 1024, 2);
                    mma_ss(tmem, da, db, idesc, (kb | k) ? 1u : 0u);
                }
                mma_commit(empty(s));
            }
            if (ok) {
                mma_commit(b_done);
            } else {
                abort_tile = 1;
                mbar_arrive(b_done);
            }
        }
        __syncwarp();
    }

    // epilogue: warp w holds tile rows [32w, 32w + 32), one per lane
    bool ok = bounded_wait_e(b_done, 0, P.status);
    tc_fence_after();
    ok = __all_sync(0xffffffffu, ok && *(volatile int32_t *)&abort_tile == 0);
    const int row = warp * 32 + lane;
    if (ok) {
        // every stage is free once the MMAs are done: stage the tile at the start of the ring
#pragma unroll 1
        for (int c = 0; c < kDv / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
            tmem_wait_ld();
            const uint32_t blk = base + (c / 2) * kOBlkE + row * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t chunk = (uint32_t)((c % 2) * 4 + q) ^ (uint32_t)(row & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(blk + chunk * 16),
                             "r"(pack2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]))),
                             "r"(pack2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]))),
                             "r"(pack2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]))),
                             "r"(pack2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7])))
                             : "memory");
            }
        }
        __syncwarp();
        const int j16 = lane & 15, b = j16 >> 3, j = j16 & 7;
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
            const int r = warp * 32 + 2 * k + (lane >> 4);
            const int tok = mt * 128 + r;
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(base + b * kOBlkE + r * 128 + ((j ^ (r & 7)) * 16)));
            if (tok < P.tokens)
                *reinterpret_cast<uint4 *>(P.o_v + ((size_t)tok * kHeads + h) * kDv + j16 * 8) = v;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemColsE);
    }
}

// ---------------------------------------------------------------- host side

std::mutex g_mutex;
bool g_attr[64];

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

extern "C" mla_status mla_epilog_uv(const mla_problem *prob, const void *o_latent, const void *w_uv,
                                    void *o_v, int32_t *device_status, mla_stream_t stream) {
    mla::NvtxRange nvtx_range("mla_epilog_uv");
    using namespace mla;
    if (!prob || prob->batch < 1 || prob->max_pages_per_seq < 1 || prob->flags != 0)
        return MLA_ERR_INVALID_ARG;
    if (prob->s_q != 1 && prob->s_q != 2) return MLA_ERR_UNSUPPORTED;
    if (prob->num_heads != kHeads || prob->page_size != kPage) return MLA_ERR_UNSUPPORTED;
    const int64_t tokens = (int64_t)prob->batch * prob->s_q;
    const int64_t ctas = (tokens + 127) / 128 * kHeads;
    if (tokens * kHeads >= (int64_t)1 << 31 || ctas >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
    if (!aligned16(o_latent) || !aligned16(w_uv) || !aligned16(o_v) || !device_status ||
        (reinterpret_cast<uintptr_t>(device_status) & 3u))
        return MLA_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
    EpilogParams p{};
    p.a_rows = tokens >= 128 ? 128 : (int32_t)((tokens + 7) / 8 * 8);
    const uint32_t stage = (((uint32_t)p.a_rows * 128 + 1023u) & ~1023u) + kBBlkE;
    // the whole K extent in flight when it fits (one CTA per SM), else a ring
    p.stages = kMaxStagesE * stage + 1024 <= kSmemMaxE ? kMaxStagesE : kRingStagesE;
    const uint32_t smem = std::max<uint32_t>(kSmemMinE, p.stages * stage + 1024);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!g_attr[dev]) {
            if (cudaFuncSetAttribute(mla_epilog_uv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemMaxE) != cudaSuccess)
                return MLA_ERR_CUDA;
            g_attr[dev] = true;
        }
    }
    const cuuint64_t H = kHeads, T = (cuuint64_t)tokens;
    // o_latent (values, tokens, K blocks, heads); W_UV (values, rows, K blocks, heads)
    if (!encode_bf16_4d(&p.tm_a, o_latent, T, kKBlocks, H, H * kDl * 2, 128, kDl * 2,
                        (cuuint32_t)p.a_rows, 1) ||
        !encode_bf16_4d(&p.tm_b, w_uv, kDv, kKBlocks, H, kDl * 2, 128, (cuuint64_t)kDv * kDl * 2, kDv, 1))
        return MLA_ERR_CUDA;
    p.o_v = static_cast<__nv_bfloat16 *>(o_v);
    p.status = device_status;
    p.tokens = (int32_t)tokens;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreadsE);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_epilog_uv_kernel, p) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
