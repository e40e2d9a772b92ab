// MLA prolog kernel: the step before decode attention, producing its inputs.
//
// What it computes ("Huawei Ascend servers: DeepSeek V3/R1 inference best
// practice" section 3.2.1 on weight absorption and section 6.1 on the fused
// MLAProlog operator; the CloudMatrix384 digest, section 3.2, on what that
// operator fuses: RMSNorm, the Q/K/V projections and RoPE):
//
//   q_latent[t][h] = q_nope[t][h] . W_UK[h]          128 -> 512 per head, bf16 out
//   q_rope[t][h]   = RoPE(q_pe[t][h], pos_t)         64 dims, pairs (2i, 2i+1)
//   cache row at pos_t of request b <- RMSNorm(kv_latent[t]) || RoPE(k_pe[t], pos_t)
//
// with pos_t = seq_len[b] - s_q + t (seq_lens count this step's tokens), the
// pair angle pos * base^(-2i/64), and RMSNorm x / sqrt(mean(x^2) + eps) * gamma.
//
// GB300 design: one launch of identical CTAs, one per (head h, 128-token
// tile, quarter of the 512 latent columns); 65 KB of shared memory and 128
// TMEM columns each, so three share an SM.
//  - Launch: a programmatic dependent of the previous kernel in the stream
//    (barriers and TMEM are set up while that kernel drains).
//  - Warp 0: TMA brings the head's q_nope tile (K-major, 128 tokens x 128
//    dims) and its W_UK quarter (MN-major: 128 dims x 128 columns, W_UK's own
//    row-major layout) in as one box each; one elected lane issues eight
//    tcgen05.mma (M=128, N=128, K=16) into TMEM.
//  - Warps 1-3, while the copies and MMAs run: RoPE of q_pe for head h, the
//    tile's tokens and the quarter's 16 position dims (two 16-byte chunks
//    per token); the quarter-0 CTA of head h also appends token 128 * tile + h
//    of the step to the cache (RMSNorm of its latent, RoPE of its k_pe).
//  - All four warps: read TMEM back (one tile row per thread), round to
//    bf16 and stage the rows in a 128-byte-swizzled tile over the W_UK buffer
//    (conflict-free); each warp then stores its own 32 rows, two contiguous
//    256-byte rows per instruction (a TMA store would queue behind the
//    other CTAs' loads on the SM's copy engine: measured 3-5 us per CTA).
//
// RoPE angles.  fp64 is a narrow pipe on this part, so each angle is formed in
// fp32 double-float arithmetic (Dekker's exact product via fma): the pair's
// turns per position g = base^(-2i/64) / (2 pi) is held as hi + lo floats
// (the model's rotary table, built once in fp64 by mla_rope_table_kernel; an
// fp64 pow in every CTA cost ~3.7 us each), pos * g is formed exactly enough, its integer
// part dropped, and the fraction of a turn (|r| <= 1/2) becomes an angle in
// [-pi, pi] for the hardware sin/cos.  The angle error stays below 1e-6 rad
// for positions below 2^20 and near 1e-5 rad at worst below 2^31 (checked
// against fp64 in an fp32 emulation), far under the bf16 rounding of the
// outputs; an fp32 product alone would be off by ~0.06 rad at a million tokens.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "mla_internal.h"
#include "mla_prolog.h"
#include "sm103_ptx.cuh"

namespace mla {
bool encode_bf16_4d(CUtensorMap *m, const void *base, cuuint64_t d1, cuuint64_t d2, cuuint64_t d3,
                    cuuint64_t s1, cuuint64_t s2, cuuint64_t s3, cuuint32_t rows, cuuint32_t blocks);
namespace {
using namespace ptx;

constexpr int kDn = MLA_D_NOPE;           // no-position query dims per head
constexpr int kBM = 128;                  // tokens per tile (MMA M)
constexpr int kBN = 128;                  // latent columns per CTA (MMA N)
constexpr int kNParts = kDl / kBN;        // CTAs per (head, token tile)
constexpr int kThreadsP = 128;
constexpr int kPairs = kDr / 2;           // RoPE pairs per 64-dim vector
constexpr int kPartPairs = kPairs / kNParts;              // pairs each quarter rotates
constexpr uint32_t kABlk = kBM * 128;     // one 64-dim block of the A tile: 128 rows x 128 B
constexpr uint32_t kABytes = (kDn / 64) * kABlk;          // 32 KB (a full 128-token tile)
constexpr uint32_t kBBlk = kDn * 128;     // one 64-column block of W_UK: 128 rows x 128 B
constexpr uint32_t kBBytes = (kBN / 64) * kBBlk;          // 32 KB
constexpr uint32_t kOBlk = kBM * 128;     // one 64-column block of the output tile
constexpr uint32_t kSmemP = kABytes + kBBytes + 1024;     // + alignment slack
// With fewer than 128 tokens the A tile holds only round_up(tokens, 8) rows, so
// four CTAs share an SM; never five: four fill the SM's 512 TMEM columns.
constexpr uint32_t kSmemMinP = 48 * 1024;
constexpr uint32_t kTmemColsP = kBN;
constexpr uint64_t kWaitLimitNsP = 2000000000ull;
constexpr int kQIters = (2 * kBM + 95) / 96;                // q_pe chunks per thread of warps 1-3
static_assert((kBN / 64) * kOBlk <= kBBytes, "output staging reuses the W_UK tile");
static_assert(kDn == 128, "eight K=16 steps over two 64-dim blocks");
static_assert(kPartPairs == 8, "a quarter rotates two 16-byte chunks (four pairs each) per token");
static_assert(kBM <= 2 * 96, "warps 1-3 find the tile's positions in two rounds");

struct PrologParams {
    CUtensorMap tm_a;    // q_nope viewed as (64 dims, tokens, 2 dim blocks, heads)
    CUtensorMap tm_b;    // W_UK viewed as (64 cols, 128 dims, 8 col blocks, heads)
    const __nv_bfloat16 *q_pe;
    const __nv_bfloat16 *kv_latent;
    const __nv_bfloat16 *k_pe;
    const __nv_bfloat16 *gamma;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const float *rope_table;   // g_hi[32], then g_lo[32] (mla_prolog_rope_table)
    __nv_bfloat16 *q_latent;
    __nv_bfloat16 *q_rope;
    __nv_bfloat16 *kv_cache;
    int32_t *status;
    int64_t num_pages;
    float eps;
    int32_t tokens, s_q, max_pages;
    int32_t a_rows;    // rows of the A tile that TMA loads: min(128, round_up(tokens, 8))
};

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, int32_t *status) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNsP) {
            atomicOr(status, MLA_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// sin and cos of the angle pos * 2 pi (g_hi + g_lo), 0 <= pos < 2^31 (see the file notes).
__device__ __forceinline__ void rope_sincos(int32_t pos, float g_hi, float g_lo, float &s, float &c) {
    const float ph = (float)(pos >> 16), pl = (float)(pos & 0xffff);   // both exact
    const float gh16 = g_hi * 65536.f, gl16 = g_lo * 65536.f;          // exact scalings
    const float a1 = ph * gh16, e1 = fmaf(ph, gh16, -a1);             // ph * gh16 = a1 + e1 exactly
    const float a2 = pl * g_hi, e2 = fmaf(pl, g_hi, -a2);
    float r = (a1 - rintf(a1)) + (a2 - rintf(a2));                      // fractions of the big terms
    r += e1 + e2 + fmaf(ph, gl16, pl * g_lo);
    r -= rintf(r);
    __sincosf(r * 6.28318530717958648f, &s, &c);
}

// Rotate the four pairs held by eight consecutive bf16 values, pairs p0 .. p0 + 3.
__device__ __forceinline__ uint4 rope8(uint4 v, int32_t pos, int p0, const float *g_hi,
                                       const float *g_lo) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float s, c;
        rope_sincos(pos, g_hi[p0 + j], g_lo[p0 + j], s, c);
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
        w[j] = pack_bf16x2(x.x * c - x.y * s, x.x * s + x.y * c);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Position of token tok, or -1 when it has no slot in its request's table.
__device__ __forceinline__ int32_t token_pos(const PrologParams &P, int tok) {
    const int b = tok / P.s_q, t = tok % P.s_q;
    const int64_t pos = (int64_t)P.seq_lens[b] - P.s_q + t;
    return pos < 0 || pos >= (int64_t)P.max_pages * kPage ? -1 : (int32_t)pos;
}

// Append token tok at position pos (-1: none) to the cache (warps 2 and 3:
// thread c owns latent chunk c, threads 0-7 also the k_pe chunks).
__device__ __forceinline__ void append_token(const PrologParams &P, int tok, int32_t pos, int c,
                                             const float *g_hi, const float *g_lo, float *red) {
    const uint4 x = reinterpret_cast<const uint4 *>(P.kv_latent + (size_t)tok * kDl)[c];
    const uint4 k = c < kDr / 8 ? reinterpret_cast<const uint4 *>(P.k_pe + (size_t)tok * kDr)[c]
                                : make_uint4(0, 0, 0, 0);
    int64_t row = -1;
    if (pos >= 0) {
        const int b = tok / P.s_q;
        const int32_t page = P.block_table[(size_t)b * P.max_pages + pos / kPage];
        if (page >= 0 && page < P.num_pages) row = (int64_t)page * kPage + pos % kPage;
    }
    if (c == 0 && row < 0) atomicOr(P.status, pos < 0 ? MLA_DEV_BAD_SEQ_LEN : MLA_DEV_BAD_PAGE);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
        ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((c & 31) == 0) red[c / 32] = ss;
    named_sync(2, 64);
    if (row < 0) return;
    __nv_bfloat16 *dst = P.kv_cache + row * kDrow;
    const float inv = rsqrtf((red[0] + red[1]) * (1.0f / kDl) + P.eps);
    const uint4 gv = reinterpret_cast<const uint4 *>(P.gamma)[c];
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
        const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gw[j]));
        o[j] = pack_bf16x2(f.x * inv * g.x, f.y * inv * g.y);
    }
    reinterpret_cast<uint4 *>(dst)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    if (c < kDr / 8) reinterpret_cast<uint4 *>(dst + kDl)[c] = rope8(k, pos, c * 4, g_hi, g_lo);
}

__global__ void __launch_bounds__(kThreadsP, 4) mla_prolog_kernel(const __grid_constant__ PrologParams P) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[2];   // 0: operands landed, 1: MMAs done
    __shared__ uint32_t tmem_slot;
    __shared__ int32_t abort_tile;                // a wait of this CTA ran out: write nothing
    __shared__ float g_hi[kPairs], g_lo[kPairs], red[2];
    __shared__ int32_t pos_s[kBM];                // positions of the tile's tokens (-1: none)
    const int warp = threadIdx.x / 32;
    const int g = blockIdx.x;
    const int np = g % kNParts;
    const int h = (g / kNParts) % kHeads;
    const int mt = g / (kNParts * kHeads);
    const uint32_t s_a = (smem_u32(smem) + 1023u) & ~1023u;
    const uint32_t a_blk = (uint32_t)P.a_rows * 128;         // bytes of one 64-dim block of A
    const uint32_t s_b = s_a + ((2 * a_blk + 1023u) & ~1023u);
    const uint32_t b_full = smem_u32(&bars[0]), b_done = smem_u32(&bars[1]);
    if (threadIdx.x == 0) {
        mbar_init(b_full, 1);
        mbar_init(b_done, 1);
        fence_mbar_init();
        abort_tile = 0;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemColsP);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // Launched as a programmatic dependent of the previous kernel in the stream:
    // the setup above overlaps its tail; every global read and write comes after.
    pdl_wait_prior();
    pdl_launch_dependents();

    if (warp == 0) {
        if (elect_one()) {
            prefetch_tmap(&P.tm_a);
            prefetch_tmap(&P.tm_b);
            mbar_arrive_expect_tx(b_full, 2 * a_blk + kBBytes);
            tma_load_4d(s_a, &P.tm_a, 0, mt * kBM, 0, h, b_full);
            tma_load_4d(s_b, &P.tm_b, 0, 0, np * (kBN / 64), h, b_full);
            if (bounded_wait(b_full, 0, P.status)) {
                tc_fence_after();
                constexpr uint32_t idesc = idesc_bf16(kBM, kBN, 0, 1);
#pragma unroll
                for (int ks = 0; ks < kDn / 16; ++ks) {
                    // A: K-major, 128-byte swizzle; a K step of 16 dims is 32 bytes inside a
                    // block.  Rows past a_rows read other bytes of this CTA's shared memory;
                    // their results fall on tokens that are never stored.
                    const uint64_t da = smem_desc(s_a + (ks / 4) * a_blk + (ks % 4) * 32, 16, 1024, 2);
                    // B: MN-major, column blocks kBBlk apart, a K step is 16 rows of 128 bytes
                    const uint64_t db = smem_desc(s_b + ks * 2048, kBBlk, 1024, 2);
                    mma_ss(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
                }
                mma_commit(b_done);
            } else {
                abort_tile = 1;
                mbar_arrive(b_done);   // time-out: release the epilogue, which writes nothing
            }
        }
        __syncwarp();
    } else {
        // ---- warps 1-3: RoPE work while the operands load and the MMAs run
        const int tid = threadIdx.x - 32;   // 0 .. 95
        const int tok0 = mt * kBM;
        // every independent load first (q_pe chunks, the rotary table, seq_lens), so
        // their latencies overlap; then the math.
        // q_pe of head h, tokens of the tile, dims [16 np, 16 np + 16): two chunks per
        // token, 256 chunks over 96 threads
        uint4 v[kQIters];
#pragma unroll
        for (int k = 0; k < kQIters; ++k) {
            const int i = tid + 96 * k;
            if (i < 2 * kBM && tok0 + i / 2 < P.tokens)
                v[k] = *reinterpret_cast<const uint4 *>(
                    P.q_pe + ((size_t)(tok0 + i / 2) * kHeads + h) * kDr + np * 16 + (i & 1) * 8);
        }
        float th = 0.f, tl = 0.f;
        if (warp == 1) {
            th = P.rope_table[tid];
            tl = P.rope_table[kPairs + tid];
        }
        const int32_t p0 = tid < kBM && tok0 + tid < P.tokens ? token_pos(P, tok0 + tid) : -1;
        const int32_t p1 = tid + 96 < kBM && tok0 + tid + 96 < P.tokens ? token_pos(P, tok0 + tid + 96) : -1;
        if (warp == 1) {
            g_hi[tid] = th;
            g_lo[tid] = tl;
        }
        pos_s[tid] = p0;
        if (tid + 96 < kBM) pos_s[tid + 96] = p1;
        named_sync(1, 96);
        if (np == 0 && warp >= 2 && tok0 + h < P.tokens)
            append_token(P, tok0 + h, pos_s[h], tid - 32, g_hi, g_lo, red);
#pragma unroll
        for (int k = 0; k < kQIters; ++k) {
            const int i = tid + 96 * k;
            if (i < 2 * kBM && tok0 + i / 2 < P.tokens) {
                const int32_t pos = pos_s[i / 2];
                *reinterpret_cast<uint4 *>(P.q_rope + ((size_t)(tok0 + i / 2) * kHeads + h) * kDr +
                                           np * 16 + (i & 1) * 8) =
                    pos < 0 ? make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u)
                            : rope8(v[k], pos, np * kPartPairs + (i & 1) * 4, g_hi, g_lo);
            }
        }
    }

    // ---- epilogue: warp w reads TMEM lanes [32w, 32w + 32) = tile rows; every lane one row
    bool ok = bounded_wait(b_done, 0, P.status);
    tc_fence_after();
    ok = ok && *(volatile int32_t *)&abort_tile == 0;
    const int row = warp * 32 + (threadIdx.x & 31);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) abort_tile = 1;
    if (ok) {
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
            tmem_wait_ld();
            const uint32_t blk = s_b + (c / 2) * kOBlk + row * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]));
                v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
                v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
                v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
                const uint32_t chunk = (uint32_t)((c % 2) * 4 + q) ^ (uint32_t)(row & 7);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(blk + chunk * 16),
                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
        }
    }
    if (ok) {
        // the warp's own 32 rows back out of the staging tile, two 256-byte rows per store
        __syncwarp();
        const int lane = threadIdx.x & 31;
        const int j16 = lane & 15, b = j16 >> 3, j = j16 & 7;
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
            const int r = warp * 32 + 2 * k + (lane >> 4);
            const int tok = mt * kBM + r;
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(s_b + b * kOBlk + r * 128 + ((j ^ (r & 7)) * 16)));
            if (tok < P.tokens)
                *reinterpret_cast<uint4 *>(P.q_latent + ((size_t)tok * kHeads + h) * kDl + np * kBN +
                                           j16 * 8) = v;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemColsP);
    }
}

// ---------------------------------------------------------------- host side

std::mutex g_prolog_mutex;
bool g_prolog_attr[64];

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Turns per position of each RoPE pair, base^(-2i/64) / (2 pi), in fp64, stored as
// hi + lo floats: table[i] = hi, table[32 + i] = lo.
__global__ void __launch_bounds__(32) mla_rope_table_kernel(double base, float *table) {
    const int i = threadIdx.x;
    const double turns = pow(base, -(double)(2 * i) / kDr) * 0.15915494309189535;
    const float hi = (float)turns;
    table[i] = hi;
    table[kPairs + i] = (float)(turns - (double)hi);
}

}  // namespace
}  // namespace mla

extern "C" mla_status mla_prolog_rope_table(double rope_base, float *table, mla_stream_t stream) {
    if (!std::isfinite(rope_base) || !(rope_base > 0.0) || !table ||
        (reinterpret_cast<uintptr_t>(table) & 3u))
        return MLA_ERR_INVALID_ARG;
    mla::mla_rope_table_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(rope_base, table);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" mla_status mla_prolog(const mla_problem *prob, const void *q_nope, const void *q_pe,
                                 const void *kv_latent, const void *k_pe, const void *w_uk,
                                 const void *kv_norm_weight, float rms_eps, const float *rope_table,
                                 void *kv_cache, int64_t num_pages, const int32_t *block_table,
                                 const int32_t *seq_lens, void *q_latent, void *q_rope,
                                 int32_t *device_status, mla_stream_t stream) {
    mla::NvtxRange nvtx_range("mla_prolog");
    using namespace mla;
    if (!prob || prob->batch < 1 || prob->max_pages_per_seq < 1 || prob->flags != 0)
        return MLA_ERR_INVALID_ARG;
    if (prob->s_q != 1 && prob->s_q != 2) return MLA_ERR_UNSUPPORTED;
    if (prob->num_heads != kHeads || prob->page_size != kPage) return MLA_ERR_UNSUPPORTED;
    if ((int64_t)prob->batch * prob->max_pages_per_seq >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
    // every position (and so every RoPE angle's integer input) stays below 2^31
    if ((int64_t)prob->max_pages_per_seq * kPage >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
    const int64_t tokens = (int64_t)prob->batch * prob->s_q;
    const int64_t m_tiles = (tokens + kBM - 1) / kBM;
    const int64_t ctas = m_tiles * kHeads * kNParts;
    if (tokens * kHeads >= (int64_t)1 << 31 || ctas >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
    if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(kv_latent) || !aligned16(k_pe) ||
        !aligned16(w_uk) || !aligned16(kv_norm_weight) || !aligned16(kv_cache) ||
        !aligned16(q_latent) || !aligned16(q_rope) || !block_table || !seq_lens || !device_status ||
        !rope_table || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u) || (reinterpret_cast<uintptr_t>(device_status) & 3u) ||
        (reinterpret_cast<uintptr_t>(rope_table) & 3u))
        return MLA_ERR_INVALID_ARG;
    if (num_pages < 1 || !std::isfinite(rms_eps) || rms_eps < 0.f) return MLA_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_prolog_mutex);
        if (!g_prolog_attr[dev]) {
            if (cudaFuncSetAttribute(mla_prolog_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemP) != cudaSuccess)
                return MLA_ERR_CUDA;
            g_prolog_attr[dev] = true;
        }
    }
    PrologParams p{};
    p.a_rows = tokens >= kBM ? kBM : (int32_t)((tokens + 7) / 8 * 8);
    const uint32_t smem = std::max<uint32_t>(kSmemMinP, ((2u * p.a_rows * 128 + 1023u) & ~1023u) + kBBytes + 1024);
    const cuuint64_t H = kHeads, T = (cuuint64_t)tokens;
    // q_nope (dims, tokens, dim blocks, heads); W_UK (cols, dims, col blocks, heads)
    if (!encode_bf16_4d(&p.tm_a, q_nope, T, kDn / 64, H, H * kDn * 2, 128, kDn * 2, (cuuint32_t)p.a_rows, kDn / 64) ||
        !encode_bf16_4d(&p.tm_b, w_uk, kDn, kDl / 64, H, kDl * 2, 128, (cuuint64_t)kDn * kDl * 2, kDn, kBN / 64))
        return MLA_ERR_CUDA;
    p.q_pe = static_cast<const __nv_bfloat16 *>(q_pe);
    p.kv_latent = static_cast<const __nv_bfloat16 *>(kv_latent);
    p.k_pe = static_cast<const __nv_bfloat16 *>(k_pe);
    p.gamma = static_cast<const __nv_bfloat16 *>(kv_norm_weight);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.rope_table = rope_table;
    p.q_latent = static_cast<__nv_bfloat16 *>(q_latent);
    p.q_rope = static_cast<__nv_bfloat16 *>(q_rope);
    p.kv_cache = static_cast<__nv_bfloat16 *>(kv_cache);
    p.status = device_status;
    p.num_pages = num_pages;
    p.eps = rms_eps;
    p.tokens = (int32_t)tokens;
    p.s_q = prob->s_q;
    p.max_pages = prob->max_pages_per_seq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreadsP);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_prolog_kernel, p) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
