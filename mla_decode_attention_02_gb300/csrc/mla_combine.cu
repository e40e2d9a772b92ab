// Split merge: rows that the schedule cut into several key ranges have one
// fp32 partial (o_i normalised, lse_i) per piece; they combine by
// log-sum-exp weights, as FlashDecoding's second phase does (Atlas 800I A3
// TPOT-jitter troubleshooting post, "MLAKernel performance root cause"):
//
//   M = max_i lse_i,  w_i = exp(lse_i - M),
//   o = sum_i w_i o_i / sum_i w_i  (-> bf16),  lse = M + ln sum_i w_i.
//
// Rows of up to kWarpParts pieces: one warp per (row, head) task, warps
// striding over all tasks (most rows of most schedules are not split and cost
// one load).  Rows of more pieces (one long request spread over many SM
// pairs): one CTA per (row, head) task, its warps sharing the pieces, so that
// the reads of a single long request are spread over many SMs.  Each lane owns
// 16 of the 512 output values as four float4 columns, so every partial row is
// read fully coalesced.  The pieces are summed in a fixed order: the result
// does not depend on timing.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kCombineGrid = 1024;  // CTAs; warps stride over (row, head) tasks

constexpr int kWarpParts = 8;      // rows with more parts are merged by a whole CTA per head
// Parts whose rows are loaded before any of them is summed.  Two, with the
// kernel held to 80 registers (three CTAs per SM): MTP's merge 16.2 -> 14.4 us,
// long-1M's 13.4 -> 12.0 us; four needs 141 registers, and the lost occupancy
// made mixed and MTP slower.
constexpr int kBatch = 2;
static_assert(kWarpParts <= 32, "one part's lse per lane");

// o = acc / W -> bf16 (lane owns four float4 columns of the 512), lse = M + ln W.
__device__ __forceinline__ void store_row(__nv_bfloat16 *orow, float *lse, const float4 (&acc)[4], float W,
                                          float M, int lane) {
    const float inv = 1.f / W;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t *>(&lo);
        packed.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(orow)[k * 32 + lane] = packed;
    }
    if (lane == 0) *lse = M + logf(W);
}

// One (row, head) task of a row of many parts, by the whole CTA: warp w sums
// parts w, w + 8, ...; the warps' sums are added in warp order (the result
// does not depend on timing).
__device__ __forceinline__ void merge_task_cta(int32_t r, int32_t h, int32_t n, const int32_t *row_part0,
                                               const float *lse_part, const float *o_part,
                                               __nv_bfloat16 *o_latent, float *lse_out, int lane, int warp,
                                               float4 (&red)[kCombineWarps][4][32], float (&red_w)[kCombineWarps],
                                               float (&red_m)[kCombineWarps]) {
    __nv_bfloat16 *orow = o_latent + ((size_t)r * kHeads + h) * kDl;
    const int32_t part0 = row_part0[r];
    // M = max over all parts (each warp over its parts, then across warps)
    float m = -INFINITY;
    for (int32_t i = warp * 32 + lane; i < n; i += kCombineWarps * 32)
        m = fmaxf(m, lse_part[(size_t)(part0 + i) * kHeads + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red_m[warp] = m;
    __syncthreads();
    float M = red_m[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) M = fmaxf(M, red_m[w]);

    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    // this warp's parts (warp, warp + 8, ...) in order, kBatch at a time: every
    // load of a batch is in flight before the first is summed
#pragma unroll 1
    for (int32_t i0 = warp; i0 < n; i0 += kBatch * kCombineWarps) {
        float lse_j[kBatch];
        float4 v[kBatch][4];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int32_t i = i0 + j * kCombineWarps;
            if (i < n) {
                const size_t slot = (size_t)(part0 + i) * kHeads + h;
                lse_j[j] = lse_part[slot];
                const float4 *src = reinterpret_cast<const float4 *>(o_part + slot * kDl);
#pragma unroll
                for (int k = 0; k < 4; ++k) v[j][k] = src[k * 32 + lane];
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (i0 + j * kCombineWarps < n) {
                const float w = expf(lse_j[j] - M);
                W += w;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc[k].x += w * v[j][k].x;
                    acc[k].y += w * v[j][k].y;
                    acc[k].z += w * v[j][k].z;
                    acc[k].w += w * v[j][k].w;
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) red[warp][k][lane] = acc[k];
    if (lane == 0) red_w[warp] = W;
    __syncthreads();
    // warp 0 sums the warps' partial sums in warp order (the result does not
    // depend on timing) and writes the row
    if (warp == 0) {
        float Wt = 0.f;
        float4 t[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) t[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < kCombineWarps; ++w) {
            Wt += red_w[w];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 v = red[w][k][lane];
                t[k].x += v.x;
                t[k].y += v.y;
                t[k].z += v.z;
                t[k].w += v.w;
            }
        }
        store_row(orow, lse_out + (size_t)r * kHeads + h, t, Wt, M, lane);
    }
    __syncthreads();   // red / red_m are reused by the next task
}

__global__ void __launch_bounds__(32 * kCombineWarps, 3)
mla_combine_kernel(const uint8_t *__restrict__ ws, __nv_bfloat16 *__restrict__ o_latent,
                   float *__restrict__ lse_out, int32_t batch, int32_t s_q, int32_t num_units) {
    __shared__ float4 red[kCombineWarps][4][32];   // per warp: its lanes' 16 partial sums
    __shared__ float red_w[kCombineWarps], red_m[kCombineWarps];
    // launched as a programmatic dependent of the main kernel
    ptx::pdl_wait_prior();
    // nothing to merge when no row was split and every row was valid: the main
    // kernel wrote every output itself
    const PlanHeader *hdr = reinterpret_cast<const PlanHeader *>(ws);
    if (hdr->num_parts == 0 && (hdr->status & MLA_DEV_BAD_SEQ_LEN) == 0) return;
    const PlanLayout L = plan_layout(batch, s_q, num_units);
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t tasks = (int64_t)L.num_rows * kHeads;
    const int32_t *row_nparts = reinterpret_cast<const int32_t *>(ws + L.row_nparts);
    const int32_t *row_part0 = reinterpret_cast<const int32_t *>(ws + L.row_part0);
    const float *lse_part = reinterpret_cast<const float *>(ws + L.lse_part);
    const float *o_part = reinterpret_cast<const float *>(ws + L.o_part);

    // Rows of a few parts: one warp per (row, head) task, warps strided over
    // the tasks; the parts are summed in index order.
    for (int64_t task = (int64_t)blockIdx.x * kCombineWarps + warp; task < tasks;
         task += (int64_t)gridDim.x * kCombineWarps) {
        const int32_t r = (int32_t)(task / kHeads);
        const int32_t h = (int32_t)(task % kHeads);
        const int32_t n = row_nparts[r];
        if (n == 1 || n > kWarpParts) continue;  // written by the main kernel / merged below
        __nv_bfloat16 *orow = o_latent + ((size_t)r * kHeads + h) * kDl;
        if (n == 0) {          // invalid row (bad seq_len): NaN, flagged in the status word
            const __nv_bfloat16 nan = __float2bfloat16(__int_as_float(0x7fc00000));
            for (int d = lane; d < kDl; d += 32) orow[d] = nan;
            if (lane == 0) lse_out[(size_t)r * kHeads + h] = __int_as_float(0x7fc00000);
            continue;
        }
        const int32_t part0 = row_part0[r];
        // lane i < n holds part i's lse and weight
        const float lse_i = lane < n ? lse_part[(size_t)(part0 + lane) * kHeads + h] : -INFINITY;
        float M = lse_i;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w_i = lane < n ? expf(lse_i - M) : 0.f;
        float4 acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        float W = 0.f;
        // the parts in index order, kBatch at a time: every load of a batch is in
        // flight before the first is summed
#pragma unroll 1
        for (int32_t i0 = 0; i0 < n; i0 += kBatch) {
            float4 v[kBatch][4];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (i0 + j < n) {
                    const float4 *src =
                        reinterpret_cast<const float4 *>(o_part + ((size_t)(part0 + i0 + j) * kHeads + h) * kDl);
#pragma unroll
                    for (int k = 0; k < 4; ++k) v[j][k] = src[k * 32 + lane];
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const float w = __shfl_sync(0xffffffffu, w_i, (i0 + j) & 31);
                if (i0 + j < n) {
                    W += w;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        acc[k].x += w * v[j][k].x;
                        acc[k].y += w * v[j][k].y;
                        acc[k].z += w * v[j][k].z;
                        acc[k].w += w * v[j][k].w;
                    }
                }
            }
        }
        store_row(orow, lse_out + (size_t)r * kHeads + h, acc, W, M, lane);
    }

    // Rows of many parts (one long request over many SM pairs): one (row,
    // head) task per CTA, tasks strided over the grid; the CTA's warps share
    // the parts (merge_task_cta).  Skipped at once when no row has that many.
    int big = 0;
    for (int32_t r = threadIdx.x; r < L.num_rows; r += blockDim.x) big |= row_nparts[r] > kWarpParts;
    if (!__syncthreads_or(big)) return;
    for (int64_t task = blockIdx.x; task < tasks; task += gridDim.x) {
        const int32_t n = row_nparts[task / kHeads];
        if (n <= kWarpParts) continue;   // CTA-uniform: every thread skips together
        merge_task_cta((int32_t)(task / kHeads), (int32_t)(task % kHeads), n, row_part0, lse_part, o_part,
                       o_latent, lse_out, lane, warp, red, red_w, red_m);
    }
}

}  // namespace

cudaError_t launch_combine(const void *ws, void *o_latent, float *lse, int32_t batch, int32_t s_q,
                           int32_t num_units, cudaStream_t stream) {
    const int64_t tasks = (int64_t)batch * s_q * kHeads;
    const int grid = (int)(tasks < kCombineGrid ? tasks : kCombineGrid);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * kCombineWarps);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_combine_kernel, static_cast<const uint8_t *>(ws),
                              static_cast<__nv_bfloat16 *>(o_latent), lse, batch, s_q, num_units);
}

}  // namespace mla
