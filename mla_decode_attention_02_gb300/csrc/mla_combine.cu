// Split merge: rows that the schedule cut into several key ranges have one
// fp32 partial (o_i normalised, lse_i) per piece; they combine by
// log-sum-exp weights, as FlashDecoding's second phase does (Atlas 800I A3
// TPOT-jitter troubleshooting post, "MLAKernel performance root cause"):
//
//   M = max_i lse_i,  w_i = exp(lse_i - M),
//   o = sum_i w_i o_i / sum_i w_i  (-> bf16),  lse = M + ln sum_i w_i.
//
// One warp per (row, head) task, warps striding over all tasks (a fixed,
// small grid: most rows of most schedules are not split and cost one load);
// each lane owns 16 of the 512 output values as four float4 columns, so
// every partial row is read fully coalesced.  The pieces are summed in index
// order: the result does not depend on timing.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kCombineGrid = 1024;  // CTAs; warps stride over (row, head) tasks

__global__ void __launch_bounds__(32 * kCombineWarps)
mla_combine_kernel(const uint8_t *__restrict__ ws, __nv_bfloat16 *__restrict__ o_latent,
                   float *__restrict__ lse_out, int32_t batch, int32_t s_q, int32_t num_units) {
    // launched as a programmatic dependent of the main kernel
    ptx::pdl_wait_prior();
    // nothing to merge when no row was split and every row was valid: the main
    // kernel wrote every output itself
    const PlanHeader *hdr = reinterpret_cast<const PlanHeader *>(ws);
    if (hdr->num_parts == 0 && (hdr->status & MLA_DEV_BAD_SEQ_LEN) == 0) return;
    const PlanLayout L = plan_layout(batch, s_q, num_units);
    const int32_t lane = threadIdx.x & 31;
    const int64_t tasks = (int64_t)L.num_rows * kHeads;
    const int64_t stride = (int64_t)gridDim.x * kCombineWarps;
    const int32_t *row_nparts = reinterpret_cast<const int32_t *>(ws + L.row_nparts);
    const int32_t *row_part0 = reinterpret_cast<const int32_t *>(ws + L.row_part0);
    const float *lse_part = reinterpret_cast<const float *>(ws + L.lse_part);
    const float *o_part = reinterpret_cast<const float *>(ws + L.o_part);
    for (int64_t task = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5); task < tasks;
         task += stride) {
        const int32_t r = (int32_t)(task / kHeads);
        const int32_t h = (int32_t)(task % kHeads);
        const int32_t n = row_nparts[r];
        if (n == 1) continue;  // the main kernel wrote this row directly
        __nv_bfloat16 *orow = o_latent + ((size_t)r * kHeads + h) * kDl;
        if (n == 0) {          // invalid row (bad seq_len): NaN, flagged in the status word
            const __nv_bfloat16 nan = __float2bfloat16(__int_as_float(0x7fc00000));
            for (int d = lane; d < kDl; d += 32) orow[d] = nan;
            if (lane == 0) lse_out[(size_t)r * kHeads + h] = __int_as_float(0x7fc00000);
            continue;
        }
        const int32_t part0 = row_part0[r];
        float M = -INFINITY;
        for (int32_t i = lane; i < n; i += 32)
            M = fmaxf(M, lse_part[(size_t)(part0 + i) * kHeads + h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

        float4 acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        float W = 0.f;
        for (int32_t i = 0; i < n; ++i) {
            const size_t slot = (size_t)(part0 + i) * kHeads + h;
            const float w = expf(lse_part[slot] - M);
            W += w;
            const float4 *src = reinterpret_cast<const float4 *>(o_part + slot * kDl);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 v = src[k * 32 + lane];
                acc[k].x += w * v.x;
                acc[k].y += w * v.y;
                acc[k].z += w * v.z;
                acc[k].w += w * v.w;
            }
        }
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
        if (lane == 0) lse_out[(size_t)r * kHeads + h] = M + logf(W);
    }
}

}  // namespace

cudaError_t launch_combine(const void *ws, void *o_latent, float *lse, int32_t batch, int32_t s_q,
                           int32_t num_units, cudaStream_t stream) {
    const int64_t tasks = (int64_t)batch * s_q * kHeads;
    const int64_t need = (tasks + kCombineWarps - 1) / kCombineWarps;
    const int grid = (int)(need < kCombineGrid ? need : kCombineGrid);
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
