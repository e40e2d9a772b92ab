// Plain CUDA-core version of the main attention kernel: one CTA per (work
// unit, head), one key at a time per warp.  It exists to validate the
// schedule, the split merge and the C ABI end to end; the tensor-core
// kernel replaces it on the hot path.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla_internal.h"

namespace mla {
namespace {

__global__ void __launch_bounds__(128)
mla_main_simt_kernel(const __nv_bfloat16 *__restrict__ q_latent,
                     const __nv_bfloat16 *__restrict__ q_rope,
                     const __nv_bfloat16 *__restrict__ kv, int64_t num_pages,
                     const int32_t *__restrict__ block_table, float scale_log2, uint8_t *ws,
                     __nv_bfloat16 *__restrict__ o_latent, float *__restrict__ lse_out,
                     int32_t batch, int32_t s_q, int32_t max_pages, int32_t num_units) {
    __shared__ float q[kDrow];
    __shared__ float s[kPage];
    const PlanLayout L = plan_layout(batch, s_q, num_units);
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(ws);
    const WorkItem *items = reinterpret_cast<const WorkItem *>(ws + L.items);
    const int32_t *unit_begin = reinterpret_cast<const int32_t *>(ws + L.unit_begin);
    float *lse_part = reinterpret_cast<float *>(ws + L.lse_part);
    float *o_part = reinterpret_cast<float *>(ws + L.o_part);
    const int u = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    if (hdr->magic != kPlanMagic || hdr->batch != batch || hdr->s_q != s_q ||
        hdr->num_units != num_units || hdr->max_pages != max_pages) {
        if (tid == 0 && h == 0) atomicOr(&hdr->status, MLA_DEV_BAD_PLAN);
        return;
    }
    for (int32_t i = unit_begin[u]; i < unit_begin[u + 1]; ++i) {
        const WorkItem it = items[i];
        const int32_t b = it.row / s_q;
        const size_t qrow = (size_t)it.row * kHeads + h;
        __syncthreads();
        for (int d = tid; d < kDrow; d += 128)
            q[d] = d < kDl ? __bfloat162float(q_latent[qrow * kDl + d])
                           : __bfloat162float(q_rope[qrow * kDr + (d - kDl)]);
        __syncthreads();
        float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
        bool bad = false;
        for (int32_t j0 = it.kv_begin; j0 < it.kv_end; j0 += kPage) {
            const int32_t page = block_table[(size_t)b * max_pages + j0 / kPage];
            const int valid = min(kPage, it.kv_end - j0);
            if (page < 0 || page >= num_pages) {
                bad = true;
                continue;
            }
            const __nv_bfloat16 *base = kv + (size_t)page * kPage * kDrow;
            for (int k = warp; k < valid; k += 4) {
                const __nv_bfloat16 *row = base + (size_t)k * kDrow;
                float acc_s = 0.f;
                for (int d = lane; d < kDrow; d += 32) acc_s += q[d] * __bfloat162float(row[d]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc_s += __shfl_xor_sync(0xffffffffu, acc_s, o);
                if (lane == 0) s[k] = acc_s * scale_log2;
            }
            __syncthreads();
            float m_loc = -INFINITY;
            for (int k = 0; k < valid; ++k) m_loc = fmaxf(m_loc, s[k]);
            const float m_new = fmaxf(m, m_loc);
            const float alpha = exp2f(m - m_new);
            l *= alpha;
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] *= alpha;
            for (int k = 0; k < valid; ++k) {
                const float p = exp2f(s[k] - m_new);
                l += p;
                const __nv_bfloat16 *row = base + (size_t)k * kDrow;
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[c] += p * __bfloat162float(row[tid + 128 * c]);
            }
            m = m_new;
            __syncthreads();
        }
        const float nan = __int_as_float(0x7fc00000);
        const float inv = bad ? nan : 1.f / l;
        const float lse = bad ? nan : (m + log2f(l)) * 0.69314718055994531f;
        if (bad && tid == 0) atomicOr(&hdr->status, MLA_DEV_BAD_PAGE);
        if (it.part < 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                o_latent[qrow * kDl + tid + 128 * c] = __float2bfloat16(acc[c] * inv);
            if (tid == 0) lse_out[qrow] = lse;
        } else {
            const size_t slot = (size_t)it.part * kHeads + h;
#pragma unroll
            for (int c = 0; c < 4; ++c) o_part[slot * kDl + tid + 128 * c] = acc[c] * inv;
            if (tid == 0) lse_part[slot] = lse;
        }
    }
}

}  // namespace

cudaError_t launch_main_simt(const void *q_latent, const void *q_rope, const void *kv,
                             int64_t num_pages, const int32_t *block_table, float scale, void *ws,
                             void *o_latent, float *lse, int32_t batch, int32_t s_q,
                             int32_t max_pages, int32_t num_units, cudaStream_t stream) {
    dim3 grid(num_units, kHeads);
    const float scale_log2 = scale * 1.4426950408889634f;
    mla_main_simt_kernel<<<grid, 128, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(q_latent), static_cast<const __nv_bfloat16 *>(q_rope),
        static_cast<const __nv_bfloat16 *>(kv), num_pages, block_table, scale_log2,
        static_cast<uint8_t *>(ws), static_cast<__nv_bfloat16 *>(o_latent), lse, batch, s_q,
        max_pages, num_units);
    return cudaGetLastError();
}

cudaError_t main_units(int32_t *units) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    *units = sms;
    return cudaSuccess;
}

cudaError_t launch_main(const void *q_latent, const void *q_rope, const void *kv,
                        int64_t num_pages, const int32_t *block_table, float scale, void *ws,
                        void *o_latent, float *lse, int32_t batch, int32_t s_q, int32_t max_pages,
                        int32_t num_units, cudaStream_t stream) {
    return launch_main_simt(q_latent, q_rope, kv, num_pages, block_table, scale, ws, o_latent,
                            lse, batch, s_q, max_pages, num_units, stream);
}

}  // namespace mla
