// fp8 (e4m3) latent cache: the quantiser of the row format in include/mla_fp8.h.
//
// One warp per row (a token): lane l owns c_kv values [16 l, 16 l + 16) as two
// 16-byte loads; the row's max |c_kv| is a warp max (exact), s = max / 448 and
// each quotient c_kv / s are IEEE fp32 divisions, and the hardware conversion
// rounds each quotient to the nearest e4m3 code (ties to even, saturating).
// Lanes 0-7 write k_rope / s (fp32 division, rounded to bf16), lane 8 writes s
// and the zero padding.  Memory-bound:
// 1152 bytes read and 656 written per row, all 16-byte accesses.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mla_fp8.h"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kRowsPerCta = 8;
constexpr int kRowIn = kDrow * 2;            // 1152 bytes
constexpr int kRowOut = MLA_FP8_ROW_BYTES;   // 656 bytes
static_assert(kRowOut % 16 == 0 && kRowOut >= kDl + 2 * kDr + 4, "row layout");

__global__ void __launch_bounds__(32 * kRowsPerCta) mla_quantize_fp8_kernel(const uint8_t *__restrict__ in,
                                                                        int64_t rows,
                                                                        uint8_t *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + threadIdx.x / 32;
    if (row >= rows) return;
    const uint8_t *src = in + row * kRowIn;
    uint8_t *dst = out + row * kRowOut;
    const uint4 a = reinterpret_cast<const uint4 *>(src)[2 * lane];
    const uint4 b = reinterpret_cast<const uint4 *>(src)[2 * lane + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float x[16];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
        x[2 * j] = f.x;
        x[2 * j + 1] = f.y;
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t v = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_fp8_storage_t code = __nv_cvt_float_to_fp8(__fdiv_rn(x[4 * q + k], s), __NV_SATFINITE,
                                                                  __NV_E4M3);
            v |= (uint32_t)code << (8 * k);
        }
        c[q] = v;
    }
    reinterpret_cast<uint4 *>(dst)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
    if (lane < kDr * 2 / 16) {
        const uint4 r = reinterpret_cast<const uint4 *>(src + kDl * 2)[lane];
        uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&rw[j]));
            const __nv_bfloat162 h = __halves2bfloat162(__float2bfloat16_rn(__fdiv_rn(f.x, s)),
                                                        __float2bfloat16_rn(__fdiv_rn(f.y, s)));
            rw[j] = *reinterpret_cast<const uint32_t *>(&h);
        }
        reinterpret_cast<uint4 *>(dst + kDl)[lane] = make_uint4(rw[0], rw[1], rw[2], rw[3]);
    } else if (lane == kDr * 2 / 16) {
        reinterpret_cast<uint4 *>(dst + kDl + kDr * 2)[0] = make_uint4(__float_as_uint(s), 0u, 0u, 0u);
    }
}

}  // namespace
}  // namespace mla

extern "C" mla_status mla_cache_quantize_fp8(const void *kv_cache, int64_t num_rows, void *kv_cache_fp8,
                                             mla_stream_t stream) {
    mla::NvtxRange nvtx_range("mla_cache_quantize_fp8");
    using namespace mla;
    if (!kv_cache || !kv_cache_fp8 || num_rows < 1 || (reinterpret_cast<uintptr_t>(kv_cache) & 15u) ||
        (reinterpret_cast<uintptr_t>(kv_cache_fp8) & 15u))
        return MLA_ERR_INVALID_ARG;
    const int64_t ctas = (num_rows + kRowsPerCta - 1) / kRowsPerCta;
    if (ctas >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
    mla_quantize_fp8_kernel<<<(unsigned)ctas, 32 * kRowsPerCta, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(kv_cache), num_rows, static_cast<uint8_t *>(kv_cache_fp8));
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
