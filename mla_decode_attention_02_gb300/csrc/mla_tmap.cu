// Tensor-map encoding for the prolog and epilog kernels: rank-4 bf16 views with a
// 128-byte-swizzled box (64 values, rows, blocks, 1), and row-major matrices
// seen as (64 values, rows, K blocks).  The driver entry point is
// looked up once through the runtime, so the library needs no link to libcuda.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace mla {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

// dims (64, d1, d2, d3), byte strides (s1, s2, s3) of dims 1-3, box (64, rows, blocks, 1).
bool encode_bf16_4d(CUtensorMap *m, const void *base, cuuint64_t d1, cuuint64_t d2, cuuint64_t d3,
                    cuuint64_t s1, cuuint64_t s2, cuuint64_t s3, cuuint32_t rows, cuuint32_t blocks) {
    auto fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[4] = {64, d1, d2, d3};
    const cuuint64_t strides[3] = {s1, s2, s3};
    const cuuint32_t box[4] = {64, rows, blocks, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major bf16 matrix [rows][cols] (cols a multiple of 64) seen as (64 values, rows,
// cols / 64 blocks) with the block stride (128 bytes) below the row stride: a box
// (64, box_rows, box_blocks) lands as box_blocks stacked [box_rows][64 values] tiles,
// 128-byte swizzled, one per 64-value block of K.  Rows past the end read zeros.
bool encode_bf16_kblocks(CUtensorMap *m, const void *base, cuuint64_t cols, cuuint64_t rows,
                         cuuint32_t box_rows, cuuint32_t box_blocks) {
    auto fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {64, rows, cols / 64};
    const cuuint64_t strides[2] = {cols * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, box_blocks};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mla
