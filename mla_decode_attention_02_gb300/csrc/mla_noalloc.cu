// Allocation-free entry point: plan + decode with the workspace in a
// file-scope static device array, for callers that cannot allocate device
// memory on their decode path (serving loops and plugin hosts that own all
// device memory, or code where cudaMalloc's implicit synchronisation and
// unbounded latency are not allowed).  The contract is in
// include/mla_decode.h (mla_decode_noalloc).
#include <cuda_runtime.h>

#include <mutex>

#include "mla_internal.h"

namespace {

constexpr size_t kScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The shared workspace.  In host code this name is only a stand-in for the
// symbol: the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" mla_status mla_decode_noalloc(const mla_problem *prob, const void *q_latent,
                                         const void *q_rope, const void *kv_cache,
                                         int64_t num_pages, const int32_t *block_table,
                                         const int32_t *seq_lens, float scale, void *o_latent,
                                         float *lse, mla_stream_t stream) {
    mla::NvtxRange nvtx_range("mla_decode_noalloc");
    // Every argument is checked before anything is enqueued: the planner below
    // would otherwise run (and rewrite the shared array) for a call that
    // mla_decode then refuses.
    mla_status st = mla::check_decode_args(prob, q_latent, q_rope, kv_cache, num_pages, block_table,
                                           seq_lens, true, scale, o_latent, lse, nullptr, 0, false);
    if (st != MLA_OK) return st;
    size_t need = 0;
    st = mla_decode_workspace_size(prob, &need);
    if (st != MLA_OK) return st;
    if (need > kScratchBytes) return MLA_ERR_WORKSPACE;
    void *ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) return MLA_ERR_CUDA;
    // The planner rewrites the schedule header, items and status word on every
    // call, and the main kernel writes each partial slot before the merge reads
    // it, so nothing left over from an earlier call is read.
    st = mla_decode_plan(prob, seq_lens, ws, kScratchBytes, stream);
    if (st != MLA_OK) return st;
    return mla_decode(prob, q_latent, q_rope, kv_cache, num_pages, block_table, scale, o_latent,
                      lse, ws, kScratchBytes, stream);
}
