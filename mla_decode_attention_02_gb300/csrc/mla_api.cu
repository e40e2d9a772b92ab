// C ABI entry points: argument validation, workspace bookkeeping and the
// launches of the planner, main and merge kernels.  See include/mla_decode.h
// for the contract of every function.
#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>

#include "mla_internal.h"

namespace mla {
mla_status plan_host(const mla_problem *prob, const int32_t *seq_lens, int32_t num_units,
                     uint8_t *ws);
cudaError_t launch_plan(const int32_t *seq_lens, void *ws, int32_t batch, int32_t s_q,
                        int32_t max_pages, int32_t num_units, cudaStream_t stream);
cudaError_t launch_combine(const void *ws, void *o_latent, float *lse, int32_t batch, int32_t s_q,
                           int32_t num_units, cudaStream_t stream);
cudaError_t main_units(int32_t *units);
bool plan_fits(int32_t rows, int32_t units);
cudaError_t launch_main(const void *q_latent, const void *q_rope, const void *kv,
                        int64_t num_pages, const int32_t *block_table, float scale, void *ws,
                        void *o_latent, float *lse, int32_t batch, int32_t s_q, int32_t max_pages,
                        int32_t num_units, uint64_t wait_limit_ns, uint32_t test_flags,
                        uint32_t flags, bool fp8, cudaStream_t stream);
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // a bounded device wait gives up after 2 s
}  // namespace mla

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mla_status check_problem(const mla_problem *p) {
    if (!p) return MLA_ERR_INVALID_ARG;
    if (p->batch < 1 || p->max_pages_per_seq < 1 || (p->flags & ~MLA_FLAG_POW2_MAX) != 0)
        return MLA_ERR_INVALID_ARG;
    if (p->s_q != 1 && p->s_q != 2) return MLA_ERR_UNSUPPORTED;
    if (p->num_heads != MLA_NUM_HEADS || p->page_size != MLA_PAGE_SIZE) return MLA_ERR_UNSUPPORTED;
    if ((int64_t)p->batch * p->max_pages_per_seq >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
    if ((int64_t)p->max_pages_per_seq * MLA_PAGE_SIZE >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
    if ((int64_t)p->batch * p->s_q * MLA_NUM_HEADS >= (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

// The smallest workspace any device could need for this problem (one work
// unit): a workspace below it is refused before any CUDA call.
size_t workspace_lower_bound(const mla_problem *p) {
    return mla::plan_layout(p->batch, p->s_q, 1).total;
}

}  // namespace

namespace mla {

// Every host-side check of a decode call that needs no CUDA call: the
// problem, the pointers (non-null, 16-byte aligned), the pool size, the
// scale (finite and > 0: the kernel takes the row maximum of the raw scores
// as the maximum of the scaled ones) and a lower bound on the workspace.
// seq_lens is checked when non-null is required (the allocation-free call).
mla_status check_decode_args(const mla_problem *prob, const void *q_latent, const void *q_rope,
                             const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                             const int32_t *seq_lens, bool need_seq_lens, float scale,
                             const void *o_latent, const float *lse, const void *workspace,
                             size_t workspace_bytes, bool need_workspace) {
    mla_status st = check_problem(prob);
    if (st != MLA_OK) return st;
    const void *ptrs[] = {q_latent, q_rope, kv_cache, block_table, o_latent, lse};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return MLA_ERR_INVALID_ARG;
    if (need_seq_lens && (!seq_lens || !aligned16(seq_lens))) return MLA_ERR_INVALID_ARG;
    if (need_workspace && (!workspace || !aligned16(workspace))) return MLA_ERR_INVALID_ARG;
    if (num_pages < 1 || num_pages > ((int64_t)1 << 31) - 1) return MLA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return MLA_ERR_INVALID_ARG;
    if (need_workspace && workspace_bytes < workspace_lower_bound(prob)) return MLA_ERR_WORKSPACE;
    return MLA_OK;
}

}  // namespace mla

extern "C" {

const char *mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "success";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported problem shape";
        case MLA_ERR_WORKSPACE: return "workspace too small";
        case MLA_ERR_CUDA: return "CUDA error";
        case MLA_ERR_DEVICE_CHECK: return "device reported an input error";
        case MLA_ERR_TIMEOUT: return "a bounded device wait timed out";
    }
    return "unknown status";
}

mla_status mla_decode_num_units(int32_t *units) {
    if (!units) return MLA_ERR_INVALID_ARG;
    return mla::main_units(units) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status mla_decode_workspace_size(const mla_problem *prob, size_t *bytes) {
    mla_status st = check_problem(prob);
    if (st != MLA_OK) return st;
    if (!bytes) return MLA_ERR_INVALID_ARG;
    int32_t units = 0;
    if (mla::main_units(&units) != cudaSuccess) return MLA_ERR_CUDA;
    *bytes = mla::plan_layout(prob->batch, prob->s_q, units).total;
    return MLA_OK;
}

size_t mla_decode_plan_bytes(const mla_problem *prob, int32_t num_units) {
    if (check_problem(prob) != MLA_OK || num_units < 1) return 0;
    return mla::plan_layout(prob->batch, prob->s_q, num_units).plan_end;
}

mla_status mla_decode_plan_host(const mla_problem *prob, const int32_t *seq_lens_host,
                                int32_t num_units, void *plan_host, size_t plan_bytes) {
    mla_status st = check_problem(prob);
    if (st != MLA_OK) return st;
    if (!seq_lens_host || !plan_host || num_units < 1) return MLA_ERR_INVALID_ARG;
    if (plan_bytes < mla::plan_layout(prob->batch, prob->s_q, num_units).plan_end)
        return MLA_ERR_WORKSPACE;
    return mla::plan_host(prob, seq_lens_host, num_units, static_cast<uint8_t *>(plan_host));
}

mla_status mla_decode_plan(const mla_problem *prob, const int32_t *seq_lens, void *workspace,
                           size_t workspace_bytes, mla_stream_t stream) {
    mla::NvtxRange nvtx_range("mla_decode_plan");
    mla_status st = check_problem(prob);
    if (st != MLA_OK) return st;
    if (!seq_lens || !aligned16(seq_lens) || !workspace || !aligned16(workspace))
        return MLA_ERR_INVALID_ARG;
    if (workspace_bytes < workspace_lower_bound(prob)) return MLA_ERR_WORKSPACE;
    int32_t units = 0;
    if (mla::main_units(&units) != cudaSuccess) return MLA_ERR_CUDA;
    if (!mla::plan_fits(prob->batch * prob->s_q, units)) return MLA_ERR_UNSUPPORTED;
    if (workspace_bytes < mla::plan_layout(prob->batch, prob->s_q, units).total)
        return MLA_ERR_WORKSPACE;
    cudaError_t e = mla::launch_plan(seq_lens, workspace, prob->batch, prob->s_q,
                                     prob->max_pages_per_seq, units,
                                     reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

static mla_status decode_impl(const mla_problem *prob, const void *q_latent, const void *q_rope,
                              const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                              float scale, void *o_latent, float *lse, void *workspace,
                              size_t workspace_bytes, mla_stream_t stream, void *const *events,
                              uint64_t wait_limit_ns = mla::kDefaultWaitLimitNs,
                              uint32_t test_flags = 0, bool fp8 = false) {
    mla_status st = mla::check_decode_args(prob, q_latent, q_rope, kv_cache, num_pages, block_table,
                                           nullptr, false, scale, o_latent, lse, workspace,
                                           workspace_bytes, true);
    if (st != MLA_OK) return st;
    int32_t units = 0;
    if (mla::main_units(&units) != cudaSuccess) return MLA_ERR_CUDA;
    if (workspace_bytes < mla::plan_layout(prob->batch, prob->s_q, units).total)
        return MLA_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Inside stream capture the events become external record nodes, so their
    // timestamps stay readable after the graph runs.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (events && cudaStreamIsCapturing(s, &capture) != cudaSuccess) return MLA_ERR_CUDA;
    auto mark = [&](int i) -> bool {
        if (!events || !events[i]) return true;
        cudaEvent_t ev = static_cast<cudaEvent_t>(events[i]);
        if (capture == cudaStreamCaptureStatusActive)
            return cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal) == cudaSuccess;
        return cudaEventRecord(ev, s) == cudaSuccess;
    };
    if (!mark(0)) return MLA_ERR_CUDA;
    cudaError_t e = mla::launch_main(q_latent, q_rope, kv_cache, num_pages, block_table, scale,
                                     workspace, o_latent, lse, prob->batch, prob->s_q,
                                     prob->max_pages_per_seq, units, wait_limit_ns, test_flags,
                                     (uint32_t)prob->flags, fp8, s);
    if (e != cudaSuccess || !mark(1)) return MLA_ERR_CUDA;
    e = mla::launch_combine(workspace, o_latent, lse, prob->batch, prob->s_q, units, s);
    if (e != cudaSuccess || !mark(2)) return MLA_ERR_CUDA;
    return MLA_OK;
}

mla_status mla_decode(const mla_problem *prob, const void *q_latent, const void *q_rope,
                      const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                      float scale, void *o_latent, float *lse, void *workspace,
                      size_t workspace_bytes, mla_stream_t stream) {
    mla::NvtxRange nvtx_range("mla_decode");
    return decode_impl(prob, q_latent, q_rope, kv_cache, num_pages, block_table, scale, o_latent,
                       lse, workspace, workspace_bytes, stream, nullptr);
}

mla_status mla_decode_timed(const mla_problem *prob, const void *q_latent, const void *q_rope,
                            const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                            float scale, void *o_latent, float *lse, void *workspace,
                            size_t workspace_bytes, mla_stream_t stream, void *const *events) {
    mla::NvtxRange nvtx_range("mla_decode_timed");
    return decode_impl(prob, q_latent, q_rope, kv_cache, num_pages, block_table, scale, o_latent,
                       lse, workspace, workspace_bytes, stream, events);
}

mla_status mla_decode_diag(const mla_problem *prob, const void *q_latent, const void *q_rope,
                           const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                           float scale, void *o_latent, float *lse, void *workspace,
                           size_t workspace_bytes, mla_stream_t stream, uint64_t wait_limit_ns,
                           uint32_t inject) {
    mla::NvtxRange nvtx_range("mla_decode_diag");
    if (wait_limit_ns < 1000ull || wait_limit_ns > 60000000000ull) return MLA_ERR_INVALID_ARG;
    if (inject & ~MLA_INJECT_WITHHOLD_K_LOAD) return MLA_ERR_INVALID_ARG;
    return decode_impl(prob, q_latent, q_rope, kv_cache, num_pages, block_table, scale, o_latent,
                       lse, workspace, workspace_bytes, stream, nullptr, wait_limit_ns, inject);
}

mla_status mla_decode_fp8(const mla_problem *prob, const void *q_latent, const void *q_rope,
                          const void *kv_cache_fp8, int64_t num_pages, const int32_t *block_table,
                          float scale, void *o_latent, float *lse, void *workspace,
                          size_t workspace_bytes, mla_stream_t stream, void *const *events) {
    mla::NvtxRange nvtx_range("mla_decode_fp8");
    return decode_impl(prob, q_latent, q_rope, kv_cache_fp8, num_pages, block_table, scale, o_latent,
                       lse, workspace, workspace_bytes, stream, events, mla::kDefaultWaitLimitNs, 0, true);
}

mla_status mla_decode_check(const void *workspace, int32_t *device_status, mla_stream_t stream) {
    if (!workspace || !device_status) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
    int32_t v = 0;
    const char *src = static_cast<const char *>(workspace) + offsetof(mla::PlanHeader, status);
    if (cudaMemcpy(&v, src, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
    *device_status = v;
    if (v == 0) return MLA_OK;
    return (v & MLA_DEV_TIMEOUT) ? MLA_ERR_TIMEOUT : MLA_ERR_DEVICE_CHECK;
}

}  // extern "C"
