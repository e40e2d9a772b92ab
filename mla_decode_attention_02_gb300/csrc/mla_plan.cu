// Length-aware split-KV planner.
//
// The Atlas 800I A3 TPOT-jitter troubleshooting post ("MLAKernel performance
// root cause") traces whole-DP-group stalls to batches that mix long and
// short sequences: the split-KV (FlashDecoding) path stopped firing and one
// long row ran on its own.  Section 8 of the Ascend DeepSeek report asks for
// sequence-load balancing for the same reason.  Inside one GPU the analogue
// is: give every work unit (an SM pair of the main kernel) the same number
// of cache pages, cutting long rows at page boundaries and packing short
// rows together, whatever the length mix.
//
// Every row (request b, query token t) costs pages + kItemCost on a cost
// line laid out token-major (line_row below); the line is cut into num_units stretches of
// `target` = ceil(total / num_units).  If no row is much longer than a
// stretch, rows stay whole and each goes to the unit whose stretch holds its
// midpoint (no partial outputs, no merge); otherwise each row is cut where a
// stretch boundary falls inside it (cut_row).  The choice compares the
// largest unit load without cuts against target + kItemCost + kSplitPenalty.  Rows keep their line order,
// items are emitted in that order, and units come out non-decreasing, so the unit of
// every item follows from prefix sums alone: no atomics, no sorting, and
// the same bytes on every run.  The host twin below runs the identical
// integer arithmetic sequentially.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kPlanThreads = 256;   // one CTA; fewer threads make its block-wide barriers cheaper
static_assert(kPlanThreads % 32 == 0 && kPlanThreads <= 1024, "planner block");
constexpr size_t kMaxPlanSmem = 200 * 1024;  // per-row working set of the planner kernel

// Row at position k of the cost line: token-major (every request's query token
// 0, then every request's token 1, ...), so with s_q = 2 the two tokens of a
// request sit half a line apart and run at the same time on units half the GPU
// apart, the second reading the request's pages while the first has just
// brought them into L2 (one pass per token otherwise streams the cache from
// DRAM twice).  With s_q = 1 this is row order.
MLA_HD int32_t line_row(int32_t k, int32_t batch, int32_t s_q) {
    return (k % batch) * s_q + k / batch;
}


// Inclusive block-wide sum of one int64 per thread (kPlanThreads threads, at
// most 32 warps).
__device__ int64_t block_inclusive_sum(int64_t v, int64_t *warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < kPlanThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    int64_t r = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    __syncthreads();
    return r;
}

// Shared-memory bytes the planner kernel needs for R rows and U units.
size_t plan_smem_bytes(int32_t R, int32_t U) {
    return sizeof(int64_t) * ((size_t)R + U) + sizeof(int32_t) * (2 * (size_t)R + U);
}

__global__ void __launch_bounds__(kPlanThreads, 1)
mla_plan_kernel(const int32_t *__restrict__ seq_lens, uint8_t *__restrict__ ws, int32_t batch,
                int32_t s_q, int32_t max_pages, int32_t num_units) {
    __shared__ int64_t warp_sums[32];
    __shared__ int64_t carry, carry_parts, max_load;
    __shared__ int32_t bad;
    extern __shared__ int64_t plan_smem[];
    const PlanLayout L = plan_layout(batch, s_q, num_units);
    const int32_t R = L.num_rows;
    int64_t *s_pos = plan_smem;                                        // [R] cost-line start
    int64_t *first_pos = s_pos + R;                                    // [U] (no-split runs)
    int32_t *s_pages = reinterpret_cast<int32_t *>(first_pos + num_units);  // [R]
    int32_t *s_unit = s_pages + R;                                     // [R + U] unit of each item
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(ws);
    WorkItem *items = reinterpret_cast<WorkItem *>(ws + L.items);
    int32_t *item_unit = reinterpret_cast<int32_t *>(ws + L.item_unit);
    int32_t *unit_begin = reinterpret_cast<int32_t *>(ws + L.unit_begin);
    int32_t *row_nparts = reinterpret_cast<int32_t *>(ws + L.row_nparts);
    int32_t *row_part0 = reinterpret_cast<int32_t *>(ws + L.row_part0);
    int32_t *row_item0 = reinterpret_cast<int32_t *>(ws + L.row_item0);
    int64_t *row_pos = reinterpret_cast<int64_t *>(ws + L.row_pos);

    // The main kernel may start its prologue now; it waits for this grid before
    // reading the schedule.
    ptx::pdl_launch_dependents();
    // Pass 1: pages of every row and its cost-line position (exclusive prefix of costs).
    if (threadIdx.x == 0) {
        carry = 0;
        carry_parts = 0;
        max_load = 0;
        bad = 0;
    }
    __syncthreads();
    for (int32_t base = 0; base < R; base += kPlanThreads) {
        const int32_t k = base + threadIdx.x;
        const int32_t r = k < R ? line_row(k, batch, s_q) : R;
        int64_t c = 0;
        if (r < R) {
            const int32_t p = row_pages(seq_lens[r / s_q], s_q, r % s_q, max_pages);
            if (p < 0) bad = 1;
            s_pages[r] = p;
            c = row_cost(p);
        }
        const int64_t incl = block_inclusive_sum(c, warp_sums);
        if (r < R) {
            s_pos[r] = carry + incl - c;
            row_pos[r] = carry + incl - c;
        }
        __syncthreads();
        if (threadIdx.x == kPlanThreads - 1) carry += incl;
        __syncthreads();
    }
    const int64_t total = carry;
    const int64_t target = total > 0 ? (total + num_units - 1) / num_units : 1;
    __syncthreads();

    // Pass 1b: largest unit load if no row is cut (rows on their midpoint units).
    for (int32_t k = threadIdx.x; k < R; k += kPlanThreads) {
        const int32_t r = line_row(k, batch, s_q);
        const int64_t u = mid_unit(s_pos[r], row_cost(s_pages[r]), target, num_units);
        const int32_t rp = k > 0 ? line_row(k - 1, batch, s_q) : 0;
        if (k == 0 || mid_unit(s_pos[rp], row_cost(s_pages[rp]), target, num_units) != u)
            first_pos[u] = s_pos[r];
    }
    __syncthreads();
    {
        int64_t my_max = 0;
        for (int32_t k = threadIdx.x; k < R; k += kPlanThreads) {
            const int32_t r = line_row(k, batch, s_q);
            const int64_t c = row_cost(s_pages[r]);
            const int64_t u = mid_unit(s_pos[r], c, target, num_units);
            const int32_t rn = k < R - 1 ? line_row(k + 1, batch, s_q) : 0;
            if (k == R - 1 || mid_unit(s_pos[rn], row_cost(s_pages[rn]), target, num_units) != u) {
                const int64_t load = s_pos[r] + c - first_pos[u];
                my_max = load > my_max ? load : my_max;
            }
        }
        atomicMax(reinterpret_cast<unsigned long long *>(&max_load), (unsigned long long)my_max);
    }
    __syncthreads();
    const bool split = target + kItemCost + kSplitPenalty < max_load;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();

    // Pass 2: pieces per row -> first item and first partial slot; emit the items.
    for (int32_t base = 0; base < R; base += kPlanThreads) {
        const int32_t k = base + threadIdx.x;
        const int32_t r = k < R ? line_row(k, batch, s_q) : R;
        int64_t n = 0, np = 0;
        if (r < R) {
            n = cut_row(s_pos[r], s_pages[r], target, num_units, split, NoEmit{});
            np = n > 1 ? n : 0;
        }
        const int64_t incl_n = block_inclusive_sum(n, warp_sums);
        const int64_t incl_p = block_inclusive_sum(np, warp_sums);
        if (r < R) {
            const int32_t first = (int32_t)(carry + incl_n - n);
            const int32_t part0 = n > 1 ? (int32_t)(carry_parts + incl_p - np) : -1;
            row_item0[r] = first;
            row_part0[r] = part0;
            row_nparts[r] = (int32_t)n;
            const int32_t t = r % s_q;
            const int32_t vis = s_pages[r] > 0 ? seq_lens[r / s_q] - s_q + 1 + t : 0;
            cut_row(s_pos[r], s_pages[r], target, num_units, split,
                    [&](int32_t i, int32_t pg0, int32_t pg1, int32_t unit) {
                        WorkItem it;
                        it.row = r;
                        it.kv_begin = pg0 * kPage;
                        it.kv_end = min(pg1 * kPage, vis);
                        it.part = part0 >= 0 ? part0 + i : -1;
                        items[first + i] = it;
                        item_unit[first + i] = unit;
                        s_unit[first + i] = unit;
                    });
        }
        __syncthreads();
        if (threadIdx.x == kPlanThreads - 1) {
            carry += incl_n;
            carry_parts += incl_p;
        }
        __syncthreads();
    }
    const int32_t num_items = (int32_t)carry;
    const int32_t num_parts = (int32_t)carry_parts;

    // Pass 3: unit_begin[u] = first item whose unit is >= u (units are
    // non-decreasing along the items).
    for (int32_t i = threadIdx.x; i < num_items; i += kPlanThreads) {
        const int32_t u = s_unit[i];
        const int32_t u_prev = i > 0 ? s_unit[i - 1] : -1;
        for (int32_t v = u_prev + 1; v <= u; ++v) unit_begin[v] = i;
        if (i == num_items - 1)
            for (int32_t v = u + 1; v <= num_units; ++v) unit_begin[v] = num_items;
    }
    if (num_items == 0)
        for (int32_t v = threadIdx.x; v <= num_units; v += kPlanThreads) unit_begin[v] = 0;

    if (threadIdx.x == 0) {
        PlanHeader h;
        h.magic = kPlanMagic;
        h.batch = batch;
        h.s_q = s_q;
        h.max_pages = max_pages;
        h.num_units = num_units;
        h.num_rows = R;
        h.max_items = L.max_items;
        h.num_items = num_items;
        h.num_parts = num_parts;
        h.status = bad ? MLA_DEV_BAD_SEQ_LEN : 0;
        h.split = split ? 1 : 0;
        h.min_split = kMinSplitPages;
        h.total_cost = total;
        h.target = target;
        *hdr = h;
    }
}

}  // namespace

// Host twin of mla_plan_kernel (same integer arithmetic, sequential).
mla_status plan_host(const mla_problem *prob, const int32_t *seq_lens, int32_t num_units,
                     uint8_t *ws) {
    const int32_t batch = prob->batch, s_q = prob->s_q, max_pages = prob->max_pages_per_seq;
    const PlanLayout L = plan_layout(batch, s_q, num_units);
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(ws);
    WorkItem *items = reinterpret_cast<WorkItem *>(ws + L.items);
    int32_t *item_unit = reinterpret_cast<int32_t *>(ws + L.item_unit);
    int32_t *unit_begin = reinterpret_cast<int32_t *>(ws + L.unit_begin);
    int32_t *row_nparts = reinterpret_cast<int32_t *>(ws + L.row_nparts);
    int32_t *row_part0 = reinterpret_cast<int32_t *>(ws + L.row_part0);
    int32_t *row_item0 = reinterpret_cast<int32_t *>(ws + L.row_item0);
    int64_t *row_pos = reinterpret_cast<int64_t *>(ws + L.row_pos);
    const int32_t R = L.num_rows;
    int bad = 0;
    int64_t total = 0;
    for (int32_t k = 0; k < R; ++k) {
        const int32_t r = line_row(k, batch, s_q);
        int32_t p = row_pages(seq_lens[r / s_q], s_q, r % s_q, max_pages);
        if (p < 0) bad = 1;
        row_pos[r] = total;
        total += row_cost(p);
    }
    const int64_t target = total > 0 ? (total + num_units - 1) / num_units : 1;
    // largest unit load if no row is cut (rows on their midpoint units)
    int64_t max_load = 0, run_first = 0, run_unit = -1;
    for (int32_t k = 0; k < R; ++k) {
        const int32_t r = line_row(k, batch, s_q);
        const int64_t c = row_cost(row_pages(seq_lens[r / s_q], s_q, r % s_q, max_pages));
        const int64_t u = mid_unit(row_pos[r], c, target, num_units);
        if (u != run_unit) {
            run_unit = u;
            run_first = row_pos[r];
        }
        const int64_t load = row_pos[r] + c - run_first;
        if (load > max_load) max_load = load;
    }
    const bool split = target + kItemCost + kSplitPenalty < max_load;
    int32_t n_items = 0, n_parts = 0, last_unit = -1;
    for (int32_t k = 0; k < R; ++k) {
        const int32_t r = line_row(k, batch, s_q);
        const int32_t b = r / s_q, t = r % s_q;
        const int32_t p = row_pages(seq_lens[b], s_q, t, max_pages);
        const int32_t n = cut_row(row_pos[r], p, target, num_units, split, NoEmit{});
        const int32_t part0 = n > 1 ? n_parts : -1;
        const int32_t vis = p > 0 ? seq_lens[b] - s_q + 1 + t : 0;
        cut_row(row_pos[r], p, target, num_units, split,
                [&](int32_t i, int32_t pg0, int32_t pg1, int32_t unit) {
                    WorkItem it;
                    it.row = r;
                    it.kv_begin = pg0 * kPage;
                    it.kv_end = pg1 * kPage < vis ? pg1 * kPage : vis;
                    it.part = part0 >= 0 ? part0 + i : -1;
                    items[n_items + i] = it;
                    item_unit[n_items + i] = unit;
                    for (int32_t v = last_unit + 1; v <= unit; ++v) unit_begin[v] = n_items + i;
                    if (unit > last_unit) last_unit = unit;
                });
        row_nparts[r] = n;
        row_part0[r] = part0;
        row_item0[r] = n_items;
        n_items += n;
        if (n > 1) n_parts += n;
    }
    for (int32_t v = last_unit + 1; v <= num_units; ++v) unit_begin[v] = n_items;
    PlanHeader h;
    h.magic = kPlanMagic;
    h.batch = batch;
    h.s_q = s_q;
    h.max_pages = max_pages;
    h.num_units = num_units;
    h.num_rows = R;
    h.max_items = L.max_items;
    h.num_items = n_items;
    h.num_parts = n_parts;
    h.status = bad ? MLA_DEV_BAD_SEQ_LEN : 0;
    h.split = split ? 1 : 0;
    h.min_split = kMinSplitPages;
    h.total_cost = total;
    h.target = target;
    *hdr = h;
    return MLA_OK;
}

cudaError_t launch_plan(const int32_t *seq_lens, void *ws, int32_t batch, int32_t s_q,
                        int32_t max_pages, int32_t num_units, cudaStream_t stream) {
    const size_t smem = plan_smem_bytes(batch * s_q, num_units);
    if (smem > kMaxPlanSmem) return cudaErrorInvalidValue;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(mla_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kMaxPlanSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    mla_plan_kernel<<<1, kPlanThreads, smem, stream>>>(seq_lens, static_cast<uint8_t *>(ws), batch,
                                                       s_q, max_pages, num_units);
    return cudaGetLastError();
}

bool plan_fits(int32_t rows, int32_t units) { return plan_smem_bytes(rows, units) <= kMaxPlanSmem; }

}  // namespace mla
