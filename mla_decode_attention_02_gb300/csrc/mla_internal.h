// Internal definitions shared by the library's CUDA sources: the workspace
// layout of the split-KV schedule and the planner's per-row arithmetic,
// which the device planner and its host twin both run so that their output
// is bit-identical.
#pragma once

#include <cstddef>
#include <cstdint>

#include <nvtx3/nvToolsExt.h>

#include "mla_decode.h"

#if defined(__CUDACC__)
#define MLA_HD __host__ __device__ __forceinline__
#else
#define MLA_HD inline
#endif

namespace mla {

// An NVTX range over a C-ABI call (the host-side enqueue of its launches), for
// timelines of profiling tools; with no tool attached push and pop return at
// once (NVTX v3 is header-only and loads nothing by itself).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

constexpr int kHeads = MLA_NUM_HEADS;    // query heads sharing one latent row
constexpr int kDl = MLA_D_LATENT;        // c_kv values per cached row (also V)
constexpr int kDr = MLA_D_ROPE;          // k_rope values per cached row
constexpr int kDrow = kDl + kDr;         // 576 values per cached row
constexpr int kPage = MLA_PAGE_SIZE;     // tokens per cache page
constexpr uint32_t kPlanMagic = 0x31414c4du;  // "MLA1"

// Planner tuning, in units of one cache page of work (about 1.1 us of an SM
// pair on this part): the fixed cost of a work item (query load, pipeline
// fill, epilogue), the shortest split, and the extra cost of splitting at all
// (fp32 partials written and merged).  Per-unit end times on the mixed
// workload put an item at about 6 us (5.7 pages) and a page at 1.05 us; of
// 5, 6, 7, 8 and 10 pages per item, 7 gave the earliest kernel end on the
// mixed, MTP and long workloads (the slowest unit decides it).
constexpr int kItemCost = 7;
// A cut that would leave a piece shorter than this moves the row's head to the
// next unit (overloading it by up to kMinSplitPages - 1 pages); 4 against 8
// lowered the largest unit load on the mixed workload from 133 to 128 and its
// main kernel by about 1%.
constexpr int kMinSplitPages = 4;
constexpr int kSplitPenalty = 8;

struct PlanHeader {  // 64 bytes at workspace offset 0
    uint32_t magic;
    int32_t batch, s_q, max_pages;
    int32_t num_units, num_rows, max_items, num_items;
    int32_t num_parts, status, split, min_split;  // split: rows may be cut (1) or not (0)
    int64_t total_cost, target;
};
static_assert(sizeof(PlanHeader) == 64, "header layout");

// One contiguous key range of one (request, query token) row.
struct WorkItem {
    int32_t row;       // b * s_q + t
    int32_t kv_begin;  // first key (a multiple of the page size)
    int32_t kv_end;    // one past the last key
    int32_t part;      // partial slot, or -1: this item is the whole row
};
static_assert(sizeof(WorkItem) == 16, "item layout");

// Byte offsets of every region of the workspace.
struct PlanLayout {
    size_t items, item_unit, unit_begin, row_nparts, row_part0, row_item0, row_pos, plan_end;
    size_t lse_part, o_part, total;
    int32_t num_rows, max_items, max_parts;
};

MLA_HD size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

MLA_HD PlanLayout plan_layout(int32_t batch, int32_t s_q, int32_t num_units) {
    PlanLayout L;
    L.num_rows = batch * s_q;
    L.max_items = L.num_rows + num_units;
    L.max_parts = L.max_items;
    size_t off = sizeof(PlanHeader);
    L.items = off;
    off += sizeof(WorkItem) * (size_t)L.max_items;
    L.item_unit = off;
    off += sizeof(int32_t) * (size_t)L.max_items;
    L.unit_begin = off;
    off += sizeof(int32_t) * ((size_t)num_units + 1);
    L.row_nparts = off;
    off += sizeof(int32_t) * (size_t)L.num_rows;
    L.row_part0 = off;
    off += sizeof(int32_t) * (size_t)L.num_rows;
    L.row_item0 = off;
    off += sizeof(int32_t) * (size_t)L.num_rows;
    off = align_up(off, 8);
    L.row_pos = off;
    off += sizeof(int64_t) * (size_t)L.num_rows;
    L.plan_end = off;
    off = align_up(off, 256);
    L.lse_part = off;
    off += sizeof(float) * (size_t)L.max_parts * kHeads;
    off = align_up(off, 256);
    L.o_part = off;
    off += sizeof(float) * (size_t)L.max_parts * kHeads * kDl;
    L.total = align_up(off, 256);
    return L;
}

// Pages row r = (b, t) must read, or -1 when its seq_len is invalid.
MLA_HD int32_t row_pages(int32_t seq_len, int32_t s_q, int32_t t, int32_t max_pages) {
    int64_t vis = (int64_t)seq_len - s_q + 1 + t;
    if (seq_len < s_q || vis < 1) return -1;
    int64_t pages = (vis + kPage - 1) / kPage;
    if (seq_len > (int64_t)max_pages * kPage) return -1;
    return (int32_t)pages;
}

MLA_HD int64_t row_cost(int32_t pages) { return pages > 0 ? (int64_t)pages + kItemCost : 0; }

// Walks the unit boundaries that fall inside one row's stretch of the cost
// line [x0, x0 + cost) and cuts the row there, except where a piece would
// be shorter than kMinSplitPages: a short leading piece moves to the next
// unit, a short trailing piece stays with the previous one.  Calls
// emit(piece, first_page, end_page, unit) for every piece and returns the
// number of pieces.
#if defined(__CUDACC__)
#pragma nv_exec_check_disable
#endif
template <typename Emit>
MLA_HD int32_t cut_row(int64_t x0, int32_t pages, int64_t target, int32_t num_units, bool split,
                       Emit emit) {
    if (pages <= 0) return 0;
    const int64_t cost = row_cost(pages);
    if (!split) {  // whole row, on the unit whose stretch holds its midpoint
        int64_t unit = (x0 + cost / 2) / target;
        emit(0, 0, pages, (int32_t)(unit < num_units ? unit : num_units - 1));
        return 1;
    }
    int64_t unit = x0 / target;
    int64_t start = 0;
    int32_t n = 0;
    for (int64_t k = unit + 1; k * target < x0 + cost && k < num_units; ++k) {
        int64_t cut = k * target - x0 - kItemCost;
        if (cut - start >= kMinSplitPages && pages - cut >= kMinSplitPages) {
            emit(n, (int32_t)start, (int32_t)cut, (int32_t)unit);
            ++n;
            start = cut;
            unit = k;
        } else if (cut - start < kMinSplitPages) {
            unit = k;
        }
    }
    emit(n, (int32_t)start, pages, (int32_t)unit);
    return n + 1;
}

// Unit of a whole (unsplit) row: the one whose stretch holds its midpoint.
MLA_HD int64_t mid_unit(int64_t x0, int64_t cost, int64_t target, int32_t num_units) {
    int64_t u = (x0 + cost / 2) / target;
    return u < num_units ? u : num_units - 1;
}

struct NoEmit {
    MLA_HD void operator()(int32_t, int32_t, int32_t, int32_t) const {}
};

// Host-side argument checks of a decode call that make no CUDA call
// (mla_api.cu); shared by mla_decode and the allocation-free entry point.
mla_status check_decode_args(const mla_problem *prob, const void *q_latent, const void *q_rope,
                             const void *kv_cache, int64_t num_pages, const int32_t *block_table,
                             const int32_t *seq_lens, bool need_seq_lens, float scale,
                             const void *o_latent, const float *lse, const void *workspace,
                             size_t workspace_bytes, bool need_workspace);

}  // namespace mla
