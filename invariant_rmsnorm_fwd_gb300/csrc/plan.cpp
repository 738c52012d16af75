// Host-side planner: turns one call's token ids into the work items executed
// by the dweight-contributing kernels.
//
// A logical block b holds logical rows [64b, 64b+64) (the last block holds
// the rows below N).  If every row of the block is in this call the block
// becomes one "whole" item listing the block's physical rows in logical
// order, and its 64-leaf tree is formed on chip.  Rows of blocks that the
// call holds only partly go, in logical order, into "spill" items of up to
// 64 rows; their FP32 contributions are written to the workspace and the
// block is reduced later by dweight_finalize with the same tree.  Padding
// slots (id -1) appear in no item.  The plan depends only on the ids, so a
// layout always gets the same plan.
#include <algorithm>
#include <cstring>
#include <utility>
#include <vector>

#include "rmsnorm_bi.h"

namespace {

constexpr int kBlockRows = 64;

struct Item {                       // must match rbi::PlanItem (528 bytes)
    int32_t kind, block, count, reserved;
    int32_t prow[kBlockRows];
    int32_t lrow[kBlockRows];
};
static_assert(sizeof(Item) == 528, "plan item layout");

void fill_item(Item &it, int32_t kind, int32_t block, const int32_t *prow, const int32_t *lrow, size_t n) {
    it.kind = kind;
    it.block = block;
    it.count = int32_t(n);
    it.reserved = 0;
    std::memcpy(it.prow, prow, n * sizeof(int32_t));
    std::memcpy(it.lrow, lrow, n * sizeof(int32_t));
    for (size_t q = n; q < size_t(kBlockRows); ++q) it.prow[q] = it.lrow[q] = -1;
}

// Per-thread working arrays, kept between calls so that planning a call every
// step does not map and fault in fresh pages each time.
struct Scratch {
    std::vector<std::pair<int32_t, int32_t>> tok;
    std::vector<int32_t> lrows, prows, sp_lrow, sp_prow;

    template <class T>
    T *reserve(std::vector<T> &v, size_t n) {                 // grows only; contents are scratch
        if (v.size() < n) v.resize(n);
        return v.data();
    }
};

Scratch &scratch() {
    thread_local Scratch s;
    return s;
}

}  // namespace

extern "C" int rmsnorm_plan_bytes(int64_t n_tokens, int32_t rows_per_token, size_t *bytes) {
    if (!bytes) return RMSNORM_ERR_NULL;
    if (n_tokens < 0 || rows_per_token < 1) return RMSNORM_ERR_LAYOUT;
    const int64_t rows = n_tokens * rows_per_token;
    const int64_t items = 2 * ((rows + kBlockRows - 1) / kBlockRows) + 2;
    *bytes = size_t(items) * sizeof(Item);
    return RMSNORM_OK;
}

extern "C" int rmsnorm_plan_build(const int32_t *tok_id, int64_t n_tokens, int32_t rows_per_token,
                                  int64_t n_logical_tokens, void *plan, size_t capacity, int64_t *plan_items,
                                  int64_t *whole_blocks, int64_t *spill_rows) {
    if (!plan_items || (n_tokens > 0 && !tok_id)) return RMSNORM_ERR_NULL;
    if (n_tokens < 0 || rows_per_token < 1 || n_logical_tokens < 0) return RMSNORM_ERR_LAYOUT;
    const int64_t R = rows_per_token;
    const int64_t N = n_logical_tokens * R;                    // logical rows
    if (n_tokens * R >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return RMSNORM_ERR_LAYOUT;
    Scratch &sc = scratch();
    using Tok = std::pair<int32_t, int32_t>;                   // (id, slot)
    const size_t n_act_max = size_t(n_tokens) * size_t(R);
    Tok *tok = sc.reserve(sc.tok, size_t(n_tokens));
    int32_t *lrows = sc.reserve(sc.lrows, n_act_max), *prows = sc.reserve(sc.prows, n_act_max);
    int32_t *sp_lrow = sc.reserve(sc.sp_lrow, n_act_max), *sp_prow = sc.reserve(sc.sp_prow, n_act_max);

    // active tokens sorted by logical id (ids of a call usually arrive ascending:
    // the sort is skipped then)
    size_t n_tok = 0;
    bool ascending = true;
    for (int64_t t = 0; t < n_tokens; ++t) {
        const int32_t id = tok_id[t];
        if (id < -1 || id >= n_logical_tokens) return RMSNORM_ERR_ID;
        if (id >= 0) {
            if (n_tok && id <= tok[n_tok - 1].first) ascending = false;
            tok[n_tok++] = Tok(id, int32_t(t));
        }
    }
    if (!ascending) {
        std::sort(tok, tok + n_tok);
        for (size_t i = 1; i < n_tok; ++i)
            if (tok[i].first == tok[i - 1].first) return RMSNORM_ERR_DUPLICATE;
    }

    // rows in logical order: token id*R + h sits at physical row slot*R + h
    const size_t n_act = n_tok * size_t(R);
    for (size_t t = 0, k = 0; t < n_tok; ++t) {
        const int32_t l0 = int32_t(int64_t(tok[t].first) * R), p0 = int32_t(int64_t(tok[t].second) * R);
        for (int32_t h = 0; h < int32_t(R); ++h, ++k) {
            lrows[k] = l0 + h;
            prows[k] = p0 + h;
        }
    }

    // whole blocks go straight to the output, cut rows are gathered for the spill items
    const size_t max_items = capacity / sizeof(Item);
    Item *out = static_cast<Item *>(plan);
    size_t n_items = 0, n_sp = 0;
    size_t i = 0;
    while (i < n_act) {
        const int32_t b = lrows[i] / kBlockRows;
        const int64_t b_rows = std::min<int64_t>(kBlockRows, N - int64_t(b) * kBlockRows);
        size_t j = i;                                          // rows of block b in this call: [i, j)
        while (j < n_act && lrows[j] / kBlockRows == b) ++j;
        if (int64_t(j - i) == b_rows) {                        // rows [64b, 64b + b_rows) in order
            if (n_items == max_items) return RMSNORM_ERR_CAPACITY;
            if (!out) return RMSNORM_ERR_NULL;
            fill_item(out[n_items++], 0, b, prows + i, lrows + i, size_t(b_rows));
        } else {
            std::memcpy(sp_lrow + n_sp, lrows + i, (j - i) * sizeof(int32_t));
            std::memcpy(sp_prow + n_sp, prows + i, (j - i) * sizeof(int32_t));
            n_sp += j - i;
        }
        i = j;
    }
    const size_t n_whole = n_items;
    for (size_t k = 0; k < n_sp; k += kBlockRows) {
        if (n_items == max_items) return RMSNORM_ERR_CAPACITY;
        if (!out) return RMSNORM_ERR_NULL;
        fill_item(out[n_items++], 1, -1, sp_prow + k, sp_lrow + k, std::min<size_t>(kBlockRows, n_sp - k));
    }
    *plan_items = int64_t(n_items);
    if (whole_blocks) *whole_blocks = int64_t(n_whole);
    if (spill_rows) *spill_rows = int64_t(n_sp);
    return RMSNORM_OK;
}
