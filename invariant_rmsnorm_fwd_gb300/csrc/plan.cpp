// Host-side planner: turns one call's token ids into the work items executed
// by the dweight-contributing kernels.
//
// A logical block b holds logical rows [64b, 64b+64) (the last block holds
// the rows below N).  If every row of the block is in this call the block
// becomes one "whole" item (kind 0) listing the block's physical rows in
// logical order, and its 64-leaf tree is formed on chip.  A block that the
// call holds only partly is cut; each of its quarters (16 aligned logical
// rows, the subtrees of the block's tree one level below its two halves)
// that the call holds completely goes into one "quarter" item of that block
// (kind 2: the present quarters' rows at their places, a bit per present
// quarter), and the kernels reduce such a quarter on chip like a quarter of
// a whole block.  The remaining rows of cut blocks go, in logical order,
// into "spill" items of up to 64 rows (kind 1); their FP32 contributions are
// written to the workspace and their quarters are reduced by
// dweight_finalize with the same tree.  Padding slots (id -1) appear in no
// item.  The plan depends only on the ids, so a layout always gets the same
// plan.
#include <algorithm>
#include <cstring>
#include <utility>
#include <vector>

#include "rmsnorm_bi.h"

namespace {

constexpr int kBlockRows = 64;

struct Item {                       // must match rbi::PlanItem (528 bytes)
    int32_t kind, block, count, quarters;
    int32_t prow[kBlockRows];
    int32_t lrow[kBlockRows];
};
static_assert(sizeof(Item) == 528, "plan item layout");

void fill_item(Item &it, int32_t kind, int32_t block, const int32_t *prow, const int32_t *lrow, size_t n) {
    it.kind = kind;
    it.block = block;
    it.count = int32_t(n);
    it.quarters = 0;
    std::memcpy(it.prow, prow, n * sizeof(int32_t));
    std::memcpy(it.lrow, lrow, n * sizeof(int32_t));
    for (size_t q = n; q < size_t(kBlockRows); ++q) it.prow[q] = it.lrow[q] = -1;
}

// Per-thread working arrays, kept between calls so that planning a call every
// step does not map and fault in fresh pages each time.
struct Scratch {
    std::vector<std::pair<int32_t, int32_t>> tok;
    std::vector<int32_t> lrows, prows, sp_lrow, sp_prow, q_lrow, q_prow, q_block, q_mask, q_at;

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

// Items of a call of `rows` physical rows: at most one whole item per 64
// rows, one quarter item per complete quarter (16 rows, or fewer at the end
// of the multiset) and one spill item per 64 cut rows.
int64_t max_items(int64_t rows) { return 2 * ((rows + kBlockRows - 1) / kBlockRows) + (rows + 15) / 16 + 3; }

extern "C" int rmsnorm_plan_bytes(int64_t n_tokens, int32_t rows_per_token, size_t *bytes) {
    if (!bytes) return RMSNORM_ERR_NULL;
    if (n_tokens < 0 || rows_per_token < 1) return RMSNORM_ERR_LAYOUT;
    *bytes = size_t(max_items(n_tokens * rows_per_token)) * sizeof(Item);
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

    // whole blocks go straight to the output; complete quarters of cut blocks
    // are gathered for the quarter items, the other cut rows for the spill items
    const size_t max_out = capacity / sizeof(Item);
    Item *out = static_cast<Item *>(plan);
    size_t n_items = 0, n_sp = 0, n_qb = 0;
    int32_t *q_prow = sc.reserve(sc.q_prow, n_act_max), *q_lrow = sc.reserve(sc.q_lrow, n_act_max);
    int32_t *q_block = sc.reserve(sc.q_block, n_act_max / 16 + 2), *q_mask = sc.reserve(sc.q_mask, n_act_max / 16 + 2);
    int32_t *q_at = sc.reserve(sc.q_at, n_act_max / 16 + 2);
    size_t n_q = 0;                                              // rows gathered for quarter items
    size_t i = 0;
    while (i < n_act) {
        const int32_t b = lrows[i] / kBlockRows;
        const int64_t b0 = int64_t(b) * kBlockRows;
        const int64_t b_rows = std::min<int64_t>(kBlockRows, N - b0);
        size_t j = i;                                          // rows of block b in this call: [i, j)
        while (j < n_act && lrows[j] / kBlockRows == b) ++j;
        if (int64_t(j - i) == b_rows) {                        // rows [64b, 64b + b_rows) in order
            if (n_items == max_out) return RMSNORM_ERR_CAPACITY;
            if (!out) return RMSNORM_ERR_NULL;
            fill_item(out[n_items++], 0, b, prows + i, lrows + i, size_t(b_rows));
        } else {
            int32_t mask = 0;
            const size_t q_first = n_q;
            for (size_t k = i; k < j;) {                       // runs of rows within one quarter
                const int32_t q = int32_t((lrows[k] - b0) / 16);
                size_t e = k;
                while (e < j && (lrows[e] - b0) / 16 == q) ++e;
                const int64_t q_rows = std::min<int64_t>(16, N - (b0 + 16 * q));
                if (int64_t(e - k) == q_rows) {                // the whole quarter is in this call
                    mask |= 1 << q;
                    std::memcpy(q_lrow + n_q, lrows + k, (e - k) * sizeof(int32_t));
                    std::memcpy(q_prow + n_q, prows + k, (e - k) * sizeof(int32_t));
                    n_q += e - k;
                } else {
                    std::memcpy(sp_lrow + n_sp, lrows + k, (e - k) * sizeof(int32_t));
                    std::memcpy(sp_prow + n_sp, prows + k, (e - k) * sizeof(int32_t));
                    n_sp += e - k;
                }
                k = e;
            }
            if (mask) {
                q_block[n_qb] = b;
                q_mask[n_qb] = mask;
                q_at[n_qb] = int32_t(q_first);
                ++n_qb;
            }
        }
        i = j;
    }
    const size_t n_whole = n_items;
    for (size_t k = 0; k < n_qb; ++k) {
        if (n_items == max_out) return RMSNORM_ERR_CAPACITY;
        if (!out) return RMSNORM_ERR_NULL;
        Item &it = out[n_items++];
        const size_t r0 = size_t(q_at[k]), r1 = k + 1 < n_qb ? size_t(q_at[k + 1]) : n_q;
        it.kind = 2;
        it.block = q_block[k];
        it.count = int32_t(r1 - r0);
        it.quarters = q_mask[k];
        for (int s = 0; s < kBlockRows; ++s) it.prow[s] = it.lrow[s] = -1;
        const int64_t b0 = int64_t(q_block[k]) * kBlockRows;
        for (size_t r = r0; r < r1; ++r) {                     // each row at its place in the block
            const int32_t slot = int32_t(q_lrow[r] - b0);
            it.prow[slot] = q_prow[r];
            it.lrow[slot] = q_lrow[r];
        }
    }
    for (size_t k = 0; k < n_sp; k += kBlockRows) {
        if (n_items == max_out) return RMSNORM_ERR_CAPACITY;
        if (!out) return RMSNORM_ERR_NULL;
        fill_item(out[n_items++], 1, -1, sp_prow + k, sp_lrow + k, std::min<size_t>(kBlockRows, n_sp - k));
    }
    *plan_items = int64_t(n_items);
    if (whole_blocks) *whole_blocks = int64_t(n_whole);
    if (spill_rows) *spill_rows = int64_t(n_sp);
    return RMSNORM_OK;
}
