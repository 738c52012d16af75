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

void clear_item(Item &it) {
    std::memset(&it, 0, sizeof it);
    for (int i = 0; i < kBlockRows; ++i) it.prow[i] = it.lrow[i] = -1;
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

    // active tokens sorted by logical id
    std::vector<std::pair<int32_t, int32_t>> tok;             // (id, slot)
    tok.reserve(size_t(n_tokens));
    for (int64_t t = 0; t < n_tokens; ++t) {
        const int32_t id = tok_id[t];
        if (id < -1 || id >= n_logical_tokens) return RMSNORM_ERR_ID;
        if (id >= 0) tok.emplace_back(id, int32_t(t));
    }
    std::sort(tok.begin(), tok.end());
    for (size_t i = 1; i < tok.size(); ++i)
        if (tok[i].first == tok[i - 1].first) return RMSNORM_ERR_DUPLICATE;

    // rows in logical order: token id*R + h sits at physical row slot*R + h
    const size_t n_act = tok.size() * size_t(R);
    std::vector<Item> whole, spill;
    std::vector<int32_t> sp_prow, sp_lrow;
    size_t i = 0;
    while (i < n_act) {
        const int64_t lrow0 = int64_t(tok[i / R].first) * R + int64_t(i % R);
        const int64_t b = lrow0 / kBlockRows;
        const int64_t b_rows = std::min<int64_t>(kBlockRows, N - b * kBlockRows);
        size_t j = i;                                          // rows of block b in this call: [i, j)
        while (j < n_act && (int64_t(tok[j / R].first) * R + int64_t(j % R)) / kBlockRows == b) ++j;
        if (int64_t(j - i) == b_rows) {
            Item it;
            clear_item(it);
            it.kind = 0;
            it.block = int32_t(b);
            it.count = int32_t(b_rows);
            for (size_t k = i; k < j; ++k) {
                const int64_t lrow = int64_t(tok[k / R].first) * R + int64_t(k % R);
                const int s = int(lrow - b * kBlockRows);
                it.prow[s] = int32_t(int64_t(tok[k / R].second) * R + int64_t(k % R));
                it.lrow[s] = int32_t(lrow);
            }
            whole.push_back(it);
        } else {
            for (size_t k = i; k < j; ++k) {
                sp_lrow.push_back(int32_t(int64_t(tok[k / R].first) * R + int64_t(k % R)));
                sp_prow.push_back(int32_t(int64_t(tok[k / R].second) * R + int64_t(k % R)));
            }
        }
        i = j;
    }
    for (size_t k = 0; k < sp_prow.size(); k += kBlockRows) {
        Item it;
        clear_item(it);
        it.kind = 1;
        it.block = -1;
        const size_t n = std::min<size_t>(kBlockRows, sp_prow.size() - k);
        it.count = int32_t(n);
        for (size_t q = 0; q < n; ++q) {
            it.prow[q] = sp_prow[k + q];
            it.lrow[q] = sp_lrow[k + q];
        }
        spill.push_back(it);
    }
    const int64_t items = int64_t(whole.size() + spill.size());
    if (size_t(items) * sizeof(Item) > capacity) return RMSNORM_ERR_CAPACITY;
    if (items > 0 && !plan) return RMSNORM_ERR_NULL;
    Item *out = static_cast<Item *>(plan);
    if (!whole.empty()) std::memcpy(out, whole.data(), whole.size() * sizeof(Item));
    if (!spill.empty()) std::memcpy(out + whole.size(), spill.data(), spill.size() * sizeof(Item));
    *plan_items = items;
    if (whole_blocks) *whole_blocks = int64_t(whole.size());
    if (spill_rows) *spill_rows = int64_t(sp_prow.size());
    return RMSNORM_OK;
}
