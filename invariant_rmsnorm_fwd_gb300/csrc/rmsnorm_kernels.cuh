// Kernels of the batch-invariant RMSNorm library (sm_103a).
//
// Two kernel families share the numeric helpers of rbi_device.cuh:
//
//  * split_kernel (hidden > 256): a warp-specialised pipeline per row team
//    of K CTAs (a thread-block cluster when K > 1).  A producer warp stages
//    rows into shared memory with 1-D bulk copies (cp.async.bulk, mbarrier
//    transaction counts), stats warps publish each row's rstd and mean, and
//    column warps write y or dx and reduce the dweight leaves.
//
//  * small_row_kernel (hidden <= 256): a team is P = next_pow2(hidden/8)
//    lanes of one warp (8 columns per lane), so a warp works on 32/P rows at
//    once; rows reach each lane's 16-byte pieces through a per-warp
//    shared-memory ring filled by cp.async ahead of use; each team owns
//    consecutive slots of a unit, so a lane's leaves are reduced in the lane,
//    and the team subtrees meet once per unit.
//
// Work units are either plan items (64 row slots: a whole logical block in
// logical order, or rows of blocks cut by a call boundary) or, without a
// plan, groups of consecutive physical rows whose tok_id says whether a row
// is active.  Which CTA processes which unit never changes a value: every
// output depends only on its row (y, dx, the leaf) or on the fixed trees.
#pragma once
#include "rbi_device.cuh"
#include "umma.cuh"

namespace rbi {

// kAdd*: the residual-add variants.  kAddFwd streams x and the residual r,
// writes h = bf16(x + r) and y = RMSNorm(h); kAddDx / kAddDxDw stream the saved
// h, dy and the gradient dres arriving at h along the residual path, and
// write dh = bf16(grad_scale * dx + dres).
enum Mode : int { kFwd = 0, kDx = 1, kDxDw = 2, kDw = 3, kAddFwd = 4, kAddDx = 5, kAddDxDw = 6 };

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

struct KParams {
    const uint16_t *x;
    const uint16_t *dy;
    const uint16_t *w;
    const uint16_t *res;             // kAddFwd: residual input r; kAddDx, kAddDxDw: dres
    uint16_t *out;                   // y (forward modes) or dx (kDx, kDxDw, kAdd*); may be null in kDxDw
    uint16_t *out2;                  // kAddFwd: h = bf16(x + r)
    float *rstd_out;                 // forward modes, optional
    float grad_scale;                // backward: dx is scaled by it (1 = no scaling)
    const int32_t *tok_id;
    int64_t n_rows;                  // physical rows of the call = n_tokens * rpt
    int64_t token_stride;            // elements
    int32_t rpt;                     // rows per token
    int32_t rpt_shift;               // log2(rpt) if rpt is a power of two, else -1
    int32_t hidden;
    float eps;
    int32_t use_plan;                // 1: units are plan items
    const PlanItem *items;
    int64_t n_units;                 // plan items, or batches / 64-row groups without a plan
    WsView ws;
};

__device__ __forceinline__ int64_t row_offset(const KParams &p, int64_t prow) {
    if (p.rpt == 1) return prow * p.token_stride;
    const uint32_t r = uint32_t(prow);                  // rows of a call are < 2^31
    const uint32_t t = p.rpt_shift >= 0 ? (r >> p.rpt_shift) : r / uint32_t(p.rpt);
    return int64_t(t) * p.token_stride + int64_t(r - t * uint32_t(p.rpt)) * int64_t(p.hidden);
}

template <int MODE>
struct ModeTraits {
    static constexpr bool kFwdLike = MODE == kFwd || MODE == kAddFwd;
    static constexpr bool kNeedDy = !kFwdLike;
    static constexpr bool kNeedGx = MODE == kDx || MODE == kDxDw || MODE == kAddDx || MODE == kAddDxDw;
    static constexpr bool kLeaves = MODE == kDxDw || MODE == kDw || MODE == kAddDxDw;
    static constexpr bool kRes = MODE == kAddFwd || MODE == kAddDx || MODE == kAddDxDw;   // streams p.res
    static constexpr bool kWritesOut = MODE != kDw;
    static constexpr int kTensors = 1 + (kNeedDy ? 1 : 0) + (kRes ? 1 : 0);
    static constexpr int kResSlot = kNeedDy ? 2 : 1;            // stage slot of p.res
};

// Book-keeping of contributions (one thread per team).  A block's four state
// bytes say how it arrived: 2 2 2 2 = one whole-block partial (slot 0),
// 1 1 1 1 = four quarter partials (slots 0..3), 0 0 0 0 = its rows were
// spilled.  Any contribution that meets an earlier one is a double count.
constexpr uint32_t kStateWhole = 0x02020202u;
constexpr uint8_t kStateQuarter = 1;
constexpr uint8_t kStateEighth0 = 4, kStateEighth1 = 8;   // the halves of a quarter split in two

__device__ __forceinline__ bool leaf_flags_clear(const WsView &ws, int64_t r0, int64_t rows) {
    bool clear = true;
    if (rows == 16 && (r0 & 7) == 0) {
        const uint64_t *f = reinterpret_cast<const uint64_t *>(ws.leaf_flag + r0);
        clear = f[0] == 0 && f[1] == 0;
    } else {
        for (int64_t i = 0; i < rows; ++i) clear &= ws.leaf_flag[r0 + i] == 0;
    }
    return clear;
}

__device__ __forceinline__ void mark_whole_block(const WsView &ws, int64_t b) {
    uint32_t *st = reinterpret_cast<uint32_t *>(ws.block_state) + b;
    const int64_t rows = min64(kBlockRows, ws.n_rows - b * kBlockRows);
    bool dup = *st != 0;
    for (int64_t r0 = 0; r0 < rows; r0 += 16) dup |= !leaf_flags_clear(ws, b * kBlockRows + r0, min64(16, rows - r0));
    if (dup) set_status(ws.hdr, kStDouble);
    *st = kStateWhole;
}

__device__ __forceinline__ void mark_quarter(const WsView &ws, int64_t b, int q) {
    uint8_t *st = ws.block_state + b * 4;
    const int64_t r0 = b * kBlockRows + q * 16;
    const int64_t rows = max64(0, min64(16, ws.n_rows - r0));
    bool dup = st[q] != 0;
    for (int i = 0; i < 4; ++i) dup |= st[i] == 2;
    if (rows > 0) dup |= !leaf_flags_clear(ws, r0, rows);
    if (dup) set_status(ws.hdr, kStDouble);
    // a word-wide OR: the two halves of another quarter of this block may be
    // marked by other CTAs at the same time
    atomicOr(reinterpret_cast<unsigned int *>(st), unsigned(kStateQuarter) << (8 * q));
}

// Half `half` (rows 8*half .. 8*half+7) of quarter q of block b arrived as an
// eighth partial.
__device__ __forceinline__ void mark_eighth(const WsView &ws, int64_t b, int q, int half) {
    uint8_t *st = ws.block_state + b * 4;
    const int64_t r0 = b * kBlockRows + q * 16 + half * 8;
    const int64_t rows = max64(0, min64(8, ws.n_rows - r0));
    const uint8_t bit = half ? kStateEighth1 : kStateEighth0;
    bool dup = (st[q] & (bit | kStateQuarter)) != 0;
    for (int i = 0; i < 4; ++i) dup |= st[i] == 2;
    if (rows > 0) dup |= !leaf_flags_clear(ws, r0, rows);
    if (dup) set_status(ws.hdr, kStDouble);
    atomicOr(reinterpret_cast<unsigned int *>(st), unsigned(bit) << (8 * q));
}

// A spilled row meets an earlier contribution if it was spilled before or if
// its quarter arrived as a partial (a whole block sets all four quarter bytes).
__device__ __forceinline__ void mark_spilled_row(const WsView &ws, int64_t lrow) {
    const uint8_t st = ws.block_state[(lrow / kBlockRows) * 4 + (lrow % kBlockRows) / 16];
    if (ws.leaf_flag[lrow] != 0 || st != 0) set_status(ws.hdr, kStDouble);
    ws.leaf_flag[lrow] = 1;
}

// =====================================================================
// Per-stage row metadata
// =====================================================================

struct StageMeta {
    int64_t off;                     // element offset of this CTA's slice of the row, -1 = empty slot
    int32_t lrow;                    // logical row (plan modes)
    int32_t prow;                    // physical row
};

template <int R>
struct SlotBatch {                   // metadata of one batch, held by the producer thread
    int32_t prow[R];
    int32_t lrow[R];
    int32_t kind, block;             // plan item header (split kernel)
};

constexpr int kMaxBatch = 8;                     // rows per pipeline stage <= 8

// =====================================================================
// Hidden sizes above 256: warp-specialised pipeline, one CTA or a K-CTA cluster per row
// =====================================================================
//
// A row team is K CTAs (a thread-block cluster when K > 1); CTA q owns the
// columns [q*H/K, (q+1)*H/K).  In each CTA:
//   warps [0, NC): column warps; thread t owns columns 8t..8t+7 of the slice;
//   warps [NC, NC+NS): stats warps; warp i handles the stages s with s % NS == i;
//   warp NC+NS: producer; lane 0 issues the bulk copies of the CTA's slice.
// Per stage s (R rows of x, dy): full[s] completes when the copies land,
// stats[s] when the stats warp has published rstd and mean(g*xhat) of its
// rows, empty[s] when every column warp is done with it.  With K > 1 the
// stats warps exchange their slice partials through distributed shared
// memory: each sends its partials to every CTA of the cluster with st.async,
// counted in bytes on that CTA's exchange barrier of the stage, then waits
// for all K slices on its own.
// No CTA-wide barrier is used in the streaming loop (the shapes that hold
// tensor memory meet once more at the end, before it is freed).  Rows of the
// dweight modes are processed in 16-row units (a quarter of a logical block):
// the column warps reduce the unit's 16 leaves with the 64-leaf tree's lower
// four levels and store the quarter partial; dweight_finalize adds the four
// quarters.
//
// Row sums (this family's canonical tree, which depends on H only): in each
// slice, lane l folds vectors l, l+32, l+64, ... in order, columns
// interleaved as two FMA chains (columns 0,2,4,6 and 1,3,5,7 of each vector,
// one chain across all of the lane's vectors), the chains are added, and the
// 32 lane sums are added by a complete tree pairing lanes 16 apart first, then
// 8, 4, 2, 1.  The K slice sums are then added in order: p0 + p1 for K = 2,
// (p0 + p1) + (p2 + p3) for K = 4.

constexpr int kSplitMaxStages = 12;
constexpr int kSplitUnitRows = 16;
constexpr int kSplitMaxK = 4;

struct SplitStats {
    float rstd;
    float mg;
};

constexpr int kSplitFlagOff = 480;                                   // after 5 x 12 barriers (480 B)
constexpr int kSplitTmemOff = 484;                                   // tensor-memory base (column warps)
constexpr int kSplitItemOff = 496;                                   // [kSplitMaxStages] int2 item headers
constexpr int kSplitMetaOff = 608;
constexpr int kSplitStatsOff = kSplitMetaOff + kSplitMaxStages * kMaxBatch * 16;
constexpr int kSplitXbufOff = kSplitStatsOff + kSplitMaxStages * kMaxBatch * 8;   // [S][2][K][R] float2
constexpr int kSplitWOff = kSplitXbufOff + kSplitMaxStages * 2 * kSplitMaxK * kMaxBatch * 8;
__host__ __device__ constexpr int split_stage_off(int slice_cols) {
    return ((kSplitWOff + slice_cols * 4) + 127) / 128 * 128;
}

template <int MODE, int R, int MAXT, int NS, int K>
__global__ void __launch_bounds__(MAXT, 1) split_kernel(const KParams p, const int S, const int NC) {
    using T = ModeTraits<MODE>;
    constexpr int kLogR = (R == 1) ? 0 : (R == 2) ? 1 : (R == 4) ? 2 : 3;
    constexpr int kUnitBatches = kSplitUnitRows / R;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *stats_bar = full + kSplitMaxStages;
    uint64_t *empty = stats_bar + kSplitMaxStages;
    uint64_t *xchg = empty + kSplitMaxStages;              // [S][2]: one per parity of a stage's use
    volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(smem + kSplitFlagOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kSplitTmemOff);
    int2 *item_hdr = reinterpret_cast<int2 *>(smem + kSplitItemOff);          // [S] (kind, block)
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + kSplitMetaOff);   // [S][R]
    SplitStats *stats = reinterpret_cast<SplitStats *>(smem + kSplitStatsOff);
    float2 *xbuf = reinterpret_cast<float2 *>(smem + kSplitXbufOff);          // [S][2][K][R]
    float *wsm = reinterpret_cast<float *>(smem + kSplitWOff);
    const int H = p.hidden;
    const int HS = H / K;                                 // columns of this CTA's slice
    const int VS = HS >> 3;                               // vectors of the slice
    uint8_t *stages = smem + split_stage_off(HS);
    const uint32_t row_bytes = uint32_t(HS) * 2u;
    auto stage_ptr = [&](int s, int t, int r) -> uint8_t * {
        return stages + ((int64_t(s) * T::kTensors + t) * R + r) * row_bytes;
    };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = (K > 1) ? cluster_rank() : 0u;
    const int64_t col0 = int64_t(rank) * HS;
    const float Hf = float(H);
    const float inv_h = row_inv_h(H);
    const bool item_units = p.use_plan && T::kLeaves;
    const int64_t per_unit = item_units ? kUnitBatches : 1;
    const int64_t cluster_id = blockIdx.x / K;
    const int64_t n_clusters = gridDim.x / K;
    // Leaf modes: quarter units round-robin over the teams.  When the last
    // round would leave at least half the teams idle (0 < rem <= teams / 2),
    // its quarters are split into two 8-row eighths instead, one per team, so
    // that every team ends after (full + 1/2) quarters.
    const int64_t q_full = p.n_units / n_clusters, q_rem = p.n_units % n_clusters;
    const bool eighths = item_units && q_rem > 0 && 2 * q_rem <= n_clusters;
    const int64_t my_units = eighths ? q_full
                             : (p.n_units > cluster_id ? (p.n_units - cluster_id + n_clusters - 1) / n_clusters : 0);
    const int64_t my_eighths = (eighths && cluster_id < 2 * q_rem) ? 1 : 0;
    const int n_batches = int(my_units * per_unit + my_eighths * (kUnitBatches / 2));   // < 2^31

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&stats_bar[s], 1);
            mbar_init(&empty[s], NC);
            mbar_init(&xchg[2 * s], 1);
            mbar_init(&xchg[2 * s + 1], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // batch k of this team -> (plan item, slot base) or physical batch index
    auto batch_slots = [&](int k, int64_t &item, int &slot0) {
        if (item_units && k >= my_units * kUnitBatches) {  // this team's eighth (cluster_id-th)
            const int64_t qg = q_full * n_clusters + (cluster_id >> 1);
            item = qg >> 2;
            slot0 = int(qg & 3) * kSplitUnitRows + int(cluster_id & 1) * (kSplitUnitRows / 2) +
                    int(k - my_units * kUnitBatches) * R;
        } else if (item_units) {
            const int64_t u = cluster_id + (k / kUnitBatches) * n_clusters;   // quarter unit
            item = u >> 2;
            slot0 = int(u & 3) * kSplitUnitRows + int(k % kUnitBatches) * R;
        } else {
            const int64_t gb = cluster_id + int64_t(k) * n_clusters;
            if (p.use_plan) {
                item = gb / (kBlockRows / R);
                slot0 = int(gb % (kBlockRows / R)) * R;
            } else {
                item = gb;
                slot0 = 0;
            }
        }
    };

    // The producer's first slot metadata is fetched before the CTA (cluster)
    // barrier, so its latency overlaps the weight fill and the barrier.
    constexpr int kPrefetch = 3;
    SlotBatch<R> ring[kPrefetch];
    auto load = [&](int k, SlotBatch<R> &mb) {
        if (k >= n_batches) return;
        int64_t item;
        int slot0;
        batch_slots(k, item, slot0);
        mb.kind = 0;
        mb.block = -1;
        if (item_units) {
            mb.kind = staged_kind(p.items[item]);
            mb.block = p.items[item].block;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            int32_t pr = -1, lr = -1;
            if (p.use_plan) {
                const PlanItem *it = p.items + item;
                pr = it->prow[slot0 + r];
                lr = it->lrow[slot0 + r];
            } else {
                const int64_t row = item * R + r;
                if (row < p.n_rows) pr = p.tok_id[row / p.rpt] >= 0 ? int32_t(row) : -1;
            }
            mb.prow[r] = pr;
            mb.lrow[r] = lr;
        }
    };
    if (warp == NC + NS && lane == 0) {
#pragma unroll
        for (int i = 0; i < kPrefetch; ++i) load(i, ring[i]);
    }
    // Under the 80-register budget (more than 640 threads) the leaf modes of
    // 2-CTA clusters and of the residual chain park level 3 of a column
    // thread's unit tree (the partial of a quarter's first 8 rows, pending while
    // the second half runs) in tensor memory, which this kernel does not
    // otherwise use; without it they spill.  Column warp w holds it in
    // tensor-memory lanes 32 (w % 4) .. +31, columns 8 (w / 4) .. +7.  Warp 0
    // allocates and, after the closing barrier, frees it.  (The single-CTA
    // fused backward fits 80 registers without it, and is 0.9% faster so on
    // hidden 5120 in 256 calls of 4096 token slots: 2.342 against 2.363 ms per
    // step.)
    constexpr bool kStash = T::kLeaves && MAXT > 640 && kLogR < 3 && (K > 1 || T::kRes);
    constexpr uint32_t kStashCols = 64;                  // 8 (ceil(NC / 4)) <= 64 for NC <= 32
    if (kStash && warp == 0) {
        umma::tmem_alloc(tmem_slot, kStashCols);
        umma::tmem_relinquish();
        umma::fence_before();
    }
    if (K > 1) cluster_barrier(); else __syncthreads();
    // The weights in shared memory are read by the stats warps only: they fill
    // them after the barrier, so the producer's first copies are not held up by
    // these loads.
    if (T::kNeedGx && warp >= NC && warp < NC + NS) {
        // 16-byte loads (8 weights each), so that a CTA's start does not wait
        // for a chain of 2-byte loads
        for (int i = tid - NC * 32; i < VS; i += NS * 32) {
            f2_t wf[4];
            f2_unpack8(*reinterpret_cast<const uint4 *>(p.w + col0 + int64_t(i) * 8), wf);
            uint4 *dst = reinterpret_cast<uint4 *>(wsm + i * 8);
            dst[0] = make_uint4(uint32_t(wf[0]), uint32_t(wf[0] >> 32), uint32_t(wf[1]), uint32_t(wf[1] >> 32));
            dst[1] = make_uint4(uint32_t(wf[2]), uint32_t(wf[2] >> 32), uint32_t(wf[3]), uint32_t(wf[3] >> 32));
        }
        asm volatile("bar.sync 1, %0;" ::"r"(NS * 32) : "memory");
    }

    if (warp == NC + NS) {
        // ------------------------------------------------ producer
        // The slot metadata of batch k comes from global memory (plan or
        // tok_id); it is loaded kPrefetch batches ahead so that issuing the
        // copies never waits on it.
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;                             // parity of the current use of stage s
            for (int k = 0; k < n_batches; ++k) {
                const SlotBatch<R> cur = ring[0];
#pragma unroll
                for (int i = 0; i + 1 < kPrefetch; ++i) ring[i] = ring[i + 1];
                load(k + kPrefetch, ring[kPrefetch - 1]);
                if (k >= S && !mbar_wait_bounded(&empty[s], ph ^ 1u)) {
                    *abort_flag = 1;
                    if (T::kLeaves) set_status(p.ws.hdr, kStTimeout);
                }
                if (*abort_flag) {
                    // let copies already issued land (bounded) before leaving
                    int ss = s;
                    uint32_t pp = ph;
                    for (int kk = k - 1; kk >= 0 && kk >= k - S; --kk) {
                        if (--ss < 0) {
                            ss = S - 1;
                            pp ^= 1u;
                        }
                        mbar_wait_bounded(&full[ss], pp);
                    }
                    break;
                }
                StageMeta *m = meta + s * R;
                item_hdr[s] = make_int2(cur.kind, cur.block);
                int64_t offs[R];
                uint32_t n_act = 0;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int32_t pr = cur.prow[r], lr = cur.lrow[r];
                    bool act = pr >= 0;
                    if (act && (pr >= p.n_rows || (T::kLeaves && (lr < 0 || lr >= p.ws.n_rows)))) {
                        if (T::kLeaves && rank == 0) set_status(p.ws.hdr, kStPlan);
                        act = false;
                    }
                    offs[r] = act ? row_offset(p, pr) : -1;
                    m[r].off = offs[r];
                    m[r].lrow = lr;
                    m[r].prow = pr;
                    n_act += act ? 1u : 0u;
                }
                mbar_arrive_expect_tx(&full[s], n_act * row_bytes * T::kTensors);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (offs[r] < 0) continue;
                    bulk_copy_g2s(stage_ptr(s, 0, r), p.x + offs[r] + col0, row_bytes, &full[s]);
                    if (T::kNeedDy) bulk_copy_g2s(stage_ptr(s, 1, r), p.dy + offs[r] + col0, row_bytes, &full[s]);
                    if (T::kRes)
                        bulk_copy_g2s(stage_ptr(s, T::kResSlot, r), p.res + offs[r] + col0, row_bytes, &full[s]);
                }
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp >= NC) {
        // ------------------------------------------------ stats warps
        const int si = warp - NC;
        int s = 0;
        uint32_t ph = 0;
        for (int k = 0; k < n_batches; ++k, ph ^= (s == S - 1) ? 1u : 0u, s = (s == S - 1) ? 0 : s + 1) {
            if (s % NS != si) continue;
            if (*abort_flag) break;
            if (!mbar_wait_bounded(&full[s], ph)) {
                *abort_flag = 1;
                if (T::kLeaves) set_status(p.ws.hdr, kStTimeout);
                break;
            }
            const StageMeta *m = meta + s * R;
            // The R rows of the stage are folded in one pass over the slice: each
            // row keeps its own two chains (the canonical order), so the rows'
            // chains are independent and run side by side, and a weight vector
            // is read once for all of them.  A row the stage does not hold is
            // folded too (its buffer holds stale bytes) and its sums are dropped.
            f2_t a2[R], b2[R];
#pragma unroll
            for (int r = 0; r < R; ++r) a2[r] = b2[r] = 0ull;   // +0.0 in both lanes
#pragma unroll 2
            for (int v = lane; v < VS; v += 32) {
                f2_t wf[4];
                if (T::kNeedGx) {
                    const float4 w0 = *reinterpret_cast<const float4 *>(wsm + v * 8);
                    const float4 w1 = *reinterpret_cast<const float4 *>(wsm + v * 8 + 4);
                    wf[0] = f2_make(w0.x, w0.y);
                    wf[1] = f2_make(w0.z, w0.w);
                    wf[2] = f2_make(w1.x, w1.y);
                    wf[3] = f2_make(w1.z, w1.w);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    f2_t xf[4];
                    f2_unpack8(ld_shared_v4(stage_ptr(s, 0, r) + v * 16), xf);
                    if (MODE == kAddFwd) {                  // the row is h = bf16(x + r)
                        f2_t rf[4];
                        f2_unpack8(ld_shared_v4(stage_ptr(s, T::kResSlot, r) + v * 16), rf);
#pragma unroll
                        for (int i = 0; i < 4; ++i) xf[i] = f2_add(xf[i], rf[i]);
                        f2_unpack8(f2_pack8(xf), xf);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) a2[r] = f2_fma(xf[i], xf[i], a2[r]);
                    if (T::kNeedGx) {
                        f2_t df[4];
                        f2_unpack8(ld_shared_v4(stage_ptr(s, 1, r) + v * 16), df);
#pragma unroll
                        for (int i = 0; i < 4; ++i) b2[r] = f2_fma(f2_mul(df[i], wf[i]), xf[i], b2[r]);
                    }
                }
            }
            float vals[2 * R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const bool held = m[r].off >= 0;
                vals[r] = held ? __fadd_rn(f2_lo(a2[r]), f2_hi(a2[r])) : 0.f;
                vals[R + r] = held ? __fadd_rn(f2_lo(b2[r]), f2_hi(b2[r])) : 0.f;
            }
            // complete tree over the 32 lanes, pairing 16 apart first
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1)
#pragma unroll
                for (int j = 0; j < (T::kNeedGx ? 2 * R : R); ++j)
                    vals[j] = __fadd_rn(vals[j], __shfl_xor_sync(kFull, vals[j], d));
            if (K > 1) {
                // send this slice's partials to every CTA of the cluster
                // Each lane c < K sends this slice's R partials to CTA c with
                // st.async, whose completion counts 8 bytes on CTA c's barrier of
                // this parity of the stage; the local arrival registers the K * R
                // * 8 bytes expected (a peer's bytes may land first).  A barrier
                // serves every second use of the stage, so its own phase parity is
                // that of k / (2S), and a peer can never be a whole phase ahead on
                // it.  The wait acquires at cluster scope (the peers' stores).
                float2 *xb = xbuf + ((s * 2 + int(ph)) * K) * R;   // [K][R] for this use of stage s
                uint64_t *xb_bar = &xchg[2 * s + int(ph)];
                const uint32_t bp = uint32_t(k / S / 2) & 1u;
                if (lane == 0) mbar_arrive_expect_tx(xb_bar, uint32_t(K * R * 8));
                if (lane < K) {
                    const uint32_t bar_c = map_to_rank(smem_addr(xb_bar), uint32_t(lane));
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        st_async_f32x2(map_to_rank(smem_addr(xb + rank * R + r), uint32_t(lane)), vals[r], vals[R + r], bar_c);
                }
                if (!mbar_wait_bounded_cluster(xb_bar, bp)) {
                    *abort_flag = 1;
                    if (T::kLeaves) set_status(p.ws.hdr, kStTimeout);
                    break;
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float2 q[kSplitMaxK];
#pragma unroll
                    for (int c = 0; c < K; ++c) q[c] = xb[c * R + r];
                    if (K == 2) {
                        vals[r] = __fadd_rn(q[0].x, q[1].x);
                        vals[R + r] = __fadd_rn(q[0].y, q[1].y);
                    } else {
                        vals[r] = __fadd_rn(__fadd_rn(q[0].x, q[1].x), __fadd_rn(q[2].x, q[3].x));
                        vals[R + r] = __fadd_rn(__fadd_rn(q[0].y, q[1].y), __fadd_rn(q[2].y, q[3].y));
                    }
                }
            }
            if (lane < R) {
                float ss = vals[0], gx = vals[R];
#pragma unroll
                for (int r = 1; r < R; ++r)
                    if (lane == r) {
                        ss = vals[r];
                        gx = vals[R + r];
                    }
                const float rstd = row_rstd(ss, Hf, inv_h, p.eps);
                SplitStats st;
                st.rstd = rstd;
                st.mg = T::kNeedGx ? row_mean_gxhat(gx, rstd, Hf, inv_h) : 0.f;
                stats[s * R + lane] = st;
                if (T::kFwdLike && rank == 0 && p.rstd_out != nullptr && m[lane].off >= 0)
                    p.rstd_out[m[lane].prow] = rstd;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&stats_bar[s]);
        }
    } else {
        // ------------------------------------------------ column warps
        const int t = tid;                                   // vector owned: slice columns 8t..8t+7
        const bool has_vec = t < VS;
        const int64_t my_col = col0 + int64_t(t) * 8;
        // In the leaf modes under the 80-register budget (more than 640
        // threads) the weights stay packed (4 registers instead of 8) and are
        // unpacked for every row.
        constexpr bool kPackW = T::kLeaves && MAXT > 640;
        uint4 wpk = make_uint4(0, 0, 0, 0);
        f2_t wv[4] = {0ull, 0ull, 0ull, 0ull};
        if (MODE != kDw && has_vec) {
            wpk = *reinterpret_cast<const uint4 *>(p.w + my_col);
            if (!kPackW) f2_unpack8(wpk, wv);
        }
        TreeStackF2<4, kStash ? 3 : 4> tree;   // levels log2(R)..3 (..2 with the stash) of the 16-leaf unit
        uint32_t stash = 0;
        if (kStash) {
            umma::fence_after();
            stash = *tmem_slot + (uint32_t((warp & 3) * 32) << 16) + uint32_t((warp >> 2) * 8);
        }
        // Of the current unit: where its partial goes (a quarter of a block, or
        // an eighth in the last round), whether it is stored, whether its rows
        // are spilled.  Set at the unit's first batch, so nothing else about
        // the item stays live across the unit.
        float *part = p.ws.block_partial;
        uint32_t part_mask = 0;
        bool spill_unit = false;
        int s = 0;
        uint32_t parity = 0;
        uint32_t u = uint32_t(cluster_id);                    // current quarter unit (low bits)
        // Leaf modes walk their 16-row units; the inner loop over the unit's
        // batches (stages of R rows) is unrolled, so `sub`, the batch's place in
        // the unit, is a compile-time constant and the tree positions are static.
        // A team's eighth (8 rows, kInner / 2 batches) comes after its quarters.
        constexpr int kInner = T::kLeaves ? kUnitBatches : 1;
        const int n_outer = T::kLeaves ? int(my_units + my_eighths) : n_batches;
        bool stop = false;
        for (int j = 0; j < n_outer && !stop; ++j, u += uint32_t(n_clusters)) {
          const bool half_unit = T::kLeaves && j >= my_units;
#pragma unroll
          for (int sub = 0; sub < kInner; ++sub) {
            if (half_unit && sub >= kInner / 2) break;
            // with the stash the warp leaves as one (tensor-memory accesses are
            // warp-wide)
            if (kStash ? __any_sync(kFull, *abort_flag != 0) : *abort_flag != 0) {
                stop = true;
                break;
            }
            const bool ready = mbar_wait_bounded(&stats_bar[s], parity) && mbar_wait_bounded(&full[s], parity);
            if (kStash ? !__all_sync(kFull, ready) : !ready) {
                *abort_flag = 1;
                if (T::kLeaves) set_status(p.ws.hdr, kStTimeout);
                stop = true;
                break;
            }
            if (T::kLeaves && sub == 0) {                    // item header, staged by the producer
                const int2 hd = item_hdr[s];
                const int quarter = half_unit ? int((q_full * n_clusters + (cluster_id >> 1)) & 3) : int(u & 3u);
                int kind = hd.x & 0xff;
                const int qmask = hd.x >> 8;
                const int32_t block = hd.y;
                const bool blocked = kind == kItemWhole || kind == kItemQuarters;
                if ((blocked && (block < 0 || block >= p.ws.n_blocks)) || (!blocked && kind != kItemSpill)) {
                    if (t == 0 && rank == 0) set_status(p.ws.hdr, kStPlan);
                    kind = kBadItem;
                }
                // a quarter of a kind-2 item that the call does not hold is skipped
                const bool keep = kind == kItemWhole || (kind == kItemQuarters && ((qmask >> quarter) & 1));
                spill_unit = kind == kItemSpill;
                const int half = int(cluster_id & 1);
                part = ((half_unit && half) ? p.ws.eighth : p.ws.block_partial) +
                       (int64_t(keep ? block : 0) * 4 + quarter) * H + my_col;
                part_mask = (keep && has_vec) ? ~0u : 0u;
                // the finalize reads the marks after this launch, so the unit is
                // marked here rather than after its partial is stored
                if (keep && t == 0 && rank == 0) {
                    if (half_unit) mark_eighth(p.ws, block, quarter, half);
                    else mark_quarter(p.ws, block, quarter);
                }
            }
            const StageMeta *m = meta + s * R;
            TreeStackF2<4, (kLogR > 0 ? kLogR : 1)> mini;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t off = m[r].off;
                const bool act = off >= 0;
                f2_t leaf[4] = {0ull, 0ull, 0ull, 0ull};
                if (act && has_vec) {
                    const SplitStats st = stats[s * R + r];
                    const f2_t r2 = f2_make(st.rstd, st.rstd);
                    f2_t xf[4], xh[4], o[4];
                    if (kPackW) f2_unpack8_v(wpk, wv);
                    f2_unpack8(ld_shared_v4(stage_ptr(s, 0, r) + t * 16), xf);
                    if (MODE == kAddFwd) {                          // h = bf16(x + r), stored, then normed
                        f2_t rf[4];
                        f2_unpack8(ld_shared_v4(stage_ptr(s, T::kResSlot, r) + t * 16), rf);
#pragma unroll
                        for (int i = 0; i < 4; ++i) xf[i] = f2_add(xf[i], rf[i]);
                        const uint4 hb = f2_pack8(xf);
                        st_global_v4(p.out2 + off + my_col, hb);
                        f2_unpack8(hb, xf);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) xh[i] = f2_mul(xf[i], r2);
                    if (T::kFwdLike) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) o[i] = f2_mul(xh[i], wv[i]);
                        st_global_v4(p.out + off + my_col, f2_pack8(o));
                    } else {
                        f2_t df[4];
                        f2_unpack8(ld_shared_v4(stage_ptr(s, 1, r) + t * 16), df);
                        if (T::kNeedGx && p.out != nullptr) {
                            const f2_t nm2 = f2_make(-st.mg, -st.mg);
                            const float rs = __fmul_rn(st.rstd, p.grad_scale);    // == rstd when unscaled
                            const f2_t rs2 = f2_make(rs, rs);
#pragma unroll
                            for (int i = 0; i < 4; ++i) o[i] = f2_mul(rs2, f2_fma(xh[i], nm2, f2_mul(df[i], wv[i])));
                            if (T::kRes) {
                                f2_t rf[4];
                                f2_unpack8(ld_shared_v4(stage_ptr(s, T::kResSlot, r) + t * 16), rf);
#pragma unroll
                                for (int i = 0; i < 4; ++i) o[i] = f2_add(o[i], rf[i]);
                            }
                            st_global_v4(p.out + off + my_col, f2_pack8(o));
                        }
                        if (T::kLeaves) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) leaf[i] = f2_mul(df[i], xh[i]);
                        }
                    }
                }
                if (T::kLeaves) {
                    // the tree runs for every unit (a quarter or eighth partial is
                    // stored only for a kept quarter of a block)
                    if (spill_unit && act && has_vec) st_global_f2x4(p.ws.spill + int64_t(m[r].lrow) * H + my_col, leaf);
                    if (R > 1) mini.template push_static<0>(leaf, r);
                    if (r == R - 1) {
                        tree.template push_static<kLogR>(leaf, sub);
                        if (kStash && !half_unit && sub == kUnitBatches / 2 - 1) {   // the first half's partial
                            uint32_t h[8];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                h[2 * c] = uint32_t(leaf[c]);
                                h[2 * c + 1] = uint32_t(leaf[c] >> 32);
                            }
                            __syncwarp();
                            umma::st_32x32_x8(stash, h);
                            umma::wait_st();
                        }
                        if (kStash && sub == kUnitBatches - 1) {     // first half + second half
                            uint32_t h[8];
                            __syncwarp();
                            umma::ld_32x32_x8(stash, h);
                            umma::wait_ld();
#pragma unroll
                            for (int c = 0; c < 4; ++c) leaf[c] = f2_add((f2_t(h[2 * c + 1]) << 32) | h[2 * c], leaf[c]);
                        }
                        // leaf[] is now the quarter partial, or the eighth partial
                        if (sub == kUnitBatches - 1 || (half_unit && sub == kUnitBatches / 2 - 1))
                            st_global_f2_if(part, leaf, part_mask);
                    }
                }
            }
            if (T::kLeaves && spill_unit && t == 0 && rank == 0) {   // the spilled rows' flags
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (m[r].off >= 0) mark_spilled_row(p.ws, m[r].lrow);
            }
            __syncwarp();
#ifndef RBI_TEST_WITHHOLD_EMPTY
            if (lane == 0) mbar_arrive(&empty[s]);
#endif
            // (A test-only build defines RBI_TEST_WITHHOLD_EMPTY: the column warps
            // never release a stage, so the producer's first wait to reuse one runs
            // out before it issues any copy into it; see the timeout test.)
            if (++s == S) {
                s = 0;
                parity ^= 1u;
            }
          }
        }
    }
    if (kStash) {
        umma::fence_before();
        if (K > 1) cluster_barrier(); else __syncthreads();
        if (warp == 0) {
            __syncwarp();
            umma::fence_after();
            umma::tmem_dealloc(*tmem_slot, kStashCols);
        }
    } else if (K > 1) {
        cluster_barrier();             // peers may still store into our exchange buffers
    }
}

__device__ __forceinline__ f2_t shfl_xor_f2(f2_t v, int k) {
    return (f2_t(__shfl_xor_sync(kFull, uint32_t(v >> 32), k)) << 32) | __shfl_xor_sync(kFull, uint32_t(v), k);
}

// Launch shape of the small-row kernel (overridable for measurements).
#ifndef RBI_SMALL_WARPS
#define RBI_SMALL_WARPS 4                               // warps per CTA
#endif
#ifndef RBI_SMALL_DEPTH
#define RBI_SMALL_DEPTH 2                               // most ring buffers per warp
#endif
#ifndef RBI_SMALL_LEAF_U
#define RBI_SMALL_LEAF_U 4                              // rows per team and group, two-tensor leaf modes
#endif
constexpr int kSmallWarps = RBI_SMALL_WARPS;
constexpr int kSmallTable = 64 * 16 + 16;               // one unit's slot table, then its header
constexpr int kSmallMinBlocks = 65536 / (128 * 32 * kSmallWarps);   // 128 registers per thread

__host__ __device__ constexpr int small_log2(int v) { return v <= 1 ? 0 : 1 + small_log2(v >> 1); }
__host__ __device__ constexpr int small_min(int a, int b) { return a < b ? a : b; }

// Everything the small-row kernel and its launcher derive from (mode, team
// lanes P).  A lane holds one 16-byte vector (8 columns) of a row.  Shared
// memory of one warp: two unit tables, a ring of kDepth group buffers (kU
// warp steps x kT tensors x 32 lane vectors; never more than one unit's
// groups ahead, since there are two tables), and in the leaf modes the
// lane's stack of pending group subtrees (kStackLevels x 32 lanes x 8 FP32).
// Measured on head_dim 128 (teams of 16 lanes, two rows per warp step): four
// rows per team and group with two ring buffers beat two rows with three
// buffers by 19% on the fused backward; 8 columns per lane beat 4 (teams of
// a whole warp, one row per step) by 12% on the step.
template <int MODE, int P>
struct SmallShape {
    using T = ModeTraits<MODE>;
    static constexpr int kStepBytes = 32 * 16;           // one tensor of one warp step
    static constexpr int TPW = 32 / P;                   // row teams per warp
    static constexpr int kTeamRows = kBlockRows / TPW;   // slots of a unit per team
    // rows per team in one group (the warp steps whose row sums share one
    // reduction): fewer for the three-tensor leaf mode (registers)
    static constexpr int U = T::kLeaves ? (T::kTensors >= 3 ? 2 : RBI_SMALL_LEAF_U) : (T::kTensors >= 2 ? 4 : 8);
    static constexpr int kU = small_min(U, kTeamRows);
    static constexpr int kGroups = kTeamRows / kU;
    static constexpr int kLogGroups = small_log2(kGroups);
    static constexpr int kT = T::kTensors;
    static constexpr int kGroupBytes = kU * kT * kStepBytes;
    static constexpr int kDepth = small_min(small_min(RBI_SMALL_DEPTH, 3 * kGroupBytes <= 12288 ? 3 : 2), kGroups + 1);
    static constexpr int kStackLevels = T::kLeaves ? kLogGroups : 0;
    static constexpr int kStackBytes = kStackLevels * 32 * 32;
    static constexpr int kWarpBytes = 2 * kSmallTable + kDepth * kGroupBytes + kStackBytes;
};

// Small hidden sizes.  Lane tl of a team holds columns 8tl .. 8tl+7; team t
// of a warp owns the consecutive slots [t*64/TPW, (t+1)*64/TPW) of each unit
// (64 row slots), TPW = 32/P teams per warp.  Each warp works through its
// units in groups of kU warp steps; the rows of a group are copied into a
// per-warp shared-memory ring with cp.async, D = depth - 1 groups ahead of the
// group being computed, so the bytes in flight are not bounded by registers.
// An empty slot, and the columns past the row of the last lanes of a team,
// are filled with zeros by the copy itself, so every value in the ring is a
// number.  Each lane copies and later reads only its own pieces, so the ring
// needs no barrier; the slot table of a unit (byte offset of the row, bytes
// to copy, logical or physical row) is written once per unit by the warp and
// read by broadcast.  Per group: (1) row sums of the kU steps, (2) rstd and
// mean(g*xhat) once per row, (3) outputs and leaves, stored under predicates.
// A lane's leaves stay in the lane: the group's kU rows form a subtree with
// static positions, the groups of a team a subtree through a stack of pending
// partials in shared memory, and at the end of the unit the TPW team subtrees
// are added across teams (adjacent teams first) into the block partial.
template <int MODE, int P>
__global__ void __launch_bounds__(kSmallWarps * 32, kSmallMinBlocks) small_row_kernel(const KParams p) {
    using Sh = SmallShape<MODE, P>;
    using T = ModeTraits<MODE>;
    constexpr int NF = 4;                                // FP32 pairs of a lane vector
    constexpr int kVB = 16;                              // bytes of a lane vector
    constexpr int kStepBytes = Sh::kStepBytes;
    constexpr int TPW = Sh::TPW;
    constexpr int kLogP = small_log2(P);
    constexpr int kTeamRows = Sh::kTeamRows;
    constexpr int kU = Sh::kU;                           // warp steps per group
    constexpr int kLogU = small_log2(kU);
    constexpr int kGroups = Sh::kGroups;
    constexpr int kLogGroups = Sh::kLogGroups;
    constexpr int kT = Sh::kT;
    constexpr int kGroupBytes = Sh::kGroupBytes;
    constexpr int kDepth = Sh::kDepth;
    constexpr int kAhead = kDepth - 1;                   // groups issued ahead of the one computed
    static_assert(P * TPW == 32 && kGroups * kU == kTeamRows && (1 << kLogGroups) == kGroups, "small shape");
    static_assert(kAhead >= 1 && kAhead <= kGroups, "the issue side stays within the next unit");

    extern __shared__ __align__(16) uint8_t small_smem[];
    const int lane = threadIdx.x & 31;
    uint8_t *wbase = small_smem + (threadIdx.x >> 5) * Sh::kWarpBytes;
    const uint32_t ring_lane = smem_addr(wbase + 2 * kSmallTable) + lane * kVB;   // this lane's piece, slot 0
    // the lane's stack of pending group subtrees (leaf modes): level l at
    // stack_lane + l * 32 * 32
    const uint32_t stack_lane = smem_addr(wbase + 2 * kSmallTable + kDepth * kGroupBytes) + lane * 32;
    const int team = lane >> kLogP, tl = lane & (P - 1);
    const int H = p.hidden;
    const bool has_vec = tl * 8 < H;
    const int col0 = has_vec ? tl * 8 : 0;              // a lane past the row reads nothing, at column 0
    const uint32_t vec_mask = has_vec ? ~0u : 0u;
    const float Hf = float(H);
    const float inv_h = row_inv_h(H);
    const int64_t gwarp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int64_t my_units = p.n_units > gwarp ? (p.n_units - gwarp + nwarps - 1) / nwarps : 0;
    // this lane's columns of row 0 of each tensor; a row adds its byte offset
    const uint8_t *gx = reinterpret_cast<const uint8_t *>(p.x + col0);
    const uint8_t *gdy = reinterpret_cast<const uint8_t *>(T::kNeedDy ? p.dy + col0 : p.x);
    const uint8_t *gres = reinterpret_cast<const uint8_t *>(T::kRes ? p.res + col0 : p.x);
    uint8_t *gout = reinterpret_cast<uint8_t *>(p.out + col0);
    const uint32_t out_mask = (T::kWritesOut && p.out != nullptr) ? vec_mask : 0u;

    f2_t wv[NF];
#pragma unroll
    for (int i = 0; i < NF; ++i) wv[i] = 0ull;
    if (MODE != kDw && has_vec) {
        const uint4 w = *reinterpret_cast<const uint4 *>(p.w + col0);
        vec_unpack(w, wv);
    }

    // unit tables: per slot the byte offset of the row (0 when empty), the
    // bytes a lane copies (kVB, or 0 when empty), and the logical row (leaf
    // modes) or the physical row (forward modes); the item header (kind,
    // block) after the 64 entries
    struct SlotEntry {
        int64_t boff;
        int32_t row;
        uint32_t nb;
    };
    auto table = [&](int64_t ord) { return reinterpret_cast<SlotEntry *>(wbase + int(ord & 1) * kSmallTable); };
    // slot metadata of unit `ord` (lane l: slots 2l, 2l+1) into registers
    auto fetch_unit = [&](int64_t ord, int2 &pr2, int2 &lr2, int2 &hd) {
        pr2 = make_int2(-1, -1);
        lr2 = make_int2(-1, -1);
        hd = make_int2(0, -1);
        if (ord >= my_units) return;
        const int64_t u = gwarp + ord * nwarps;
        if (p.use_plan) {
            const PlanItem *it = p.items + u;
            pr2 = reinterpret_cast<const int2 *>(it->prow)[lane];
            lr2 = reinterpret_cast<const int2 *>(it->lrow)[lane];
            hd = make_int2(it->kind, it->block);
        } else {
            const int64_t r0 = u * kBlockRows + 2 * lane;
            if (r0 < p.n_rows && p.tok_id[r0 / p.rpt] >= 0) pr2.x = int32_t(r0);
            if (r0 + 1 < p.n_rows && p.tok_id[(r0 + 1) / p.rpt] >= 0) pr2.y = int32_t(r0 + 1);
        }
    };
    int2 pr_next, lr_next, hdr_next;
    fetch_unit(0, pr_next, lr_next, hdr_next);

    // the issue side walks the groups in order: unit i_ord, group i_g, ring slot i_slot
    int64_t i_ord = 0;
    int i_g = 0, i_slot = 0;
    auto issue_next = [&]() {
        if (i_ord < my_units) {
            if (i_g == 0) {                              // entering a unit: its table, the next one's metadata
                __syncwarp();                            // readers of the table being replaced are done
                SlotEntry *tb = table(i_ord);
                const int32_t prs[2] = {pr_next.x, pr_next.y}, lrs[2] = {lr_next.x, lr_next.y};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int32_t pr = prs[h], lr = lrs[h];
                    bool act = pr >= 0;
                    if (act && (pr >= p.n_rows || (T::kLeaves && (lr < 0 || lr >= p.ws.n_rows)))) {
                        if (T::kLeaves) set_status(p.ws.hdr, kStPlan);
                        act = false;
                    }
                    SlotEntry e;
                    e.boff = act ? row_offset(p, pr) * 2 : 0;
                    e.row = T::kLeaves ? lr : pr;
                    e.nb = act ? uint32_t(kVB) : 0u;
                    tb[2 * lane + h] = e;
                }
                if (lane == 0) *reinterpret_cast<int2 *>(reinterpret_cast<uint8_t *>(tb) + 64 * 16) = hdr_next;
                fetch_unit(i_ord + 1, pr_next, lr_next, hdr_next);
                __syncwarp();
            }
            const SlotEntry *tb = table(i_ord) + team * kTeamRows + i_g * kU;
            const uint32_t dst = ring_lane + i_slot * kGroupBytes;
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const SlotEntry e = tb[q];
                const uint32_t nb = e.nb & vec_mask;
                cp_async_zfill(dst + (q * kT + 0) * kStepBytes, gx + e.boff, nb);
                if (T::kNeedDy) cp_async_zfill(dst + (q * kT + 1) * kStepBytes, gdy + e.boff, nb);
                if (T::kRes) cp_async_zfill(dst + (q * kT + T::kResSlot) * kStepBytes, gres + e.boff, nb);
            }
            if (++i_g == kGroups) {
                i_g = 0;
                ++i_ord;
            }
            if (++i_slot == kDepth) i_slot = 0;
        }
        cp_async_commit();
    };

#pragma unroll
    for (int a = 0; a < kAhead; ++a) issue_next();
    int c_slot = 0;
#pragma unroll 1
    for (int64_t ord = 0; ord < my_units; ++ord) {
        // the unit's header is kept with its table: the issue side may have
        // moved on to the next unit already
        int32_t kind, block;
        {
            const int2 hd = *reinterpret_cast<const int2 *>(reinterpret_cast<const uint8_t *>(table(ord)) + 64 * 16);
            // quarter items (kind 2) are spilled row by row here: a unit of this
            // kernel is a whole block, and the finalize rebuilds those quarters
            kind = hd.x & 0xff;
            block = hd.y;
            if (kind == kItemQuarters) kind = kItemSpill;
            if (T::kLeaves && ((kind == kItemWhole && (block < 0 || block >= p.ws.n_blocks)) ||
                               (kind != kItemWhole && kind != kItemSpill))) {
                if (lane == 0) set_status(p.ws.hdr, kStPlan);
                kind = kBadItem;                           // malformed item: contributes nothing
            }
        }
        // whole: the leaves enter the tree; spill_mask: they are spilled (the
        // stores are predicated on it, so no row branches on the kind)
        const bool whole = T::kLeaves && kind == kItemWhole;
        const uint32_t spill_mask = (T::kLeaves && kind == kItemSpill) ? vec_mask : 0u;
        f2_t node[NF];                                     // the last group's subtree, then the team's
#pragma unroll
        for (int i = 0; i < NF; ++i) node[i] = 0ull;
#pragma unroll 1
        for (int g = 0; g < kGroups; ++g) {
            __syncwarp();                                  // every lane is done with the buffer reused next
            issue_next();
            cp_async_wait<kAhead>();                       // this lane's copies of this group have landed
            const SlotEntry *tb = table(ord) + team * kTeamRows + g * kU;
            const uint32_t src = ring_lane + c_slot * kGroupBytes;
            if (++c_slot == kDepth) c_slot = 0;

            uint4 xv[kU], dv[kU];
            constexpr bool kDres = T::kRes && T::kNeedDy;           // dres streamed (kAddDx*)
            constexpr int kRv = kDres ? kU : 1;                     // its registers
            uint4 rv[kRv];
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                ld_shared_vec(src + (q * kT + 0) * kStepBytes, xv[q]);
                if (T::kNeedDy || MODE == kAddFwd) ld_shared_vec(src + (q * kT + 1) * kStepBytes, dv[q]);
                else vec_zero(dv[q]);
                if (kDres) ld_shared_vec(src + (q * kT + T::kResSlot) * kStepBytes, rv[q % kRv]);
            }
            // phase 1: the lane partials of every row sum of the group (two FMA
            // chains per lane vector, even and odd columns, then added); values
            // 0..kU-1 are the sums of squares of the kU steps, kU..2kU-1 the
            // sums of g*x
            constexpr int kNV = kU * (T::kNeedGx ? 2 : 1);
            constexpr int kLogNV = small_log2(kNV);
            constexpr int kHalvings = kLogNV < kLogP ? kLogNV : kLogP;
            constexpr int kCnt = kNV >> kHalvings;       // values a lane holds after the reduction
            float vals[kNV];
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                f2_t xf[NF], df[NF];
                vec_unpack(xv[q], xf);
                vec_unpack(dv[q], df);
                if (MODE == kAddFwd) {                              // the row is h = bf16(x + r)
#pragma unroll
                    for (int i = 0; i < NF; ++i) xf[i] = f2_add(xf[i], df[i]);
                    vec_pack(xf, xv[q]);                             // h replaces x from here on
                    vec_unpack(xv[q], xf);
                }
                f2_t a2 = f2_mul(xf[0], xf[0]);
#pragma unroll
                for (int i = 1; i < NF; ++i) a2 = f2_fma(xf[i], xf[i], a2);
                vals[q] = __fadd_rn(f2_lo(a2), f2_hi(a2));
                if (T::kNeedGx) {
                    f2_t b2 = f2_mul(f2_mul(df[0], wv[0]), xf[0]);
#pragma unroll
                    for (int i = 1; i < NF; ++i) b2 = f2_fma(f2_mul(df[i], wv[i]), xf[i], b2);
                    vals[kU + q] = __fadd_rn(f2_lo(b2), f2_hi(b2));
                }
            }
            // the team tree over the P lanes (lanes 1 apart first, then 2, 4, ...)
            // as a transposing reduction: at distance d a lane keeps half of its
            // values and adds its partner's copy of them, so every value is still
            // the sum over the same lane pairs (addition is commutative) but the
            // kNV trees cost kNV - 1 exchanges instead of kNV * log2(P)
#pragma unroll
            for (int lv = 0; lv < kLogP; ++lv) {
                const int d = 1 << lv;
                if (lv < kHalvings) {
                    constexpr int kMaxHalf = kNV / 2;
                    const int half = kNV >> (lv + 1);
                    const bool upper = (lane & d) != 0;
#pragma unroll
                    for (int jj = 0; jj < kMaxHalf; ++jj) {
                        if (jj < half) {
                            const float send = upper ? vals[jj] : vals[jj + half];
                            const float keep = upper ? vals[jj + half] : vals[jj];
                            vals[jj] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, d));
                        }
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < kCnt; ++jj) vals[jj] = __fadd_rn(vals[jj], __shfl_xor_sync(kFull, vals[jj], d));
                }
            }
            // value index held in vals[jj]: (lane bits of the halvings, highest
            // weight at distance 1) + jj
            auto holder = [&](int idx) {                   // team lane holding value idx
                int l = 0;
#pragma unroll
                for (int lv = 0; lv < kHalvings; ++lv) l |= ((idx >> (kLogNV - 1 - lv)) & 1) << lv;
                return team * P + l;
            };
            // phase 2: rstd and mean(g*xhat), once per row: each lane evaluates the
            // values it holds; a lane holding g*x of step q takes rstd of step q
            // from the lane (or register) holding its sum of squares
            float rloc[kCnt], mloc[kCnt];
#pragma unroll
            for (int jj = 0; jj < kCnt; ++jj) rloc[jj] = row_rstd(vals[jj], Hf, inv_h, p.eps);
            if (T::kNeedGx) {
#pragma unroll
                for (int jj = 0; jj < kCnt; ++jj) {
                    float rs_q;
                    if (kHalvings >= 1) rs_q = __shfl_xor_sync(kFull, rloc[jj], 1);   // distance 1 splits ss / gx
                    else rs_q = rloc[jj % (kCnt / 2 > 0 ? kCnt / 2 : 1)];           // one lane holds all values
                    mloc[jj] = row_mean_gxhat(vals[jj], rs_q, Hf, inv_h);
                }
            }
            // phase 3: outputs and leaves.  An empty slot holds zeros; its rstd is
            // taken as 0, so its leaf is exactly +0 (the tree of a whole block adds
            // +0 for ids past the last row) whatever eps is.  The group's rows form
            // a complete subtree with static positions (sub: its pending partials)
            TreeStackF2<NF, (kLogU > 0 ? kLogU : 1)> sub;
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const SlotEntry e = tb[q];
                const uint32_t act = e.nb;
                const float rs_row = __shfl_sync(kFull, rloc[q & (kCnt - 1)], holder(q));   // every lane
                const float rstd = act ? rs_row : 0.f;
                const f2_t r2 = f2_make(rstd, rstd);
                f2_t xf[NF], xh[NF], o[NF];
                vec_unpack_v(xv[q], xf);
#pragma unroll
                for (int i = 0; i < NF; ++i) xh[i] = f2_mul(xf[i], r2);
                if (T::kFwdLike) {
#pragma unroll
                    for (int i = 0; i < NF; ++i) o[i] = f2_mul(xh[i], wv[i]);
                    uint4 ov;
                    vec_pack(o, ov);
                    st_global_vec_if(gout + e.boff, ov, act & out_mask);
                    if (MODE == kAddFwd)
                        st_global_vec_if(reinterpret_cast<uint8_t *>(p.out2 + col0) + e.boff, xv[q], act & vec_mask);
                    if (p.rstd_out != nullptr) st_global_f32_if(p.rstd_out + e.row, rstd, act && tl == 0);
                } else {
                    f2_t df[NF];
                    vec_unpack_v(dv[q], df);
                    if (T::kNeedGx) {
                        const float mg = __shfl_sync(kFull, mloc[(kU + q) & (kCnt - 1)], holder(kU + q));
                        const f2_t nm2 = f2_make(-mg, -mg);
                        const float rs = __fmul_rn(rstd, p.grad_scale);    // == rstd when unscaled
                        const f2_t rs2 = f2_make(rs, rs);
#pragma unroll
                        for (int i = 0; i < NF; ++i) o[i] = f2_mul(rs2, f2_fma(xh[i], nm2, f2_mul(df[i], wv[i])));
                        if (kDres) {
                            f2_t rf[NF];
                            vec_unpack_v(rv[q % kRv], rf);
#pragma unroll
                            for (int i = 0; i < NF; ++i) o[i] = f2_add(o[i], rf[i]);
                        }
                        uint4 ov;
                        vec_pack(o, ov);
                        st_global_vec_if(gout + e.boff, ov, act & out_mask);
                    }
                    if (T::kLeaves) {
                        f2_t leaf[NF];
#pragma unroll
                        for (int i = 0; i < NF; ++i) leaf[i] = f2_mul(df[i], xh[i]);
                        st_global_f2_if(p.ws.spill + int64_t(e.row) * H + col0, leaf, act ? spill_mask : 0u);
                        if (kLogU > 0) sub.template push_static<0>(leaf, q);
                        if (q == kU - 1) {
#pragma unroll
                            for (int i = 0; i < NF; ++i) node[i] = leaf[i];   // the group's subtree
                        }
                    }
                }
            }
            if (spill_mask != 0 && tl == 0) {                // the spilled rows' flags
#pragma unroll
                for (int q = 0; q < kU; ++q) {
                    const SlotEntry e = tb[q];
                    if (e.nb) mark_spilled_row(p.ws, e.row);
                }
            }
            if (whole && kLogGroups > 0) push_group_subtree<NF, kLogGroups>(node, g, stack_lane, 32 * 32);
        }
        if (whole) {
            // node is the team's subtree; the TPW subtrees, adjacent teams first
#pragma unroll
            for (int kk = P; kk < 32; kk <<= 1)
#pragma unroll
                for (int i = 0; i < NF; ++i) node[i] = f2_add(node[i], shfl_xor_f2(node[i], kk));
            if (team == 0) st_global_f2_if(p.ws.block_partial + int64_t(block) * 4 * H + col0, node, vec_mask);
            if (lane == 0) mark_whole_block(p.ws, block);
        }
    }
    cp_async_wait<0>();
}

}  // namespace rbi
