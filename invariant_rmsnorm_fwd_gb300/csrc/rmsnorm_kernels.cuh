// Kernels of the batch-invariant RMSNorm library (sm_103a).
//
// Two kernel families share the numeric helpers of rbi_device.cuh:
//
//  * row_team_kernel (hidden > 256): a "team" of K CTAs (a thread-block
//    cluster when K > 1) owns one row at a time; every thread owns one
//    16-byte vector of 8 columns.  Rows are staged into shared memory by 1-D
//    bulk copies (cp.async.bulk + mbarrier transaction counts) issued S
//    batches ahead by one elected thread; each batch holds R rows.  Per batch
//    the team forms the row sums (lane butterfly, then a butterfly over the
//    warp partials, exchanged through distributed shared memory when K > 1),
//    then writes y or dx and feeds the dweight leaves of the batch into the
//    64-leaf tree held in registers.  CTAs are persistent: cluster c takes
//    work units c, c + n_clusters, ...
//
//  * small_row_kernel (hidden <= 256): a team is P2 = next_pow2(hidden/8)
//    lanes of one warp, so a warp works on 32/P2 rows at once with 16-byte
//    vector loads straight into registers; the rows of a step are combined
//    across teams by a butterfly before entering the 64-leaf tree.
//
// Work units are either plan items (64 row slots: a whole logical block in
// logical order, or rows of blocks cut by a call boundary) or, without a
// plan, 64 consecutive physical rows / R-row batches whose tok_id says
// whether a row is active.  Which unit a CTA processes never changes a
// value: every output depends only on its row (y, dx, the leaf) or on the
// fixed trees.
#pragma once
#include "rbi_device.cuh"

namespace rbi {

enum Mode : int { kFwd = 0, kDx = 1, kDxDw = 2, kDw = 3 };

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

struct KParams {
    const uint16_t *x;
    const uint16_t *dy;
    const uint16_t *w;
    uint16_t *out;                   // y (kFwd) or dx (kDx, kDxDw); may be null in kDxDw
    float *rstd_out;                 // kFwd, optional
    const int32_t *tok_id;
    int64_t n_rows;                  // physical rows of the call = n_tokens * rpt
    int64_t token_stride;            // elements
    int32_t rpt;                     // rows per token
    int32_t hidden;
    float eps;
    int32_t use_plan;                // 1: units are plan items
    const PlanItem *items;
    int64_t n_units;                 // plan items, or batches / 64-row groups without a plan
    WsView ws;
};

__device__ __forceinline__ int64_t row_offset(const KParams &p, int64_t prow) {
    if (p.rpt == 1) return prow * p.token_stride;
    const int64_t t = prow / p.rpt;
    return t * p.token_stride + (prow - t * p.rpt) * int64_t(p.hidden);
}

template <int MODE>
struct ModeTraits {
    static constexpr bool kNeedDy = MODE != kFwd;
    static constexpr bool kNeedGx = MODE == kDx || MODE == kDxDw;   // sum(g*x) for dx
    static constexpr bool kLeaves = MODE == kDxDw || MODE == kDw;
    static constexpr bool kWritesOut = MODE != kDw;
    static constexpr int kTensors = kNeedDy ? 2 : 1;
};

// Book-keeping of contributions (one thread per team).  A block's four state
// bytes say how it arrived: 2 2 2 2 = one whole-block partial (slot 0),
// 1 1 1 1 = four quarter partials (slots 0..3), 0 0 0 0 = its rows were
// spilled.  Any contribution that meets an earlier one is a double count.
constexpr uint32_t kStateWhole = 0x02020202u;
constexpr uint8_t kStateQuarter = 1;

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
    st[q] = kStateQuarter;
}

__device__ __forceinline__ void mark_spilled_row(const WsView &ws, int64_t lrow) {
    const uint32_t st = reinterpret_cast<const uint32_t *>(ws.block_state)[lrow / kBlockRows];
    if (ws.leaf_flag[lrow] != 0 || st != 0) set_status(ws.hdr, kStDouble);
    ws.leaf_flag[lrow] = 1;
}

// =====================================================================
// Large hidden sizes: team = K CTAs, one vector per thread, bulk-copy staging
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

// Shared-memory header of row_team_kernel: barriers, abort flag, per-stage
// row metadata, and the warp partials of the row sums.
constexpr int kMaxStages = 8;
constexpr int kMaxBatch = 8;                     // R <= 8
constexpr int kMaxTeamWarps = 64;                // W <= 64
constexpr int kMaxVals = 16;                     // row sums per batch <= 16
constexpr int kSmemMetaOff = 128;
constexpr int kSmemRedOff = kSmemMetaOff + kMaxStages * kMaxBatch * 16;
constexpr int kSmemStageOff = kSmemRedOff + 2 * 16 * kMaxVals * 4;   // [2 parity][16 local warps][kMaxVals]
static_assert(kSmemStageOff % 128 == 0, "stage buffers are 128-byte aligned");

template <int MODE, int K, int R>
__global__ void __launch_bounds__(512, 1) row_team_kernel(const KParams p, const int S) {
    using T = ModeTraits<MODE>;
    constexpr int kNB = kBlockRows / R;                 // batches per plan item
    constexpr int kLogR = (R == 1) ? 0 : (R == 2) ? 1 : (R == 4) ? 2 : 3;
    constexpr int NV = T::kNeedGx ? 2 * R : R;          // row sums reduced per batch
    constexpr int kLogNV = (NV == 2) ? 1 : (NV == 4) ? 2 : (NV == 8) ? 3 : 4;
    constexpr int kSh = 5 - kLogNV;                     // lane >> kSh = value index after reduce
    static_assert(NV <= kMaxVals && R <= kMaxBatch, "batch too large");

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);                       // [kMaxStages]
    int32_t *abort_flag = reinterpret_cast<int32_t *>(smem + 64);
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + kSmemMetaOff);      // [S][R]
    float *red = reinterpret_cast<float *>(smem + kSmemRedOff);                // [2][16][NV]
    uint8_t *stages = smem + kSmemStageOff;                                    // [S][T][R][slice]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t rank = (K > 1) ? cluster_rank() : 0u;
    const int H = p.hidden;
    const int V = H >> 3;
    const int Vc = V / K;                                // vectors per CTA
    const bool has_vec = tid < Vc;
    const int W = nwarps * K;                            // warps in the team
    const uint32_t slice_bytes = uint32_t(Vc) * 16u;
    const int64_t col0 = int64_t(rank) * Vc * 8;        // first column of this CTA
    const int64_t my_col = col0 + int64_t(tid) * 8;     // first column of this thread
    const float Hf = float(H);

    // Work units: plan items (64 slots) for the dweight modes; single R-row
    // batches otherwise (a batch of a plan item, or R consecutive physical rows).
    const bool item_units = p.use_plan && T::kLeaves;
    const int64_t cluster_id = blockIdx.x / K;
    const int64_t n_clusters = gridDim.x / K;
    const int64_t my_units = p.n_units > cluster_id ? (p.n_units - cluster_id + n_clusters - 1) / n_clusters : 0;
    const int64_t per_unit = item_units ? kNB : 1;
    const int64_t n_batches = my_units * per_unit;

    auto stage_ptr = [&](int s, int t, int r) -> uint8_t * {
        return stages + ((int64_t(s) * T::kTensors + t) * R + r) * slice_bytes;
    };

    // ---- producer (thread 0): metadata of batch k, loaded one batch ahead
    auto load_meta = [&](int64_t k, SlotBatch<R> &mb) {
        if (k >= n_batches) return;
        if (p.use_plan) {
            int64_t item;
            int sub;
            if (item_units) {
                item = cluster_id + (k / kNB) * n_clusters;
                sub = int(k % kNB);
            } else {
                const int64_t gb = cluster_id + k * n_clusters;
                item = gb / kNB;
                sub = int(gb % kNB);
            }
            const PlanItem *it = p.items + item;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                mb.prow[r] = it->prow[sub * R + r];
                mb.lrow[r] = it->lrow[sub * R + r];
            }
        } else {
            const int64_t gb = cluster_id + k * n_clusters;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = gb * R + r;
                int32_t id = -1;
                if (row < p.n_rows) id = p.tok_id[row / p.rpt];
                mb.prow[r] = id >= 0 ? int32_t(row) : -1;
                mb.lrow[r] = -1;
            }
        }
    };
    auto issue = [&](int64_t k, const SlotBatch<R> &mb) {
        if (k >= n_batches) return;
        const int s = int(k % S);
        StageMeta *m = meta + s * R;
        uint32_t n_act = 0;
        int64_t offs[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int32_t pr = mb.prow[r], lr = mb.lrow[r];
            bool act = pr >= 0;
            if (act && (pr >= p.n_rows || (T::kLeaves && (lr < 0 || lr >= p.ws.n_rows)))) {
                if (T::kLeaves) set_status(p.ws.hdr, kStPlan);
                act = false;
            }
            offs[r] = act ? row_offset(p, pr) + col0 : -1;
            m[r].off = offs[r];
            m[r].lrow = lr;
            m[r].prow = pr;
            n_act += act ? 1u : 0u;
        }
        mbar_arrive_expect_tx(&bars[s], n_act * slice_bytes * T::kTensors);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (offs[r] < 0) continue;
            bulk_copy_g2s(stage_ptr(s, 0, r), p.x + offs[r], slice_bytes, &bars[s]);
            if (T::kNeedDy) bulk_copy_g2s(stage_ptr(s, 1, r), p.dy + offs[r], slice_bytes, &bars[s]);
        }
    };

    SlotBatch<R> next_meta;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (K > 1) cluster_barrier(); else __syncthreads();
    if (tid == 0) {
        SlotBatch<R> mb;
        for (int64_t k = 0; k < S - 1; ++k) {
            load_meta(k, mb);
            issue(k, mb);
        }
        load_meta(S - 1, next_meta);
    }

    float2 wv[4];
    if (MODE != kDw && has_vec) unpack8x2(*reinterpret_cast<const uint4 *>(p.w + my_col), wv);

    TreeStack2<4> tree;                 // levels >= log2(R): partials of the current block
    int32_t kind = 0, block = -1;

#pragma unroll 1
    for (int64_t k = 0; k < n_batches; ++k) {
        const int s = int(k % S);
        const uint32_t parity = uint32_t((k / S) & 1);
        const int sub = int(k % per_unit);
        if (item_units && sub == 0) {
            const PlanItem *it = p.items + (cluster_id + (k / kNB) * n_clusters);
            kind = it->kind;
            block = it->block;
            if ((kind == 0 && (block < 0 || block >= p.ws.n_blocks)) || (kind != 0 && kind != 1)) {
                if (tid == 0 && rank == 0) set_status(p.ws.hdr, kStPlan);
                kind = 2;                                  // malformed item: contributes nothing
            }
        }
        if (!mbar_wait_bounded(&bars[s], parity)) {
            *abort_flag = 1;
            if (T::kLeaves) set_status(p.ws.hdr, kStTimeout);
        }
        const StageMeta *m = meta + s * R;

        // ---- per-thread partial row sums, then the warp transpose-reduce
        float val[NV];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float a = 0.f, b = 0.f;
            if (m[r].off >= 0 && has_vec) {
                float2 xf[4];
                unpack8x2(ld_shared_v4(stage_ptr(s, 0, r) + tid * 16), xf);
                a = dot8x2(xf, xf);
                if (T::kNeedGx) {
                    float2 df[4], gf[4];
                    unpack8x2(ld_shared_v4(stage_ptr(s, 1, r) + tid * 16), df);
#pragma unroll
                    for (int i = 0; i < 4; ++i) gf[i] = mul2(df[i], wv[i]);
                    b = dot8x2(gf, xf);
                }
            }
            val[r] = a;
            if (T::kNeedGx) val[R + r] = b;
        }
        const float wsum = warp_transpose_reduce<NV>(val, lane);
        float *rb = red + (k & 1) * (16 * kMaxVals);     // [16 local warps][NV] per parity
        if ((lane & ((1 << kSh) - 1)) == 0) rb[warp * kMaxVals + (lane >> kSh)] = wsum;
        if (K > 1) cluster_barrier(); else __syncthreads();
        {
            int ab = *abort_flag;
            if (K > 1) {
#pragma unroll
                for (int q = 0; q < K; ++q)
                    ab |= __float_as_int(ld_cluster_f32(map_to_rank(smem_addr(abort_flag), uint32_t(q))));
            }
            if (ab) {
                // give copies still in flight into our stages a bounded time to land
                if (tid == 0)
                    for (int64_t kk = k + 1; kk < k + S - 1 && kk < n_batches; ++kk)
                        mbar_wait_bounded(&bars[kk % S], uint32_t((kk / S) & 1));
                break;
            }
        }
        if (tid == 0) {
            SlotBatch<R> cur = next_meta;
            issue(k + S - 1, cur);
            load_meta(k + S, next_meta);
        }

        // ---- team sums: lane w takes warp w (+ warp w+32), then the same
        // transpose-reduce over the 32 slots; every warp does it redundantly.
        {
            float tv[NV];
#pragma unroll
            for (int j = 0; j < NV; ++j) tv[j] = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int w = lane + 32 * half;
                if (w < W) {
                    const int cta = w / nwarps, lw = w - cta * nwarps;
                    const float *src = rb + lw * kMaxVals;
#pragma unroll
                    for (int j = 0; j < NV; ++j) {
                        float v;
                        if (K == 1) v = src[j];
                        else v = ld_cluster_f32(map_to_rank(smem_addr(src + j), uint32_t(cta)));
                        tv[j] = half ? __fadd_rn(tv[j], v) : v;
                    }
                }
            }
            const float tsum = warp_transpose_reduce<NV>(tv, lane);
            // lane l now holds team sum j = l >> kSh: ss_j (j < R) or gx_{j-R}
            const int j = lane >> kSh;
            const float rs = row_rstd(tsum, Hf, p.eps);               // meaningful for j < R
            if (T::kNeedGx) {
                const int src_lane = (j >= R ? j - R : j) << kSh;
                const float rs_row = __shfl_sync(kFull, rs, src_lane);
                const float mg = row_mean_gxhat(tsum, rs_row, Hf);    // meaningful for j >= R
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    val[r] = __shfl_sync(kFull, rs, r << kSh);
                    val[R + r] = __shfl_sync(kFull, mg, (R + r) << kSh);
                }
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) val[r] = __shfl_sync(kFull, rs, r << kSh);
            }
        }

        // ---- outputs and dweight leaves
        TreeStack2<4, (kLogR > 0 ? kLogR : 1)> mini;   // levels < log2(R): the batch's own subtree
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool act = m[r].off >= 0;
            const float rstd = val[r];
            float2 leaf[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) leaf[i] = make_float2(0.f, 0.f);
            if (act && has_vec) {
                const float2 r2 = make_float2(rstd, rstd);
                float2 xf[4], xh[4], o[4];
                unpack8x2(ld_shared_v4(stage_ptr(s, 0, r) + tid * 16), xf);
#pragma unroll
                for (int i = 0; i < 4; ++i) xh[i] = mul2(xf[i], r2);
                if (MODE == kFwd) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = mul2(xh[i], wv[i]);
                    st_global_v4(p.out + m[r].off + tid * 8, pack8x2(o));
                } else {
                    float2 df[4];
                    unpack8x2(ld_shared_v4(stage_ptr(s, 1, r) + tid * 16), df);
                    if (T::kNeedGx && p.out != nullptr) {
                        const float nm = -val[R + r];
                        const float2 nm2 = make_float2(nm, nm);
#pragma unroll
                        for (int i = 0; i < 4; ++i) o[i] = mul2(r2, fma2(xh[i], nm2, mul2(df[i], wv[i])));
                        st_global_v4(p.out + m[r].off + tid * 8, pack8x2(o));
                    }
                    if (T::kLeaves) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) leaf[i] = mul2(df[i], xh[i]);
                    }
                }
            }
            if (MODE == kFwd && act && p.rstd_out != nullptr && tid == 0 && rank == 0)
                p.rstd_out[m[r].prow] = rstd;
            if (T::kLeaves) {
                if (kind == 0) {
                    if (R > 1) mini.template push_static<0>(leaf, r);
                    if (r == R - 1) {
                        tree.template push_dyn<kLogR>(leaf, sub);
                        if (sub == kNB - 1) {             // leaf[] is the block partial
                            if (has_vec) {
                                float *dst = p.ws.block_partial + int64_t(block) * 4 * H + my_col;
                                st_global_f32x4(dst, leaf[0].x, leaf[0].y, leaf[1].x, leaf[1].y);
                                st_global_f32x4(dst + 4, leaf[2].x, leaf[2].y, leaf[3].x, leaf[3].y);
                            }
                            if (tid == 0 && rank == 0) mark_whole_block(p.ws, block);
                        }
                    }
                } else if (kind == 1 && act) {
                    if (has_vec) {
                        float *dst = p.ws.spill + int64_t(m[r].lrow) * H + my_col;
                        st_global_f32x4(dst, leaf[0].x, leaf[0].y, leaf[1].x, leaf[1].y);
                        st_global_f32x4(dst + 4, leaf[2].x, leaf[2].y, leaf[3].x, leaf[3].y);
                    }
                    if (tid == 0 && rank == 0) mark_spilled_row(p.ws, m[r].lrow);
                }
            }
        }
    }
    if (K > 1) cluster_barrier();      // peers may still read our partials
}

// =====================================================================
// Hidden sizes 264..5120: warp-specialised pipeline in one CTA
// =====================================================================
//
// Warps [0, NC): column warps; thread t owns columns 8t..8t+7 of every row.
// Warps [NC, NC+NS): stats warps; warp i handles the stages s with s % NS == i.
// Warp NC+NS: producer; lane 0 issues the bulk copies.
//
// Per stage s (R rows of x, dy): full[s] completes when the copies land,
// stats[s] when a stats warp has published rstd and mean(g*xhat) for its
// rows, empty[s] when every column warp is done with it.  No CTA-wide
// barrier is used after set-up.  Rows of the dweight modes are processed in
// 16-row units (a quarter of a logical block): the column warps reduce the
// unit's 16 leaves with the 64-leaf tree's lower four levels and store the
// quarter partial; dweight_finalize adds the four quarters (levels 5, 6).
//
// Row sums (this family's canonical tree, which depends on H only): lane l
// folds vectors l, l+32, l+64, ... in order, columns interleaved as two FMA
// chains (columns 0,2,4,6 and 1,3,5,7 of each vector, one chain across all
// of the lane's vectors), the chains are added, and the 32 lane sums are
// added by a complete tree pairing lanes 16 apart first, then 8, 4, 2, 1.

constexpr int kSplitMaxStages = 12;
constexpr int kSplitUnitRows = 16;

struct SplitStats {
    float rstd;
    float mg;
};

constexpr int kSplitItemOff = 320;                                   // [kSplitMaxStages] int2 item headers
constexpr int kSplitMetaOff = 512;                                   // after 3 x 12 barriers (288 B) + flag
constexpr int kSplitStatsOff = kSplitMetaOff + kSplitMaxStages * kMaxBatch * 16;
constexpr int kSplitWOff = kSplitStatsOff + kSplitMaxStages * kMaxBatch * 8;   // FP32 weight [H]
__host__ __device__ constexpr int split_stage_off(int H) { return ((kSplitWOff + H * 4) + 127) / 128 * 128; }

template <int MODE, int R, int MAXT, int NS>
__global__ void __launch_bounds__(MAXT, 1) split_kernel(const KParams p, const int S, const int NC) {
    using T = ModeTraits<MODE>;
    constexpr int kLogR = (R == 1) ? 0 : (R == 2) ? 1 : (R == 4) ? 2 : 3;
    constexpr int kUnitBatches = kSplitUnitRows / R;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *stats_bar = full + kSplitMaxStages;
    uint64_t *empty = stats_bar + kSplitMaxStages;
    volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(smem + 3 * kSplitMaxStages * 8);
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + kSplitMetaOff);   // [S][R]
    int2 *item_hdr = reinterpret_cast<int2 *>(smem + kSplitItemOff);          // [S] (kind, block)
    SplitStats *stats = reinterpret_cast<SplitStats *>(smem + kSplitStatsOff);
    float *wsm = reinterpret_cast<float *>(smem + kSplitWOff);
    const int H = p.hidden;
    const int V = H >> 3;
    uint8_t *stages = smem + split_stage_off(H);
    const uint32_t row_bytes = uint32_t(H) * 2u;
    auto stage_ptr = [&](int s, int t, int r) -> uint8_t * {
        return stages + ((int64_t(s) * T::kTensors + t) * R + r) * row_bytes;
    };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float Hf = float(H);
    const bool item_units = p.use_plan && T::kLeaves;
    const int64_t per_unit = item_units ? kUnitBatches : 1;
    const int64_t my_units = p.n_units > blockIdx.x ? (p.n_units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int n_batches = int(my_units * per_unit);      // < 2^31: units are bounded by rows / 2

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&stats_bar[s], 1);
            mbar_init(&empty[s], NC);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (MODE != kDw && T::kNeedGx) {
        for (int i = tid; i < H; i += blockDim.x) wsm[i] = __uint_as_float(uint32_t(p.w[i]) << 16);
    }
    __syncthreads();

    // batch k of this CTA -> (plan item, slot base) or physical row base
    auto batch_slots = [&](int k, int64_t &item, int &slot0) {
        if (item_units) {
            const int64_t u = blockIdx.x + (k / kUnitBatches) * gridDim.x;      // quarter unit
            item = u >> 2;
            slot0 = int(u & 3) * kSplitUnitRows + int(k % kUnitBatches) * R;
        } else {
            const int64_t gb = blockIdx.x + k * gridDim.x;
            if (p.use_plan) {
                item = gb / (kBlockRows / R);
                slot0 = int(gb % (kBlockRows / R)) * R;
            } else {
                item = gb;                                                     // physical batch index
                slot0 = 0;
            }
        }
    };

    if (warp == NC + NS) {
        // ------------------------------------------------ producer
        // The slot metadata of batch k comes from global memory (plan or
        // tok_id); it is loaded kPrefetch batches ahead so that issuing the
        // copies never waits on it.
        if (lane == 0) {
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
                    mb.kind = p.items[item].kind;
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
#pragma unroll
            for (int i = 0; i < kPrefetch; ++i) load(i, ring[i]);
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
                        if (T::kLeaves) set_status(p.ws.hdr, kStPlan);
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
                    bulk_copy_g2s(stage_ptr(s, 0, r), p.x + offs[r], row_bytes, &full[s]);
                    if (T::kNeedDy) bulk_copy_g2s(stage_ptr(s, 1, r), p.dy + offs[r], row_bytes, &full[s]);
                }
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        return;
    }

    if (warp >= NC) {
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
            float vals[2 * R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                f2_t a2 = 0ull, b2 = 0ull;                      // +0.0 in both lanes
                if (m[r].off >= 0) {
                    const uint8_t *xr = stage_ptr(s, 0, r);
                    const uint8_t *dr = stage_ptr(s, 1, r);
#pragma unroll 4
                    for (int v = lane; v < V; v += 32) {
                        f2_t xf[4];
                        f2_unpack8(ld_shared_v4(xr + v * 16), xf);
#pragma unroll
                        for (int i = 0; i < 4; ++i) a2 = f2_fma(xf[i], xf[i], a2);
                        if (T::kNeedGx) {
                            f2_t df[4];
                            f2_unpack8(ld_shared_v4(dr + v * 16), df);
                            const f2_t *wf = reinterpret_cast<const f2_t *>(wsm + v * 8);
#pragma unroll
                            for (int i = 0; i < 4; ++i) b2 = f2_fma(f2_mul(df[i], wf[i]), xf[i], b2);
                        }
                    }
                }
                vals[r] = __fadd_rn(f2_lo(a2), f2_hi(a2));
                vals[R + r] = __fadd_rn(f2_lo(b2), f2_hi(b2));
            }
            // complete tree over the 32 lanes, pairing 16 apart first
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1)
#pragma unroll
                for (int j = 0; j < (T::kNeedGx ? 2 * R : R); ++j)
                    vals[j] = __fadd_rn(vals[j], __shfl_xor_sync(kFull, vals[j], d));
            if (lane < R) {
                float ss = vals[0], gx = vals[R];
#pragma unroll
                for (int r = 1; r < R; ++r)
                    if (lane == r) {
                        ss = vals[r];
                        gx = vals[R + r];
                    }
                const float rstd = row_rstd(ss, Hf, p.eps);
                SplitStats st;
                st.rstd = rstd;
                st.mg = T::kNeedGx ? row_mean_gxhat(gx, rstd, Hf) : 0.f;
                stats[s * R + lane] = st;
                if (MODE == kFwd && p.rstd_out != nullptr && m[lane].off >= 0) p.rstd_out[m[lane].prow] = rstd;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&stats_bar[s]);
        }
        return;
    }

    // ---------------------------------------------------- column warps
    const int t = tid;                                   // vector owned: columns 8t..8t+7
    const bool has_vec = t < V;
    f2_t wv[4];
    if (MODE != kDw && has_vec) f2_unpack8(*reinterpret_cast<const uint4 *>(p.w + t * 8), wv);
    TreeStackF2<4, 4> tree;            // levels log2(R)..3 of the 16-leaf unit
    int32_t kind = 0, block = -1, quarter = 0;
    int s = 0, sub = 0;
    uint32_t parity = 0;
    int64_t u = blockIdx.x;                               // current quarter unit
    for (int k = 0; k < n_batches; ++k) {
        if (k > 0) {
            if (++s == S) {
                s = 0;
                parity ^= 1u;
            }
            if (++sub == per_unit) {
                sub = 0;
                u += gridDim.x;
            }
        }
        if (*abort_flag) break;
        if (!mbar_wait_bounded(&stats_bar[s], parity) || !mbar_wait_bounded(&full[s], parity)) {
            *abort_flag = 1;
            if (T::kLeaves) set_status(p.ws.hdr, kStTimeout);
            break;
        }
        if (item_units && sub == 0) {                    // item header, staged by the producer
            const int2 hd = item_hdr[s];
            quarter = int(u & 3);
            kind = hd.x;
            block = hd.y;
            if ((kind == 0 && (block < 0 || block >= p.ws.n_blocks)) || (kind != 0 && kind != 1)) {
                if (t == 0) set_status(p.ws.hdr, kStPlan);
                kind = 2;
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
                f2_unpack8(ld_shared_v4(stage_ptr(s, 0, r) + t * 16), xf);
#pragma unroll
                for (int i = 0; i < 4; ++i) xh[i] = f2_mul(xf[i], r2);
                if (MODE == kFwd) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = f2_mul(xh[i], wv[i]);
                    st_global_v4(p.out + off + t * 8, f2_pack8(o));
                } else {
                    f2_t df[4];
                    f2_unpack8(ld_shared_v4(stage_ptr(s, 1, r) + t * 16), df);
                    if (T::kNeedGx && p.out != nullptr) {
                        const f2_t nm2 = f2_make(-st.mg, -st.mg);
#pragma unroll
                        for (int i = 0; i < 4; ++i) o[i] = f2_mul(r2, f2_fma(xh[i], nm2, f2_mul(df[i], wv[i])));
                        st_global_v4(p.out + off + t * 8, f2_pack8(o));
                    }
                    if (T::kLeaves) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) leaf[i] = f2_mul(df[i], xh[i]);
                    }
                }
            }
            if (T::kLeaves) {
                if (kind == 0) {
                    if (R > 1) mini.template push_static<0>(leaf, r);
                    if (r == R - 1) {
                        tree.template push_dyn<kLogR>(leaf, sub);
                        if (sub == kUnitBatches - 1) {           // leaf[] is the quarter partial
                            if (has_vec)
                                st_global_f2x4(p.ws.block_partial + (int64_t(block) * 4 + quarter) * H + t * 8, leaf);
                            if (t == 0) mark_quarter(p.ws, block, quarter);
                        }
                    }
                } else if (kind == 1 && act) {
                    if (has_vec) st_global_f2x4(p.ws.spill + int64_t(m[r].lrow) * H + t * 8, leaf);
                    if (t == 0) mark_spilled_row(p.ws, m[r].lrow);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// =====================================================================
// Small hidden sizes: team = P2 lanes of a warp, register-direct loads
// =====================================================================

template <int MODE, int P2, int U>
__global__ void __launch_bounds__(256) small_row_kernel(const KParams p) {
    using T = ModeTraits<MODE>;
    constexpr int TPW = 32 / P2;                         // teams (rows) per warp step
    constexpr int kSteps = kBlockRows / TPW;             // steps per 64-slot unit
    constexpr int kLogTPW = (TPW == 1) ? 0 : (TPW == 2) ? 1 : (TPW == 4) ? 2 : (TPW == 8) ? 3 : (TPW == 16) ? 4 : 5;
    static_assert(kSteps % U == 0 || U >= kSteps, "steps per unit must be a multiple of U");
    constexpr int kU = U < kSteps ? U : kSteps;

    const int lane = threadIdx.x & 31;
    const int team = lane / P2, tl = lane % P2;
    const int H = p.hidden, V = H >> 3;
    const bool has_vec = tl < V;
    const float Hf = float(H);
    const int64_t gwarp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;

    float wv[8];
    if (MODE != kDw && has_vec) unpack8(*reinterpret_cast<const uint4 *>(p.w + tl * 8), wv);

#pragma unroll 1
    for (int64_t u = gwarp; u < p.n_units; u += nwarps) {
        const PlanItem *it = p.use_plan ? p.items + u : nullptr;
        int32_t kind = 0, block = -1;
        if (it) {
            kind = it->kind;
            block = it->block;
            if (T::kLeaves && ((kind == 0 && (block < 0 || block >= p.ws.n_blocks)) || (kind != 0 && kind != 1))) {
                if (lane == 0) set_status(p.ws.hdr, kStPlan);
                kind = 2;                                  // malformed item: contributes nothing
            }
        }
        TreeStack<8> tree;
#pragma unroll 1
        for (int st0 = 0; st0 < kSteps; st0 += kU) {
            // resolve slots and issue loads for kU steps
            int64_t off[kU];
            int32_t lrow[kU], prow[kU];
            uint4 xv[kU], dv[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int slot = (st0 + q) * TPW + team;
                int32_t pr, lr = -1;
                if (it) {
                    pr = it->prow[slot];
                    lr = it->lrow[slot];
                } else {
                    const int64_t row = u * kBlockRows + slot;
                    pr = (row < p.n_rows && p.tok_id[row / p.rpt] >= 0) ? int32_t(row) : -1;
                }
                bool act = pr >= 0;
                if (act && (pr >= p.n_rows || (T::kLeaves && (lr < 0 || lr >= p.ws.n_rows)))) {
                    if (T::kLeaves && tl == 0) set_status(p.ws.hdr, kStPlan);
                    act = false;
                }
                off[q] = act ? row_offset(p, pr) + tl * 8 : -1;
                lrow[q] = lr;
                prow[q] = pr;
                xv[q] = make_uint4(0, 0, 0, 0);
                dv[q] = make_uint4(0, 0, 0, 0);
                if (act && has_vec) {
                    xv[q] = ld_global_stream_v4(p.x + off[q]);
                    if (T::kNeedDy) dv[q] = ld_global_stream_v4(p.dy + off[q]);
                }
            }
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const bool act = off[q] >= 0;
                float xf[8], df[8];
                unpack8(xv[q], xf);
                unpack8(dv[q], df);
                float ss = 0.f, gx = 0.f;
                if (act && has_vec) {
                    ss = dot8(xf, xf);
                    if (T::kNeedGx) {
                        float gf[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) gf[i] = __fmul_rn(df[i], wv[i]);
                        gx = dot8(gf, xf);
                    }
                }
                ss = lane_tree(ss, P2);
                if (T::kNeedGx) gx = lane_tree(gx, P2);
                const float rstd = row_rstd(ss, Hf, p.eps);
                float leaf[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) leaf[i] = 0.f;
                if (act && has_vec) {
                    float xh[8], o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) xh[i] = __fmul_rn(xf[i], rstd);
                    if (MODE == kFwd) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) o[i] = __fmul_rn(xh[i], wv[i]);
                        st_global_v4(p.out + off[q], pack8(o));
                    } else {
                        if (T::kNeedGx && p.out != nullptr) {
                            const float mg = row_mean_gxhat(gx, rstd, Hf);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float g = __fmul_rn(df[i], wv[i]);
                                o[i] = __fmul_rn(rstd, __fmaf_rn(-xh[i], mg, g));
                            }
                            st_global_v4(p.out + off[q], pack8(o));
                        }
                        if (T::kLeaves) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) leaf[i] = __fmul_rn(df[i], xh[i]);
                        }
                    }
                }
                if (MODE == kFwd && act && p.rstd_out != nullptr && tl == 0) p.rstd_out[prow[q]] = rstd;
                if (T::kLeaves) {
                    if (kind == 0) {
                        // combine the TPW rows of this step (adjacent teams first)
#pragma unroll
                        for (int kk = P2; kk < 32; kk <<= 1)
#pragma unroll
                            for (int i = 0; i < 8; ++i) leaf[i] = __fadd_rn(leaf[i], __shfl_xor_sync(kFull, leaf[i], kk));
                        tree.push(leaf, st0 + q, kLogTPW);
                        if (st0 + q == kSteps - 1 && team == 0 && has_vec) {
                            float *dst = p.ws.block_partial + int64_t(block) * 4 * H + tl * 8;
                            st_global_f32x4(dst, leaf[0], leaf[1], leaf[2], leaf[3]);
                            st_global_f32x4(dst + 4, leaf[4], leaf[5], leaf[6], leaf[7]);
                        }
                        if (st0 + q == kSteps - 1 && lane == 0) mark_whole_block(p.ws, block);
                    } else if (kind == 1 && act) {
                        if (has_vec) {
                            float *dst = p.ws.spill + int64_t(lrow[q]) * H + tl * 8;
                            st_global_f32x4(dst, leaf[0], leaf[1], leaf[2], leaf[3]);
                            st_global_f32x4(dst + 4, leaf[4], leaf[5], leaf[6], leaf[7]);
                        }
                        if (tl == 0) mark_spilled_row(p.ws, lrow[q]);
                    }
                }
            }
        }
    }
}

// =====================================================================
// Workspace set-up and the final reduction
// =====================================================================

__global__ void ws_begin_kernel(WsView ws) {
    const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = int64_t(gridDim.x) * blockDim.x;
    // block_state and leaf_flag are contiguous up to the partials: clear both
    uint8_t *base = ws.block_state;
    const int64_t bytes = reinterpret_cast<uint8_t *>(ws.block_partial) - base;   // multiple of 256
    uint4 *b4 = reinterpret_cast<uint4 *>(base);
    for (int64_t i = tid; i < bytes / 16; i += nthr) b4[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        ws.hdr->n_rows = ws.n_rows;
        ws.hdr->hidden = ws.hidden;
        ws.hdr->n_blocks = ws.n_blocks;
        ws.hdr->status = 0;
        ws.hdr->magic = kWsMagic;
    }
}

// One pass of the block-partial tree.  Warp (g, v) reduces the partials
// [32g, 32g+32) of columns 8v..8v+7: lane b holds partial 32g+b, and the 32
// lanes are combined by butterflies xor 1, 2, 4, 8, 16 where a pair is added
// only if its right half is non-empty, which is exactly the pairwise tree
// with odd carry restricted to an aligned group of 32 (later passes reduce
// the group results the same way).  In the first pass (from_blocks) lane b
// first forms block b's partial: the four quarter partials as
// (q0 + q1) + (q2 + q3) (levels 5 and 6 of the 64-leaf tree), a whole-block
// partial as is, or, for a block cut by a call boundary, the 64-leaf tree
// over its spilled rows, computed by the whole warp (lane l adds rows 2l and
// 2l+1, then butterflies xor 1..16): the same tree as the in-kernel path.
__device__ __forceinline__ void load8(const float *src, float (&v)[8]) {
    const float4 a = ld_global_f32x4(src), b = ld_global_f32x4(src + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

constexpr int kTreeWarps = 8;                            // warps (vectors) per CTA

__global__ void __launch_bounds__(kTreeWarps * 32) tree_pass_kernel(WsView ws, const float *in, float *out,
                                                                    int64_t n_in, int from_blocks) {
    const int H = int(ws.hidden), V = H >> 3;
    const int lane = threadIdx.x & 31;
    const int v = blockIdx.y * kTreeWarps + (threadIdx.x >> 5);
    if (v >= V) return;                                  // whole warp leaves together
    const int64_t g = blockIdx.x;
    const int64_t b = g * 32 + lane;
    const int m = int(min64(32, n_in - g * 32));          // inputs in this group
    if (from_blocks && !header_ok(ws)) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) set_status(ws.hdr, kStHeader);
        return;
    }
    float val[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) val[c] = 0.f;
    const bool present = lane < m;
    uint32_t state = kStateWhole;
    if (present && from_blocks) state = reinterpret_cast<const uint32_t *>(ws.block_state)[b];
    if (present) {
        if (!from_blocks) {
            load8(in + b * int64_t(H) + int64_t(v) * 8, val);
        } else if (state == 0x01010101u) {
            float q0[8], q1[8], q2[8], q3[8];
            const float *src = ws.block_partial + b * 4 * int64_t(H) + int64_t(v) * 8;
            load8(src, q0);
            load8(src + H, q1);
            load8(src + 2 * int64_t(H), q2);
            load8(src + 3 * int64_t(H), q3);
#pragma unroll
            for (int c = 0; c < 8; ++c) val[c] = __fadd_rn(__fadd_rn(q0[c], q1[c]), __fadd_rn(q2[c], q3[c]));
        } else if (state == kStateWhole) {
            load8(ws.block_partial + b * 4 * int64_t(H) + int64_t(v) * 8, val);
        } else if (state != 0) {
            if (v == 0) set_status(ws.hdr, kStMissing);  // partly contributed block
        }
    }
    // blocks cut by a call boundary: rebuilt by the whole warp, one at a time
    uint32_t cut = __ballot_sync(kFull, present && from_blocks && state == 0);
    while (cut) {
        const int bb = __ffs(cut) - 1;
        cut &= cut - 1;
        const int64_t blk = g * 32 + bb;
        const int64_t rows = min64(kBlockRows, ws.n_rows - blk * kBlockRows);
        const int64_t r0 = blk * kBlockRows + 2 * lane;
        float a[8], c2[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) a[c] = c2[c] = 0.f;
        bool missing = false;
        if (2 * lane < rows) {
            load8(ws.spill + r0 * int64_t(H) + int64_t(v) * 8, a);
            missing |= ws.leaf_flag[r0] == 0;
        }
        if (2 * lane + 1 < rows) {
            load8(ws.spill + (r0 + 1) * int64_t(H) + int64_t(v) * 8, c2);
            missing |= ws.leaf_flag[r0 + 1] == 0;
        }
        if (__any_sync(kFull, missing) && v == 0 && lane == 0) set_status(ws.hdr, kStMissing);
#pragma unroll
        for (int c = 0; c < 8; ++c) a[c] = __fadd_rn(a[c], c2[c]);            // level 1: rows 2l, 2l+1
#pragma unroll
        for (int k = 1; k < 32; k <<= 1)
#pragma unroll
            for (int c = 0; c < 8; ++c) a[c] = __fadd_rn(a[c], __shfl_xor_sync(kFull, a[c], k));
        if (lane == bb) {
#pragma unroll
            for (int c = 0; c < 8; ++c) val[c] = a[c];
        }
    }
    // carry tree over the group's (up to) 32 partials
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
        const int base = lane & ~(2 * k - 1);
        const bool add = base + k < m;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float o = __shfl_xor_sync(kFull, val[c], k);
            val[c] = add ? __fadd_rn(val[c], o) : val[c];
        }
    }
    if (lane == 0) {
        float *dst = out + g * int64_t(H) + int64_t(v) * 8;
        st_global_f32x4(dst, val[0], val[1], val[2], val[3]);
        st_global_f32x4(dst + 4, val[4], val[5], val[6], val[7]);
    }
}

__global__ void zero_f32_kernel(float *p, int64_t n) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
        p[i] = 0.f;
}

}  // namespace rbi
