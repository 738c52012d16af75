// Launch shapes of the row kernels.  They depend on the hidden size, the mode
// and the device's SM count only; which CTA handles which row never changes a
// value, so results are identical for every grid.
#pragma once
#include "host.cuh"

// Fewest rows a team of a small call is given (see launch_split_t).
#ifndef RBI_MIN_TEAM_ROWS
#define RBI_MIN_TEAM_ROWS 128
#endif

namespace rbi {

// ---------------------------------------------------------------- launches

template <int MODE, int R, int MAXT, int NS, int K>
int launch_split_t(const KParams &p, const Shape &sh, const DeviceInfo &d, cudaStream_t stream) {
    constexpr int nt = ModeTraits<MODE>::kTensors;
    const int slice = p.hidden / K;
    const int64_t stage_bytes = int64_t(R) * nt * slice * 2;
    const int64_t off = split_stage_off(slice);
    int S = int((int64_t(d.max_smem) - off) / stage_bytes);
    if (S > kSplitMaxStages) S = kSplitMaxStages;
    if (S < 2) return RMSNORM_ERR_HIDDEN;
    const int smem = int(off + S * stage_bytes);
    const int threads = (sh.nc + NS + 1) * 32;
    if (threads > MAXT) return RMSNORM_ERR_HIDDEN;
    auto kern = split_kernel<MODE, R, MAXT, NS, K>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int64_t teams;
    if (K > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = K;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(K * d.sms);
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active < 1) return RMSNORM_ERR_CUDA;
        teams = active;
    } else {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
            return RMSNORM_ERR_CUDA;
        teams = int64_t(per_sm) * d.sms;
    }
    // Every team pays the pipeline's ramp (barrier set-up, first metadata and
    // bulk-copy latency).  A call too small to give every resident team 64 rows
    // gives each team at least 128 rows instead of spreading a few rows over
    // every SM, but keeps at least an eighth of the resident teams; calls
    // issued on other streams fill the rest.  Measured on the many-call layouts
    // (calls of 4096 slots at hidden 5120, 2048 slots at hidden 8192): 128 rows
    // beat 64 by 1-2%, 32 and 256 rows lost 2-9%; a call that fills the GPU at
    // 64 rows per team (13,322 rows at hidden 4096) keeps every team.
    {
        const int64_t rows_per_unit = (p.use_plan && ModeTraits<MODE>::kLeaves) ? kSplitUnitRows : R;
        const int64_t units64 = (64 + rows_per_unit - 1) / rows_per_unit;
        if ((p.n_units + units64 - 1) / units64 < teams) {
            const int64_t min_units = (RBI_MIN_TEAM_ROWS + rows_per_unit - 1) / rows_per_unit;
            int64_t want = (p.n_units + min_units - 1) / min_units;
            if (want < teams / 8) want = teams / 8;
            if (want < teams) teams = want;
        }
    }
    if (teams > p.n_units) teams = p.n_units;
    if (teams < 1) return RMSNORM_OK;
    cfg.gridDim = dim3(unsigned(teams * K));
    if (cudaLaunchKernelEx(&cfg, kern, p, S, sh.nc) != cudaSuccess) return RMSNORM_ERR_CUDA;
    count_launch();
    return RMSNORM_OK;
}

// The CTA shape: column warps (from the hidden size), stats warps and one
// producer.  A CTA's warps are spread over the SM's four sub-partitions, so
// up to 20 warps (640 threads) leave 96 registers per thread and 21 to 24
// warps 80.  Three stats warps whenever the CTA stays within 640 threads;
// beyond that the backward takes three in 768 threads (the same 80
// registers as 736; hidden 5120 in 256 calls of 4096 token slots: -0.9% per
// step) and the forward two in
// 736; a single CTA's forward keeps two.  Measured: hidden 4096 backward
// 0.73 -> 0.75 of the peak with three; on the 2-CTA clusters of hidden 8192,
// with the row-sum exchange by st.async, three beat six (736 threads) by 5%
// on hidden 8192 in 117 calls of 2048 token slots and four by 7%.  Only the shapes that hidden sizes up to
// 16384 reach are instantiated: a slice has at most 20 column warps, and at
// most 16 on 4-CTA clusters.
template <int MODE, int R, int K>
int launch_split_k(const KParams &p, const Shape &sh, const DeviceInfo &d, cudaStream_t stream) {
    constexpr bool kFwd = ModeTraits<MODE>::kFwdLike;
    constexpr int kStats = (kFwd && K == 1) ? kSplitStatsWarps : 3;
    if ((sh.nc + kStats + 1) * 32 <= 640) return launch_split_t<MODE, R, 640, kStats, K>(p, sh, d, stream);
    if constexpr (K == 4) {
        return RMSNORM_ERR_HIDDEN;
    } else if constexpr (!kFwd) {
        return launch_split_t<MODE, R, 768, 3, K>(p, sh, d, stream);
    } else {
        if (kStats > kSplitStatsWarps && (sh.nc + kSplitStatsWarps + 1) * 32 <= 640)
            return launch_split_t<MODE, R, 640, kSplitStatsWarps, K>(p, sh, d, stream);
        return launch_split_t<MODE, R, 736, kSplitStatsWarps, K>(p, sh, d, stream);
    }
}

template <int MODE, int R>
int launch_split(const KParams &p, const Shape &sh, const DeviceInfo &d, cudaStream_t stream) {
    switch (sh.k) {
        case 1: return launch_split_k<MODE, R, 1>(p, sh, d, stream);
        case 2: return launch_split_k<MODE, R, 2>(p, sh, d, stream);
        case 4: return launch_split_k<MODE, R, 4>(p, sh, d, stream);
        default: return RMSNORM_ERR_HIDDEN;
    }
}

template <int MODE, int P>
int launch_small(const KParams &p, const DeviceInfo &d, cudaStream_t stream) {
    constexpr int smem = kSmallWarps * SmallShape<MODE, P>::kWarpBytes;
    constexpr int threads = kSmallWarps * 32;
    auto kern = small_row_kernel<MODE, P>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
        return RMSNORM_ERR_CUDA;
    int64_t blocks = int64_t(per_sm) * d.sms;
    const int64_t need = (p.n_units + kSmallWarps - 1) / kSmallWarps;   // one unit per warp at least
    if (blocks > need) blocks = need;
    if (blocks < 1) return RMSNORM_OK;
    kern<<<unsigned(blocks), threads, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
    count_launch();
    return RMSNORM_OK;
}

template <int MODE>
int launch_small_p(const KParams &p, const Shape &sh, const DeviceInfo &d, cudaStream_t s) {
    switch (sh.p2) {
        case 1: return launch_small<MODE, 1>(p, d, s);
        case 2: return launch_small<MODE, 2>(p, d, s);
        case 4: return launch_small<MODE, 4>(p, d, s);
        case 8: return launch_small<MODE, 8>(p, d, s);
        case 16: return launch_small<MODE, 16>(p, d, s);
        case 32: return launch_small<MODE, 32>(p, d, s);
        default: return RMSNORM_ERR_HIDDEN;
    }
}

template <int MODE>
int run_rows(KParams p, const Shape &sh, const rmsnorm_layout_t *L, cudaStream_t stream) {
    DeviceInfo *d = nullptr;
    int rc = device_info(&d);
    if (rc != RMSNORM_OK) return rc;
    constexpr bool leaves = ModeTraits<MODE>::kLeaves;
    const bool plan = p.use_plan != 0;
    if (sh.small) {
        p.n_units = plan ? L->plan_items : (p.n_rows + kBlockRows - 1) / kBlockRows;
        if (p.n_units == 0) return RMSNORM_OK;
        return launch_small_p<MODE>(p, sh, *d, stream);
    }
    constexpr int R = (MODE == kFwd) ? 4 : 2;            // rows per pipeline stage (measured best)
    if (plan) p.n_units = leaves ? L->plan_items * 4 : L->plan_items * (kBlockRows / R);
    else p.n_units = (p.n_rows + R - 1) / R;
    if (p.n_units == 0) return RMSNORM_OK;
    return launch_split<MODE, R>(p, sh, *d, stream);
}

}  // namespace rbi
