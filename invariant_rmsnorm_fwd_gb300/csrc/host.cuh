// Host-side pieces shared by the translation units of the library: device
// properties, the hidden-size shapes and the per-mode row launcher, whose
// instantiations live in rows_*.cu so that they compile in parallel.
#pragma once
#include <cuda_runtime.h>

#include "rmsnorm_bi.h"
#include "rmsnorm_kernels.cuh"

namespace rbi {

struct DeviceInfo {
    bool ready = false;
    int status = RMSNORM_OK;
    int sms = 0;
    int max_smem = 0;
};
int device_info(DeviceInfo **out);   // cached per device; RMSNORM_ERR_DEVICE unless sm_103
void count_launch();                 // one more kernel of this library enqueued

// ---------------------------------------------------------------- shapes

struct Shape {
    bool small = false;   // small_row_kernel
    int p2 = 0;           // lanes per row (small)
    int k = 1;            // CTAs per row team (split_kernel), a cluster when > 1
    int nc = 0;           // column warps per CTA (split_kernel)
};

constexpr int kSplitStatsWarps = 2;
constexpr int kSliceMaxVectors = 640;                    // columns per CTA <= 5120

inline bool hidden_shape(int64_t H, Shape *s) {
    if (H < 8 || H % 8 != 0 || H > 16384) return false;
    const int64_t V = H / 8;
    if (V <= 32) {
        s->small = true;
        int p = 1;
        while (p < V) p <<= 1;
        s->p2 = p;
        return true;
    }
    for (int k = 1; k <= kSplitMaxK; k *= 2) {
        if (V % k == 0 && V / k <= kSliceMaxVectors) {
            s->k = k;
            s->nc = int((V / k + 31) / 32);
            return true;
        }
    }
    return false;
}

// Runs the rows of one call in the given mode (rows_*.cu instantiate it).
template <int MODE>
int run_rows(KParams p, const Shape &sh, const rmsnorm_layout_t *L, cudaStream_t stream);

}  // namespace rbi
