// Kernels of the workspace: set-up, the finalize tree and the top of the
// tree over roots gathered from several ranks.  Included by the C-ABI
// translation unit only.
#pragma once
#include "rmsnorm_kernels.cuh"

namespace rbi {

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

// One pass of the block-partial tree over groups of 32 inputs.  CTA (g, c)
// reduces inputs [32g, 32g+32) for the 32 vectors (256 columns) of chunk c:
// lane l owns vector 32c+l, so every load of a warp is one contiguous 512-byte
// row piece.  Warp w forms inputs 2w and 2w+1 and adds them (level 1); the 16
// pair results go through shared memory, and levels 2-5 are added in
// registers by 8 warps (one column of the 32 vectors each) for a full group,
// level by level by the CTA's warps for the last, partial group of a pass.
// Pairs are added only when their right half is non-empty, which is the
// pairwise tree with odd carry restricted to an aligned group of 32; later
// passes reduce the group results the same way.
// In the first pass (from_blocks) an input is a block partial: the four
// quarter partials as (q0 + q1) + (q2 + q3) (levels 5 and 6 of the 64-leaf
// tree), a whole-block partial as is, or, for a block cut by a call boundary,
// its four quarters, each one a quarter partial computed by the call that
// held the whole quarter or the 16-leaf tree over the quarter's spilled rows,
// rebuilt by each lane for its own 8-column vector (pairs (0,1), (2,3), ...
// at every level): the same tree as the in-kernel path.
__device__ __forceinline__ void load8(const float *src, float (&v)[8]) {
    const float4 a = ld_global_f32x4(src), b = ld_global_f32x4(src + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Every quarter of the block arrived, each as one quarter partial (byte 1) or
// as two eighth partials (byte 12).
__device__ __forceinline__ bool quarter_state(uint32_t state) {
    bool ok = true;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t b = (state >> (8 * k)) & 0xffu;
        ok &= b == kStateQuarter || b == (kStateEighth0 | kStateEighth1);
    }
    return ok;
}
__device__ __forceinline__ void add_second_eighth(uint32_t state, int q, const float *src, float (&v)[8]) {
    if (((state >> (8 * q)) & 0xffu) != (kStateEighth0 | kStateEighth1)) return;
    float e[8];
    load8(src, e);
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = __fadd_rn(v[c], e[c]);
}

// The 16-leaf subtree of quarter q of a block from its spilled rows, for one
// 8-column vector (src points at the block's row 0 of that vector): rows at or
// beyond `rows` (past the multiset) are +0.0 leaves.  Four rows are loaded at a
// time (levels 1-2 of the tree over them), then the four quads are added
// pairwise (levels 3-4), earlier rows always on the left.
__device__ __forceinline__ void quarter_from_spill(const float *src, int H, int q, int64_t rows, float (&out)[8]) {
    float n[2][8];
#pragma unroll
    for (int quad = 0; quad < 4; ++quad) {
        float x[4][8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = 16 * q + 4 * quad + k;
            if (r < rows) {
                load8(src + int64_t(r) * H, x[k]);
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) x[k][c] = 0.f;
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float e = __fadd_rn(__fadd_rn(x[0][c], x[1][c]), __fadd_rn(x[2][c], x[3][c]));
            if ((quad & 1) == 0) n[quad >> 1][c] = e;
            else n[quad >> 1][c] = __fadd_rn(n[quad >> 1][c], e);
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) out[c] = __fadd_rn(n[0][c], n[1][c]);
}

constexpr int kTreeWarps = 16;                           // warps per CTA: 2 inputs each
constexpr int kTreeVecs = 32;                            // vectors (8 columns) per CTA

__global__ void __launch_bounds__(kTreeWarps * 32) tree_pass_kernel(WsView ws, const float *in, float *out,
                                                                    int64_t n_in, int from_blocks,
                                                                    int64_t block_base, float scale) {
    __shared__ float part[kTreeWarps][8][kTreeVecs];      // [pair][column][vector]
    const int H = int(ws.hidden), V = H >> 3;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int v = blockIdx.y * kTreeVecs + lane;         // this lane's vector
    const bool has_vec = v < V;
    const int64_t g = blockIdx.x;
    const int m = int(min64(32, n_in - g * 32));          // inputs in this group
    // Everything the warp reads first is requested before any of it is used:
    // the states of the group's inputs (one per lane) and, for each of the
    // warp's two inputs, its four partial slots (the quarters of a block, or
    // its whole partial in slot 0; for a cut block they are read again below)
    // or the group result of the previous pass.  The slots lie inside the
    // workspace whatever the state says, so nothing waits on the state.
    const int64_t base = (from_blocks ? block_base : 0) + g * 32;
    uint32_t st_lane = kStateWhole;
    if (from_blocks && lane < m) st_lane = reinterpret_cast<const uint32_t *>(ws.block_state)[base + lane];
    float slot[2][4][8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = 2 * w + h;
        if (i < m && has_vec) {
            if (from_blocks) {
                const float *src = ws.block_partial + (base + i) * 4 * int64_t(H) + int64_t(v) * 8;
#pragma unroll
                for (int k = 0; k < 4; ++k) load8(src + k * int64_t(H), slot[h][k]);
            } else {
                load8(in + (base + i) * int64_t(H) + int64_t(v) * 8, slot[h][0]);
            }
        }
    }
    const uint32_t states[2] = {__shfl_sync(kFull, st_lane, 2 * w), __shfl_sync(kFull, st_lane, 2 * w + 1)};
    if (from_blocks && !header_ok(ws)) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) set_status(ws.hdr, kStHeader);
        return;                                          // uniform across the CTA
    }
    // The inputs that the slots already give (the previous pass's results,
    // whole blocks, blocks that arrived as quarters or eighths) first, so that
    // the slots are dead before a cut block, which is rebuilt from scratch,
    // needs its registers.
    float val[2][8];
    bool cut[2] = {false, false};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int c = 0; c < 8; ++c) val[h][c] = 0.f;
        const int i = 2 * w + h;
        if (i >= m) continue;                            // uniform per warp
        const int64_t b = base + i;
        const uint32_t state = states[h];
        if (!from_blocks || state == kStateWhole) {
            if (has_vec) {
#pragma unroll
                for (int c = 0; c < 8; ++c) val[h][c] = slot[h][0][c];
            }
        } else if (quarter_state(state)) {
            if (has_vec) {
                const float *src2 = ws.eighth + b * 4 * int64_t(H) + int64_t(v) * 8;
                // a quarter that arrived as two eighths: the halves make level 4
#pragma unroll
                for (int k = 0; k < 4; ++k) add_second_eighth(state, k, src2 + k * int64_t(H), slot[h][k]);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    val[h][c] = __fadd_rn(__fadd_rn(slot[h][0][c], slot[h][1][c]), __fadd_rn(slot[h][2][c], slot[h][3][c]));
            }
        } else {
            cut[h] = true;
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (!cut[h]) continue;                           // uniform per warp
        const int64_t b = base + 2 * w + h;
        const uint32_t state = states[h];
        float (&out8)[8] = val[h];
        // a block cut by a call boundary: each quarter arrived as a partial
        // (byte 1), as two eighth partials (byte 12), or as spilled rows
        // (byte 0), which each lane rebuilds for its own 8-column vector;
        // then the block is (q0 + q1) + (q2 + q3) as in the other paths
        const int64_t rows = min64(kBlockRows, ws.n_rows - b * kBlockRows);
        bool bad = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t by = (state >> (8 * q)) & 0xffu;
            bad |= by != 0 && by != kStateQuarter && by != (kStateEighth0 | kStateEighth1);
        }
        bool missing = bad;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = 2 * lane + k;
            if (r < rows && ((state >> (8 * (r / 16))) & 0xffu) == 0 && ws.leaf_flag[b * kBlockRows + r] == 0)
                missing = true;
        }
        if (__any_sync(kFull, missing) && lane == 0 && blockIdx.y == 0) set_status(ws.hdr, kStMissing);
        if (has_vec) {
            const float *part = ws.block_partial + b * 4 * int64_t(H) + int64_t(v) * 8;
            const float *part2 = ws.eighth + b * 4 * int64_t(H) + int64_t(v) * 8;
            const float *src = ws.spill + b * kBlockRows * int64_t(H) + int64_t(v) * 8;
            float h0[8], acc[8];
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                const uint32_t by = (state >> (8 * q)) & 0xffu;
                float qv[8];
                if (by == kStateQuarter) {
                    load8(part + q * int64_t(H), qv);
                } else if (by == (kStateEighth0 | kStateEighth1)) {
                    load8(part + q * int64_t(H), qv);
                    add_second_eighth(state, q, part2 + q * int64_t(H), qv);
                } else {
                    quarter_from_spill(src, H, q, rows, qv);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if (q == 0 || q == 2) acc[c] = qv[c];
                    else if (q == 1) h0[c] = __fadd_rn(acc[c], qv[c]);
                    else out8[c] = __fadd_rn(h0[c], __fadd_rn(acc[c], qv[c]));
                }
            }
        }
    }
    float pair[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) pair[c] = 2 * w + 1 < m ? __fadd_rn(val[0][c], val[1][c]) : val[0][c];
#pragma unroll
    for (int c = 0; c < 8; ++c) part[w][c][lane] = pair[c];
    if (m == 32) {
        // a full group: the 16 pair results make a complete tree (levels 2-5),
        // formed in registers after one barrier, warp c < 8 taking column c of
        // the CTA's 32 vectors
        __syncthreads();
        if (w < 8 && has_vec) {
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = part[i][w][lane];
#pragma unroll
            for (int n = 8; n >= 1; n >>= 1)
#pragma unroll
                for (int i = 0; i < n; ++i) x[i] = __fadd_rn(x[2 * i], x[2 * i + 1]);
            const float r = scale != 1.f ? __fmul_rn(x[0], scale) : x[0];   // scaled only at the root
            out[g * int64_t(H) + int64_t(v) * 8 + w] = r;
        }
        return;
    }
    // a partial group (the last of a pass): the pair results, level by level:
    // element i of the next level is
    // (2i) + (2i + 1), an odd last element carried up unchanged; warp i forms
    // element i (operands into registers, barrier, store, barrier)
    for (int n = (m + 1) / 2; n > 1; n = (n + 1) / 2) {    // uniform across the CTA
        __syncthreads();
        float a[8];
        const bool act = w < (n + 1) / 2;
        if (act) {
#pragma unroll
            for (int c = 0; c < 8; ++c) a[c] = part[2 * w][c][lane];
            if (2 * w + 1 < n) {
#pragma unroll
                for (int c = 0; c < 8; ++c) a[c] = __fadd_rn(a[c], part[2 * w + 1][c][lane]);
            }
        }
        __syncthreads();
        if (act) {
#pragma unroll
            for (int c = 0; c < 8; ++c) part[w][c][lane] = a[c];
        }
    }
    __syncthreads();
    if (w == 0 && has_vec) {
        float res[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            res[c] = part[0][c][lane];
            if (scale != 1.f) res[c] = __fmul_rn(res[c], scale);   // only on the root of a scaled finalize
        }
        float *dst = out + g * int64_t(H) + int64_t(v) * 8;
        st_global_f32x4(dst, res[0], res[1], res[2], res[3]);
        st_global_f32x4(dst + 4, res[4], res[5], res[6], res[7]);
    }
}

// Carry tree over n partials [n][H] (n <= 2^11), one lane per 8-column
// vector, folded with the binary-counter stack: the top of the dweight tree
// above aligned subtrees whose roots were gathered from several ranks.
__global__ void __launch_bounds__(128) combine_kernel(const float *roots, int64_t n, int H, float scale,
                                                      float *out) {
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= (H >> 3)) return;
    float s[11][8];
    for (int64_t i = 0; i < n; ++i) {
        float x[8];
        load8(roots + i * int64_t(H) + int64_t(v) * 8, x);
        // binary counter: combine with pending partials while the bit of i is set
        int l = 0;
        while ((i >> l) & 1) {
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = __fadd_rn(s[l][c], x[c]);
            ++l;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) s[l][c] = x[c];
    }
    float res[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) res[c] = 0.f;
    bool have = false;
    for (int l = 0; l < 11; ++l) {
        if (!((n >> l) & 1)) continue;
#pragma unroll
        for (int c = 0; c < 8; ++c) res[c] = have ? __fadd_rn(s[l][c], res[c]) : s[l][c];
        have = true;
    }
    if (scale != 1.f) {
#pragma unroll
        for (int c = 0; c < 8; ++c) res[c] = __fmul_rn(res[c], scale);
    }
    st_global_f32x4(out + int64_t(v) * 8, res[0], res[1], res[2], res[3]);
    st_global_f32x4(out + int64_t(v) * 8 + 4, res[4], res[5], res[6], res[7]);
}

__global__ void zero_f32_kernel(float *p, int64_t n) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
        p[i] = 0.f;
}

}  // namespace rbi
