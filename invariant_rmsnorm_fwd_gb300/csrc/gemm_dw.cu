// Deterministic weight gradient of a linear layer (det_gemm dW) over a logical
// token multiset, bitwise identical for every physical layout.
//
// "WS1 C4 (#270) closeout evidence", runtime table and "Historical finding -
// RMSNorm dweight is not chunk/batch decomposable": det_gemm's dW failed the
// chunk and singleton-aggregate checks for the same reason as the norm's
// dweight, an accumulation whose shape follows the rows of each call.  Here
// a call only places its rows: x_g and dy_g of every active token go to row g
// (the canonical logical id) of two logical-order buffers in the workspace.
// The finalize then forms dW = sum_g dy_g^T x_g over all N logical rows,
// dW[o][i] = sum_g DY[g][o] * X[g][i], in FP32 from the bf16 rows, with the
// hand-written tensor-core kernel below: every 256 x 256 tile of dW is owned
// by one pair of CTAs, which walks k = the logical token id upward in slabs
// of 64 tokens and accumulates them in tensor memory in that order.  The
// summation order therefore depends only on (N, I, O), never on how the rows
// arrived.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "host.cuh"
#include "rmsnorm_bi.h"
#include "umma.cuh"

namespace {

constexpr uint32_t kGemmMagic = 0x47445732u;   // "GDW2"

// Tile shape of the contraction: dW rows (o) in tiles of 128, columns (i) in
// tiles of up to 256, tokens (k) in slabs of 64; four slabs in flight.
constexpr int kBM = 128, kBK = 64;                       // rows of a CTA's half tile, tokens per slab
constexpr int kChunk = 64;                               // elements of one 128-byte swizzle row
constexpr int kChunkBytes = kChunk * kBK * 2;            // one TMA box: 64 (o or i) x 64 tokens, 8 KB
constexpr int kGemmThreads = 192;                        // producer, MMA, four epilogue warps

struct GemmWsHeader {
    uint32_t magic;
    int32_t status;
    int64_t n_rows, in_features, out_features;
};

// Logical-order copies of x and dy.  Row pitches are padded (i to a multiple
// of 128, o to a multiple of 256) and the token count to a multiple of 64, so
// every TMA box lies inside its tensor.  Padding rows are zeroed by begin (they
// enter every sum); padding columns are never written and only ever reach
// rows or columns of the product that are not stored.
struct GemmWs {
    GemmWsHeader *hdr;
    int32_t *flag;          // [N] 1 once the row arrived
    uint16_t *x;            // [Np][Ip] bf16
    uint16_t *dy;           // [Np][Op] bf16
    int64_t np, ip, op;
};

int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

bool gemm_sizes_ok(int64_t N, int64_t I, int64_t O) {
    return N >= 0 && N < (int64_t(1) << 31) - 64 && I >= 8 && O >= 8 && I % 8 == 0 && O % 8 == 0 && I <= 65536 &&
           O <= 65536;
}

struct GemmLayout {
    int64_t np, ip, op, off_flag, off_x, off_dy, total;
    GemmLayout(int64_t N, int64_t I, int64_t O) {
        np = align_up(N, kBK);
        ip = align_up(I, 2 * kChunk);                    // a CTA pair splits each tile's columns in two
        op = align_up(O, 2 * kBM);                       // a CTA pair's tile has 256 rows
        off_flag = 256;
        off_x = align_up(off_flag + N * 4, 1024);
        off_dy = align_up(off_x + np * ip * 2, 1024);
        total = align_up(off_dy + np * op * 2, 1024);
    }
};

GemmWs gemm_view(void *ws, int64_t N, int64_t I, int64_t O) {
    const GemmLayout L(N, I, O);
    uint8_t *b = static_cast<uint8_t *>(ws);
    GemmWs v;
    v.hdr = reinterpret_cast<GemmWsHeader *>(b);
    v.flag = reinterpret_cast<int32_t *>(b + L.off_flag);
    v.x = reinterpret_cast<uint16_t *>(b + L.off_x);
    v.dy = reinterpret_cast<uint16_t *>(b + L.off_dy);
    v.np = L.np;
    v.ip = L.ip;
    v.op = L.op;
    return v;
}

__device__ __forceinline__ bool gemm_header_ok(const GemmWs &ws, int64_t N, int64_t I, int64_t O) {
    return ws.hdr->magic == kGemmMagic && ws.hdr->n_rows == N && ws.hdr->in_features == I &&
           ws.hdr->out_features == O;
}

// Clears the flags and the padding token rows [N, Np) of both copies.
__global__ void gemm_begin_kernel(GemmWs ws, int64_t N, int64_t I, int64_t O) {
    const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = tid; i < N; i += nthr) ws.flag[i] = 0;
    const int64_t px = (ws.np - N) * ws.ip / 8, pd = (ws.np - N) * ws.op / 8;   // uint4 units
    uint4 *xz = reinterpret_cast<uint4 *>(ws.x + N * ws.ip);
    uint4 *dz = reinterpret_cast<uint4 *>(ws.dy + N * ws.op);
    for (int64_t i = tid; i < px; i += nthr) xz[i] = make_uint4(0, 0, 0, 0);
    for (int64_t i = tid; i < pd; i += nthr) dz[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        ws.hdr->magic = kGemmMagic;
        ws.hdr->status = 0;
        ws.hdr->n_rows = N;
        ws.hdr->in_features = I;
        ws.hdr->out_features = O;
    }
}

// One warp per token slot: the row's x and dy move to their logical row with
// 16-byte loads and stores; lane 0 sets the row's flag (a flag already set is
// a double contribution).
__global__ void gemm_place_kernel(GemmWs ws, const uint16_t *x, int64_t x_stride, const uint16_t *dy,
                                  int64_t dy_stride, const int32_t *tok_id, int64_t n_tokens, int64_t N, int64_t I,
                                  int64_t O) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    if (!gemm_header_ok(ws, N, I, O)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&ws.hdr->status, RMSNORM_STATUS_HEADER);
        return;
    }
    for (int64_t t = warp; t < n_tokens; t += nwarps) {
        const int32_t g = tok_id[t];
        if (g < 0) continue;                              // padding
        if (g >= N) {
            if (lane == 0) atomicOr(&ws.hdr->status, RMSNORM_STATUS_PLAN);
            continue;
        }
        const uint4 *xs = reinterpret_cast<const uint4 *>(x + t * x_stride);
        uint4 *xd = reinterpret_cast<uint4 *>(ws.x + int64_t(g) * ws.ip);
        for (int64_t v = lane; v < I / 8; v += 32) xd[v] = xs[v];
        const uint4 *ds = reinterpret_cast<const uint4 *>(dy + t * dy_stride);
        uint4 *dd = reinterpret_cast<uint4 *>(ws.dy + int64_t(g) * ws.op);
        for (int64_t v = lane; v < O / 8; v += 32) dd[v] = ds[v];
        if (lane == 0 && atomicExch(&ws.flag[g], 1) != 0) atomicOr(&ws.hdr->status, RMSNORM_STATUS_DOUBLE);
    }
}

__global__ void gemm_check_kernel(GemmWs ws, int64_t N, int64_t I, int64_t O) {
    const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = int64_t(gridDim.x) * blockDim.x;
    if (!gemm_header_ok(ws, N, I, O)) {
        if (tid == 0) atomicOr(&ws.hdr->status, RMSNORM_STATUS_HEADER);
        return;
    }
    bool missing = false;
    for (int64_t i = tid; i < N; i += nthr) missing |= ws.flag[i] == 0;
    if (__any_sync(0xffffffffu, missing) && (threadIdx.x & 31) == 0) atomicOr(&ws.hdr->status, RMSNORM_STATUS_MISSING);
}

__global__ void gemm_zero_kernel(float *p, int64_t n) {
    const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = tid; i < n; i += nthr) p[i] = 0.f;
}

// ---------------------------------------------------------------- the contraction

struct GemmParams {
    float *dw;                 // [O][I] row-major
    int32_t *status;           // workspace status word
    int32_t O, I;
    int32_t ip;                // padded i extent (multiple of 128)
    int32_t m_tiles, n_tiles, k_slabs;
    float scale;
};

// dW = scale * DY^T X on the tensor cores.  A = DY^T (o x k) and B = X (k x i)
// are both read MN-major straight from the logical-order copies: a TMA box is
// 64 tokens (k) by 64 consecutive o (or i), stored with the 128-byte swizzle,
// which is the canonical MN-major operand layout of the MMA.  Persistent CTA
// pairs take the tiles t = pair, pair + pairs, ... with o-tile t % m_tiles;
// each tile walks the token slabs in ascending order and its first MMA
// overwrites the accumulator, so every element's summation order depends on
// (N, I, O) only.
// ---------------------------------------------------------------- the contraction on CTA pairs
//
// The same product with 256 x 256 tiles of dW per pair of CTAs (a 2-CTA
// cluster on two SMs): CTA r holds rows [128 r, 128 r + 128) of the tile's A
// and columns [r N/2, (r + 1) N/2) of its B, and one K = 16 MMA of the pair
// (tcgen05.mma.cta_group::2, M = 256) reads both halves of both operands, so
// each CTA's shared memory carries half of B instead of all of it.  Each
// CTA's tensor memory receives its 128 rows of the tile.
// Roles (per CTA, both ranks unless noted):
//   warp 0, lane 0: producer: the CTA's A and B boxes of each slab into its
//                   own ring.  Both producers arrive on rank 0's full[s]
//                   (count 2) with the bytes they expect; rank 1's copies
//                   count their bytes there too (cta_group::2 copies);
//   warp 1, lane 0, rank 0: MMA issuer: waits for full[s], four pair MMAs,
//                   then one commit that arrives on empty[s] of both CTAs;
//                   after a tile's last slab, on acc_full[a] of both;
//   warps 2-5:      epilogue of the CTA's 128 rows; each warp then arrives on
//                   rank 0's acc_empty[a] (count 8), which the MMA issuer
//                   waits for before it overwrites that accumulator (two of
//                   256 columns, so one tile's epilogue overlaps the next).
// Every wait is bounded.  At the end rank 1's producer tells rank 0 how many
// slabs it issued; rank 0's producer makes the arrivals that either side did
// not make for the last slabs and waits for those phases, so no copy of
// either CTA is in flight when the pair meets at the final cluster barrier
// and frees its tensor memory.
constexpr int kPairStages = 7;
constexpr int kPairABytes = kBM * kBK * 2;               // 16 KB: this CTA's 128 rows of A
constexpr int kPairBBytes = kBM * kBK * 2;               // 16 KB: this CTA's half (<= 128 columns) of B
constexpr int kPairStageBytes = kPairABytes + kPairBBytes;
constexpr int kPairSmem = kPairStages * kPairStageBytes + 1024;
constexpr uint32_t kPairTmemCols = 512;                  // two 256-column accumulators per CTA

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_dw_pair_kernel(const __grid_constant__ CUtensorMap tmap_dy, const __grid_constant__ CUtensorMap tmap_x,
                        const GemmParams p) {
    using namespace rbi;
    extern __shared__ uint8_t gemm_smem[];
    __shared__ uint64_t full[kPairStages], empty[kPairStages], acc_full[2], acc_empty[2], mma_done, peer_done;
    __shared__ uint32_t tmem_slot;
    __shared__ uint32_t peer_issued;                      // rank 0: slabs rank 1 issued (written by rank 1)
    __shared__ volatile int32_t abort_flag;
    uint8_t *tiles = gemm_smem + ((1024u - (smem_addr(gemm_smem) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = int(blockIdx.x >> 1), n_pairs = int(gridDim.x >> 1);
    const int total = p.m_tiles * p.n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&full[s], 2);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 8);
        }
        mbar_init(&mma_done, 1);
        mbar_init(&peer_done, 1);
        peer_issued = 0;
        abort_flag = 0;
        fence_mbar_init();
    }
    cluster_barrier();                                    // both CTAs' barriers exist before any remote arrival
    if (warp == 1) {
        umma::tmem_alloc_pair(&tmem_slot, kPairTmemCols);
        umma::tmem_relinquish_pair();
    }
    umma::fence_before();
    cluster_barrier();
    umma::fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t leader_full = map_to_rank(smem_addr(&full[0]), 0);
    const uint32_t leader_acc_empty = map_to_rank(smem_addr(&acc_empty[0]), 0);

    auto give_up = [&]() {
        abort_flag = 1;
        atomicOr(p.status, RMSNORM_STATUS_TIMEOUT);
    };

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ producer (both CTAs)
        int g = 0;
        for (int t = pair; t < total && !abort_flag; t += n_pairs) {
            const int mt = t % p.m_tiles, nt = t / p.m_tiles;
            const int n0 = nt * 2 * kBM;
            const int half = min(2 * kBM, p.ip - n0) / 2;          // this CTA's columns: 64 or 128
            const int nb = half / kChunk;
            const int m0 = mt * 2 * kBM + int(rank) * kBM;
            const int c0 = n0 + int(rank) * half;
            const uint32_t bytes = uint32_t(kPairABytes + nb * kChunkBytes);
            bool ok = true;
            for (int kb = 0; kb < p.k_slabs; ++kb) {
                const int s = g % kPairStages, u = g / kPairStages;
                if (u > 0 && !mbar_wait_spin_bounded(&empty[s], uint32_t(u - 1) & 1u)) {
                    give_up();
                    ok = false;
                    break;
                }
                if (abort_flag) {
                    ok = false;
                    break;
                }
                uint8_t *a = tiles + s * kPairStageBytes;
                uint8_t *b = a + kPairABytes;
                if (rank == 0) {
                    mbar_arrive_expect_tx(&full[s], bytes);
                    umma::tma_load_2d(a, &tmap_dy, m0, kb * kBK, &full[s]);
                    umma::tma_load_2d(a + kChunkBytes, &tmap_dy, m0 + kChunk, kb * kBK, &full[s]);
                    for (int j = 0; j < nb; ++j)
                        umma::tma_load_2d(b + j * kChunkBytes, &tmap_x, c0 + j * kChunk, kb * kBK, &full[s]);
                } else {
                    const uint32_t fb = leader_full + uint32_t(s) * 8u;
                    mbar_arrive_expect_tx_remote(fb, bytes);
                    umma::tma_load_2d_to_peer_bar(a, &tmap_dy, m0, kb * kBK, fb);
                    umma::tma_load_2d_to_peer_bar(a + kChunkBytes, &tmap_dy, m0 + kChunk, kb * kBK, fb);
                    for (int j = 0; j < nb; ++j)
                        umma::tma_load_2d_to_peer_bar(b + j * kChunkBytes, &tmap_x, c0 + j * kChunk, kb * kBK, fb);
                }
                ++g;
            }
            if (!ok) break;
        }
        if (rank == 1) {
            // tell rank 0 how many slabs this CTA issued
            st_cluster_u32(map_to_rank(smem_addr(&peer_issued), 0), uint32_t(g));
            mbar_arrive_remote(map_to_rank(smem_addr(&peer_done), 0));
        } else {
            // the last slabs of either CTA: make the arrivals the other side did
            // not make, then wait until every copy of those phases has landed
            int gp = g;
            // rank 1 may itself be in a wait that runs out: allow it two limits
            if (mbar_wait_bounded_cluster(&peer_done, 0) || mbar_wait_bounded_cluster(&peer_done, 0))
                gp = int(peer_issued);
            const int hi = g > gp ? g : gp;
            for (int i = hi - 1; i >= 0 && i >= hi - kPairStages; --i) {
                const int s = i % kPairStages;
                if (i >= g) mbar_arrive(&full[s]);          // rank 0 never armed this phase
                if (i >= gp) mbar_arrive(&full[s]);         // rank 1 never armed it
                mbar_wait_bounded_cluster(&full[s], uint32_t(i / kPairStages) & 1u);
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------ rank 0: MMA issuer for the pair
        int g = 0, it = 0;
        for (int t = pair; t < total && !abort_flag; t += n_pairs, ++it) {
            const int nt = t / p.m_tiles;
            const int bn = min(2 * kBM, p.ip - nt * 2 * kBM);
            const int acc = it & 1, ua = it >> 1;
            if (ua > 0 && !mbar_wait_spin_bounded_cluster(&acc_empty[acc], uint32_t(ua - 1) & 1u)) {
                give_up();
                break;
            }
            umma::fence_after();
            const uint32_t d = tmem + uint32_t(acc * 2 * kBM);
            const uint32_t idesc = umma::idesc_bf16_mn(2 * kBM, uint32_t(bn));
            bool ok = true;
            for (int kb = 0; kb < p.k_slabs; ++kb, ++g) {
                const int s = g % kPairStages, u = g / kPairStages;
                if (!mbar_wait_spin_bounded(&full[s], uint32_t(u) & 1u)) {
                    give_up();
                    ok = false;
                    break;
                }
                if (abort_flag) {
                    ok = false;
                    break;
                }
                umma::fence_after();
                const uint32_t a = smem_addr(tiles + s * kPairStageBytes);
                const uint32_t b = a + kPairABytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = umma::desc_sw128(a + kk * 2048, kChunkBytes, 1024);
                    const uint64_t bd = umma::desc_sw128(b + kk * 2048, kChunkBytes, 1024);
                    umma::mma_bf16_pair(d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                }
                umma::commit_pair_multicast(&empty[s], 3);   // the stage is free in both CTAs
            }
            if (!ok) break;
            umma::commit_pair_multicast(&acc_full[acc], 3); // the tile is complete in both CTAs
        }
        umma::commit_pair_multicast(&mma_done, 1);
        mbar_wait_bounded(&mma_done, 0);                      // no MMA in flight past this point
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue (both CTAs): this CTA's 128 rows
        const int q = warp & 3;
        int it = 0;
        for (int t = pair; t < total; t += n_pairs, ++it) {
            const int mt = t % p.m_tiles, nt = t / p.m_tiles;
            const int n0 = nt * 2 * kBM;
            const int bn = min(2 * kBM, p.ip - n0);
            const int acc = it & 1, ua = it >> 1;
            bool done = mbar_wait_bounded(&acc_full[acc], uint32_t(ua) & 1u);
            done = __all_sync(kFull, done);
            if (!done) {
                if (lane == 0) give_up();
                break;
            }
            umma::fence_after();
            const int64_t m = int64_t(mt) * 2 * kBM + int64_t(rank) * kBM + q * 32 + lane;
            float *row = p.dw + m * p.I;
            for (int c = 0; c < bn; c += 32) {
                uint32_t v[32];
                __syncwarp();
                umma::ld_32x32(tmem + (uint32_t(q * 32) << 16) + uint32_t(acc * 2 * kBM + c), v);
                umma::wait_ld();
                if (m < p.O) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const int col = n0 + c + j;
                        if (col < p.I) {
                            float f[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                f[e] = __uint_as_float(v[j + e]);
                                if (p.scale != 1.f) f[e] = __fmul_rn(f[e], p.scale);
                            }
                            st_global_f32x4(row + col, f[0], f[1], f[2], f[3]);
                        }
                    }
                }
            }
            umma::fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive(&acc_empty[acc]);
                else mbar_arrive_remote(leader_acc_empty + uint32_t(acc) * 8u);
            }
        }
    }
    __syncwarp();
    umma::fence_before();
    cluster_barrier();                                    // no remote arrival, copy or MMA targets an exited CTA
    if (warp == 1) {
        __syncwarp();
        umma::fence_after();
        umma::tmem_dealloc_pair(tmem, kPairTmemCols);
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int tensor_map_2d(CUtensorMap *map, void *base, int64_t inner, int64_t outer) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return RMSNORM_ERR_CUDA;
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    const cuuint64_t strides[1] = {cuuint64_t(inner) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kChunk), cuuint32_t(kBK)};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int grid_for(int64_t work, int threads, const rbi::DeviceInfo &d) {
    int64_t b = (work + threads - 1) / threads;
    const int64_t cap = int64_t(d.sms) * 8;
    if (b > cap) b = cap;
    return int(b < 1 ? 1 : b);
}

}  // namespace

extern "C" size_t gemm_dw_workspace_bytes(int64_t n_logical_rows, int64_t in_features, int64_t out_features) {
    if (!gemm_sizes_ok(n_logical_rows, in_features, out_features)) return 0;
    return size_t(GemmLayout(n_logical_rows, in_features, out_features).total);
}

extern "C" int gemm_dw_begin(void *workspace, size_t bytes, int64_t n_logical_rows, int64_t in_features,
                             int64_t out_features, rmsnorm_stream_t stream) {
    if (!workspace) return RMSNORM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RMSNORM_ERR_ALIGN;
    if (!gemm_sizes_ok(n_logical_rows, in_features, out_features)) return RMSNORM_ERR_HIDDEN;
    if (bytes < gemm_dw_workspace_bytes(n_logical_rows, in_features, out_features)) return RMSNORM_ERR_WORKSPACE;
    rbi::DeviceInfo *d = nullptr;
    int rc = rbi::device_info(&d);
    if (rc) return rc;
    GemmWs ws = gemm_view(workspace, n_logical_rows, in_features, out_features);
    const int64_t work = n_logical_rows + (ws.np - n_logical_rows) * (ws.ip + ws.op) / 8;
    gemm_begin_kernel<<<grid_for(work, 256, *d), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        ws, n_logical_rows, in_features, out_features);
    if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
    rbi::count_launch();
    return RMSNORM_OK;
}

extern "C" int gemm_dw_contrib(const uint16_t *x, int64_t x_stride, const uint16_t *dy, int64_t dy_stride,
                               int64_t in_features, int64_t out_features, const rmsnorm_layout_t *layout,
                               void *workspace, rmsnorm_stream_t stream) {
    if (!layout || !workspace) return RMSNORM_ERR_NULL;
    if (!gemm_sizes_ok(layout->n_logical_tokens, in_features, out_features)) return RMSNORM_ERR_HIDDEN;
    if (layout->n_tokens < 0 || layout->rows_per_token != 1 || layout->reserved0 != 0) return RMSNORM_ERR_LAYOUT;
    if (layout->n_tokens == 0) return RMSNORM_OK;
    if (!x || !dy || !layout->tok_id) return RMSNORM_ERR_NULL;
    if (x_stride < in_features || dy_stride < out_features) return RMSNORM_ERR_STRIDE;
    if (!aligned16(x) || !aligned16(dy) || x_stride % 8 != 0 || dy_stride % 8 != 0 ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return RMSNORM_ERR_ALIGN;
    rbi::DeviceInfo *d = nullptr;
    int rc = rbi::device_info(&d);
    if (rc) return rc;
    const int64_t N = layout->n_logical_tokens;
    GemmWs ws = gemm_view(workspace, N, in_features, out_features);
    const int threads = 256;
    gemm_place_kernel<<<grid_for(layout->n_tokens * 32, threads, *d), threads, 0,
                        reinterpret_cast<cudaStream_t>(stream)>>>(ws, x, x_stride, dy, dy_stride, layout->tok_id,
                                                                  layout->n_tokens, N, in_features, out_features);
    if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
    rbi::count_launch();
    return RMSNORM_OK;
}

extern "C" int gemm_dw_finalize(void *workspace, int64_t n_logical_rows, int64_t in_features, int64_t out_features,
                                float grad_scale, float *dw, rmsnorm_stream_t stream) {
    if (!workspace || !dw) return RMSNORM_ERR_NULL;
    if (!std::isfinite(grad_scale)) return RMSNORM_ERR_VALUE;
    if (!gemm_sizes_ok(n_logical_rows, in_features, out_features)) return RMSNORM_ERR_HIDDEN;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || !aligned16(dw)) return RMSNORM_ERR_ALIGN;
    rbi::DeviceInfo *d = nullptr;
    int rc = rbi::device_info(&d);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t N = n_logical_rows, I = in_features, O = out_features;
    GemmWs ws = gemm_view(workspace, N, I, O);
    gemm_check_kernel<<<grid_for(N, 256, *d), 256, 0, s>>>(ws, N, I, O);
    if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
    rbi::count_launch();
    if (N == 0) {
        gemm_zero_kernel<<<grid_for(I * O, 256, *d), 256, 0, s>>>(dw, I * O);
        if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
        rbi::count_launch();
        return RMSNORM_OK;
    }
    CUtensorMap tm_dy, tm_x;
    if ((rc = tensor_map_2d(&tm_dy, ws.dy, ws.op, ws.np)) || (rc = tensor_map_2d(&tm_x, ws.x, ws.ip, ws.np)))
        return rc;
    GemmParams gp;
    gp.dw = dw;
    gp.status = &ws.hdr->status;
    gp.O = int32_t(O);
    gp.I = int32_t(I);
    gp.ip = int32_t(ws.ip);
    gp.k_slabs = int32_t(ws.np / kBK);
    gp.scale = grad_scale;
    gp.m_tiles = int32_t(ws.op / (2 * kBM));
    gp.n_tiles = int32_t((ws.ip + 2 * kBM - 1) / (2 * kBM));
    static std::once_flag attr_once;
    static cudaError_t attr_rc = cudaSuccess;
    static int max_pairs = 0;
    std::call_once(attr_once, [] {
        attr_rc = cudaFuncSetAttribute(gemm_dw_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
        if (attr_rc != cudaSuccess) return;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kGemmThreads);
        cfg.dynamicSmemBytes = kPairSmem;
        attr_rc = cudaOccupancyMaxActiveClusters(&max_pairs, gemm_dw_pair_kernel, &cfg);
    });
    if (attr_rc != cudaSuccess || max_pairs < 1) return RMSNORM_ERR_CUDA;
    const int64_t tiles = int64_t(gp.m_tiles) * gp.n_tiles;   // persistent pairs, one per SM pair
    const int pairs = int(tiles < max_pairs ? tiles : max_pairs);
    gemm_dw_pair_kernel<<<2 * pairs, kGemmThreads, kPairSmem, s>>>(tm_dy, tm_x, gp);
    if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
    rbi::count_launch();
    return RMSNORM_OK;
}

extern "C" int gemm_dw_status(const void *workspace, rmsnorm_stream_t stream, int32_t *status) {
    if (!workspace || !status) return RMSNORM_ERR_NULL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const GemmWsHeader *h = static_cast<const GemmWsHeader *>(workspace);
    if (cudaMemcpyAsync(status, &h->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}
