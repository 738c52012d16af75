// Deterministic weight gradient of a linear layer (det_gemm dW) over a logical
// token multiset, bitwise identical for every physical layout.
//
// "WS1 C4 (#270) closeout evidence", runtime table and "Historical finding -
// RMSNorm dweight is not chunk/batch decomposable": det_gemm's dW failed the
// chunk and singleton-aggregate checks for the same reason as the norm's
// dweight, an accumulation whose shape follows the rows of each call.  Here
// a call only places its rows: x_g and dy_g of every active token go to row g
// (the canonical logical id) of two logical-order buffers in the workspace.
// The finalize then forms dW = sum_g dy_g^T x_g as one GEMM over all N logical
// rows, dW[o][i] = sum_g DY[g][o] * X[g][i], in FP32 from the bf16 rows.  Its
// summation order is the GEMM's and depends only on (N, I, O), never on how
// the rows arrived.  The contraction is a plain library GEMM (cuBLAS, FP32
// compute, no atomics); the placement, the contribution flags and the checks
// are kernels of this file.
#include <cublas_v2.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "host.cuh"
#include "rmsnorm_bi.h"

namespace {

constexpr uint32_t kGemmMagic = 0x47445731u;   // "GDW1"

struct GemmWsHeader {
    uint32_t magic;
    int32_t status;
    int64_t n_rows, in_features, out_features;
};

struct GemmWs {
    GemmWsHeader *hdr;
    int32_t *flag;          // [N] 1 once the row arrived
    uint16_t *x;            // [N][I] bf16, logical order
    uint16_t *dy;           // [N][O] bf16, logical order
};

int64_t align256(int64_t v) { return (v + 255) / 256 * 256; }

bool gemm_sizes_ok(int64_t N, int64_t I, int64_t O) {
    return N >= 0 && N < (int64_t(1) << 31) && I >= 8 && O >= 8 && I % 8 == 0 && O % 8 == 0 && I <= 65536 &&
           O <= 65536;
}

int64_t gemm_ws_bytes(int64_t N, int64_t I, int64_t O) {
    return 256 + align256(N * 4) + align256(N * I * 2) + align256(N * O * 2);
}

GemmWs gemm_view(void *ws, int64_t N, int64_t I) {
    uint8_t *b = static_cast<uint8_t *>(ws);
    GemmWs v;
    v.hdr = reinterpret_cast<GemmWsHeader *>(b);
    v.flag = reinterpret_cast<int32_t *>(b + 256);
    v.x = reinterpret_cast<uint16_t *>(b + 256 + align256(N * 4));
    v.dy = reinterpret_cast<uint16_t *>(b + 256 + align256(N * 4) + align256(N * I * 2));
    return v;
}

__global__ void gemm_begin_kernel(GemmWs ws, int64_t N, int64_t I, int64_t O) {
    const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = tid; i < N; i += nthr) ws.flag[i] = 0;
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
    const bool header_ok = ws.hdr->magic == kGemmMagic && ws.hdr->n_rows == N && ws.hdr->in_features == I &&
                           ws.hdr->out_features == O;
    if (!header_ok) {
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
        uint4 *xd = reinterpret_cast<uint4 *>(ws.x + int64_t(g) * I);
        for (int64_t v = lane; v < I / 8; v += 32) xd[v] = xs[v];
        const uint4 *ds = reinterpret_cast<const uint4 *>(dy + t * dy_stride);
        uint4 *dd = reinterpret_cast<uint4 *>(ws.dy + int64_t(g) * O);
        for (int64_t v = lane; v < O / 8; v += 32) dd[v] = ds[v];
        if (lane == 0 && atomicExch(&ws.flag[g], 1) != 0) atomicOr(&ws.hdr->status, RMSNORM_STATUS_DOUBLE);
    }
}

__global__ void gemm_check_kernel(GemmWs ws, int64_t N, int64_t I, int64_t O) {
    const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = int64_t(gridDim.x) * blockDim.x;
    const bool header_ok = ws.hdr->magic == kGemmMagic && ws.hdr->n_rows == N && ws.hdr->in_features == I &&
                           ws.hdr->out_features == O;
    if (!header_ok) {
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

// One cuBLAS handle per device, created on first use; calls are serialised
// by the mutex (the handle's stream is set per call).
std::mutex g_blas_mu;
cublasHandle_t g_blas[64] = {nullptr};

int blas_handle(cublasHandle_t *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RMSNORM_ERR_CUDA;
    if (g_blas[dev] == nullptr) {
        if (cublasCreate(&g_blas[dev]) != CUBLAS_STATUS_SUCCESS) return RMSNORM_ERR_CUDA;
        // atomics stay off (the default): every reduction order is fixed by the shapes
        if (cublasSetAtomicsMode(g_blas[dev], CUBLAS_ATOMICS_NOT_ALLOWED) != CUBLAS_STATUS_SUCCESS)
            return RMSNORM_ERR_CUDA;
        if (cublasSetMathMode(g_blas[dev], CUBLAS_DEFAULT_MATH) != CUBLAS_STATUS_SUCCESS) return RMSNORM_ERR_CUDA;
    }
    *out = g_blas[dev];
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
    return size_t(gemm_ws_bytes(n_logical_rows, in_features, out_features));
}

extern "C" int gemm_dw_begin(void *workspace, size_t bytes, int64_t n_logical_rows, int64_t in_features,
                             int64_t out_features, rmsnorm_stream_t stream) {
    if (!workspace) return RMSNORM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RMSNORM_ERR_ALIGN;
    if (!gemm_sizes_ok(n_logical_rows, in_features, out_features)) return RMSNORM_ERR_HIDDEN;
    if (bytes < size_t(gemm_ws_bytes(n_logical_rows, in_features, out_features))) return RMSNORM_ERR_WORKSPACE;
    rbi::DeviceInfo *d = nullptr;
    int rc = rbi::device_info(&d);
    if (rc) return rc;
    GemmWs ws = gemm_view(workspace, n_logical_rows, in_features);
    gemm_begin_kernel<<<grid_for(n_logical_rows, 256, *d), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
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
    GemmWs ws = gemm_view(workspace, N, in_features);
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
    GemmWs ws = gemm_view(workspace, N, I);
    gemm_check_kernel<<<grid_for(N, 256, *d), 256, 0, s>>>(ws, N, I, O);
    if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
    rbi::count_launch();
    if (N == 0) {
        gemm_zero_kernel<<<grid_for(I * O, 256, *d), 256, 0, s>>>(dw, I * O);
        if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
        rbi::count_launch();
        return RMSNORM_OK;
    }
    std::lock_guard<std::mutex> lk(g_blas_mu);
    cublasHandle_t h = nullptr;
    if ((rc = blas_handle(&h))) return rc;
    if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return RMSNORM_ERR_CUDA;
    // column-major view: X is I x N (ld I), DY is O x N (ld O), dW (row-major
    // [O][I]) is I x O (ld I):  dW = X * DY^T, k = N in logical order
    const float alpha = grad_scale, beta = 0.f;
    if (cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_T, int(I), int(O), int(N), &alpha, ws.x, CUDA_R_16BF, int(I), ws.dy,
                     CUDA_R_16BF, int(O), &beta, dw, CUDA_R_32F, int(I), CUBLAS_COMPUTE_32F,
                     CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
        return RMSNORM_ERR_CUDA;
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
