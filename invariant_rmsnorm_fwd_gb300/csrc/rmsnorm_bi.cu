// C-ABI entry points of the batch-invariant RMSNorm library (sm_103a).
//
// Launch shapes depend on the hidden size and the device's SM count only;
// which CTA handles which row never changes a value (see rmsnorm_kernels.cuh),
// so results are identical for every layout and every grid.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "finalize_kernels.cuh"
#include "host.cuh"
#include "rmsnorm_bi.h"

using namespace rbi;

namespace {

std::atomic<int64_t> g_launches{0};
std::mutex g_mu;
DeviceInfo g_dev[64];

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_layout(const rmsnorm_layout_t *L, int64_t H) {
    if (!L) return RMSNORM_ERR_NULL;
    if (L->n_tokens < 0 || L->rows_per_token < 1 || L->reserved0 != 0 || L->n_logical_tokens < 0 ||
        L->plan_items < 0)
        return RMSNORM_ERR_LAYOUT;
    if (L->n_tokens > 0 && !L->tok_id) return RMSNORM_ERR_NULL;
    if (L->token_stride % 8 != 0) return RMSNORM_ERR_ALIGN;
    if (L->token_stride < int64_t(L->rows_per_token) * H) return RMSNORM_ERR_STRIDE;
    const int64_t rows = L->n_tokens * L->rows_per_token;
    if (rows >= (int64_t(1) << 31) || L->n_logical_tokens * L->rows_per_token >= (int64_t(1) << 31))
        return RMSNORM_ERR_LAYOUT;
    return RMSNORM_OK;
}

KParams base_params(const rmsnorm_layout_t *L, int64_t H, float eps) {
    KParams p = {};
    p.tok_id = L->tok_id;
    p.n_rows = L->n_tokens * L->rows_per_token;
    p.token_stride = L->token_stride;
    p.rpt = L->rows_per_token;
    p.rpt_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((int64_t(1) << sh) == int64_t(p.rpt)) p.rpt_shift = sh;
    p.hidden = int32_t(H);
    p.eps = eps;
    p.grad_scale = 1.f;
    p.items = static_cast<const PlanItem *>(L->plan);
    p.use_plan = L->plan != nullptr ? 1 : 0;
    return p;
}

int ws_checks(const void *ws, int64_t N, int64_t H) {
    if (!ws) return RMSNORM_ERR_NULL;
    if (!aligned16(ws) || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return RMSNORM_ERR_ALIGN;
    if (N < 0) return RMSNORM_ERR_LAYOUT;
    Shape sh;
    if (!hidden_shape(H, &sh)) return RMSNORM_ERR_HIDDEN;
    return RMSNORM_OK;
}

}  // namespace

namespace rbi {

int device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RMSNORM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
        d.status = (major == 10 && minor == 3) ? RMSNORM_OK : RMSNORM_ERR_DEVICE;
        d.ready = true;
    }
    *out = &d;
    return d.status;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace rbi

// ==================================================================== C ABI

extern "C" int rmsnorm_fwd(const uint16_t *x, const uint16_t *weight, int64_t hidden, float eps,
                           const rmsnorm_layout_t *layout, uint16_t *y, float *rstd, rmsnorm_stream_t stream) {
    Shape sh;
    if (!hidden_shape(hidden, &sh)) return RMSNORM_ERR_HIDDEN;
    int rc = check_layout(layout, hidden);
    if (rc) return rc;
    if (layout->n_tokens == 0) return RMSNORM_OK;
    if (!x || !weight || !y) return RMSNORM_ERR_NULL;
    if (!aligned16(x) || !aligned16(weight) || !aligned16(y)) return RMSNORM_ERR_ALIGN;
    KParams p = base_params(layout, hidden, eps);
    p.x = x;
    p.w = weight;
    p.out = y;
    p.rstd_out = rstd;
    return run_rows<kFwd>(p, sh, layout, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int rmsnorm_bwd_dx(const uint16_t *x, const uint16_t *weight, const uint16_t *dy, int64_t hidden,
                              float eps, const rmsnorm_layout_t *layout, uint16_t *dx, void *workspace,
                              rmsnorm_stream_t stream) {
    Shape sh;
    if (!hidden_shape(hidden, &sh)) return RMSNORM_ERR_HIDDEN;
    int rc = check_layout(layout, hidden);
    if (rc) return rc;
    if (!workspace && !dx) return RMSNORM_ERR_NULL;
    if (workspace && !layout->plan && layout->n_tokens > 0) return RMSNORM_ERR_PLAN;
    const int64_t N = layout->n_logical_tokens * layout->rows_per_token;
    if (workspace && (rc = ws_checks(workspace, N, hidden))) return rc;
    if (layout->n_tokens == 0) return RMSNORM_OK;
    if (!x || !weight || !dy) return RMSNORM_ERR_NULL;
    if (!aligned16(x) || !aligned16(weight) || !aligned16(dy) || (dx && !aligned16(dx))) return RMSNORM_ERR_ALIGN;
    KParams p = base_params(layout, hidden, eps);
    p.x = x;
    p.w = weight;
    p.dy = dy;
    p.out = dx;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!workspace) return run_rows<kDx>(p, sh, layout, s);
    p.ws = ws_view(workspace, N, hidden);
    return run_rows<kDxDw>(p, sh, layout, s);
}

extern "C" int rmsnorm_add_fwd(const uint16_t *x, const uint16_t *residual, const uint16_t *weight,
                               int64_t hidden, float eps, const rmsnorm_layout_t *layout, uint16_t *h_out,
                               uint16_t *y, float *rstd, rmsnorm_stream_t stream) {
    Shape sh;
    if (!hidden_shape(hidden, &sh)) return RMSNORM_ERR_HIDDEN;
    int rc = check_layout(layout, hidden);
    if (rc) return rc;
    if (layout->n_tokens == 0) return RMSNORM_OK;
    if (!x || !residual || !weight || !h_out || !y) return RMSNORM_ERR_NULL;
    if (h_out == y) return RMSNORM_ERR_LAYOUT;
    if (!aligned16(x) || !aligned16(residual) || !aligned16(weight) || !aligned16(h_out) || !aligned16(y))
        return RMSNORM_ERR_ALIGN;
    KParams p = base_params(layout, hidden, eps);
    p.x = x;
    p.res = residual;
    p.w = weight;
    p.out = y;
    p.out2 = h_out;
    p.rstd_out = rstd;
    return run_rows<kAddFwd>(p, sh, layout, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int rmsnorm_add_bwd(const uint16_t *x, const uint16_t *weight, const uint16_t *dy, const uint16_t *dres,
                               int64_t hidden, float eps, float grad_scale, const rmsnorm_layout_t *layout,
                               uint16_t *dx, void *workspace, rmsnorm_stream_t stream) {
    Shape sh;
    if (!hidden_shape(hidden, &sh)) return RMSNORM_ERR_HIDDEN;
    int rc = check_layout(layout, hidden);
    if (rc) return rc;
    if (!std::isfinite(grad_scale)) return RMSNORM_ERR_VALUE;
    if (!workspace && !dx) return RMSNORM_ERR_NULL;
    if (dres && !dx) return RMSNORM_ERR_NULL;
    if (workspace && !layout->plan && layout->n_tokens > 0) return RMSNORM_ERR_PLAN;
    const int64_t N = layout->n_logical_tokens * layout->rows_per_token;
    if (workspace && (rc = ws_checks(workspace, N, hidden))) return rc;
    if (layout->n_tokens == 0) return RMSNORM_OK;
    if (!x || !weight || !dy) return RMSNORM_ERR_NULL;
    if (!aligned16(x) || !aligned16(weight) || !aligned16(dy) || (dx && !aligned16(dx)) || (dres && !aligned16(dres)))
        return RMSNORM_ERR_ALIGN;
    KParams p = base_params(layout, hidden, eps);
    p.x = x;
    p.w = weight;
    p.dy = dy;
    p.res = dres;
    p.out = dx;
    p.grad_scale = grad_scale;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (workspace) p.ws = ws_view(workspace, N, hidden);
    if (dres) return workspace ? run_rows<kAddDxDw>(p, sh, layout, s) : run_rows<kAddDx>(p, sh, layout, s);
    return workspace ? run_rows<kDxDw>(p, sh, layout, s) : run_rows<kDx>(p, sh, layout, s);
}

extern "C" int rmsnorm_bwd_dweight_contrib(const uint16_t *x, const uint16_t *dy, int64_t hidden, float eps,
                                           const rmsnorm_layout_t *layout, void *workspace,
                                           rmsnorm_stream_t stream) {
    Shape sh;
    if (!hidden_shape(hidden, &sh)) return RMSNORM_ERR_HIDDEN;
    int rc = check_layout(layout, hidden);
    if (rc) return rc;
    const int64_t N = layout->n_logical_tokens * layout->rows_per_token;
    if ((rc = ws_checks(workspace, N, hidden))) return rc;
    if (layout->n_tokens == 0) return RMSNORM_OK;
    if (!layout->plan) return RMSNORM_ERR_PLAN;
    if (!x || !dy) return RMSNORM_ERR_NULL;
    if (!aligned16(x) || !aligned16(dy)) return RMSNORM_ERR_ALIGN;
    KParams p = base_params(layout, hidden, eps);
    p.x = x;
    p.dy = dy;
    p.ws = ws_view(workspace, N, hidden);
    return run_rows<kDw>(p, sh, layout, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t rmsnorm_dweight_workspace_bytes(int64_t n_logical_rows, int64_t hidden) {
    Shape sh;
    if (n_logical_rows < 0 || n_logical_rows >= (int64_t(1) << 31) || !hidden_shape(hidden, &sh)) return 0;
    return size_t(WsLayout(n_logical_rows, hidden).total);
}

extern "C" int rmsnorm_dweight_begin(void *workspace, size_t bytes, int64_t n_logical_rows, int64_t hidden,
                                     rmsnorm_stream_t stream) {
    int rc = ws_checks(workspace, n_logical_rows, hidden);
    if (rc) return rc;
    const size_t need = rmsnorm_dweight_workspace_bytes(n_logical_rows, hidden);
    if (need == 0) return RMSNORM_ERR_LAYOUT;
    if (bytes < need) return RMSNORM_ERR_WORKSPACE;
    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    WsView ws = ws_view(workspace, n_logical_rows, hidden);
    const int64_t flag_bytes = reinterpret_cast<uint8_t *>(ws.block_partial) - ws.block_state;
    int64_t blocks = (flag_bytes / 16 + 255) / 256;
    if (blocks > int64_t(d->sms) * 4) blocks = int64_t(d->sms) * 4;
    if (blocks < 1) blocks = 1;
    ws_begin_kernel<<<unsigned(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ws);
    if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return RMSNORM_OK;
}

namespace {
// Tree passes over blocks [lo, lo + count) of the workspace, leaving one value in out.
int finalize_blocks(const WsView &ws, int64_t lo, int64_t count, float *out, float scale, cudaStream_t s) {
    const int V = int(ws.hidden / 8);
    const unsigned gy = unsigned((V + kTreeVecs - 1) / kTreeVecs);
    int64_t n = count;
    const float *in = nullptr;
    bool first = true;
    int flip = 0;
    while (true) {
        const int64_t groups = (n + 31) / 32;
        float *dst = groups == 1 ? out : (flip ? ws.scratch_b : ws.scratch_a);
        tree_pass_kernel<<<dim3(unsigned(groups), gy), kTreeWarps * 32, 0, s>>>(
            ws, in, dst, n, first ? 1 : 0, first ? lo : 0, groups == 1 ? scale : 1.f);
        if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (groups == 1) break;
        in = dst;
        n = groups;
        first = false;
        flip ^= 1;
    }
    return RMSNORM_OK;
}
}  // namespace

extern "C" int dweight_finalize(void *workspace, int64_t n_logical_rows, int64_t hidden, float *dweight,
                                rmsnorm_stream_t stream) {
    return dweight_finalize_scaled(workspace, n_logical_rows, hidden, 1.f, dweight, stream);
}

extern "C" int dweight_finalize_scaled(void *workspace, int64_t n_logical_rows, int64_t hidden, float grad_scale,
                                       float *dweight, rmsnorm_stream_t stream) {
    if (!std::isfinite(grad_scale)) return RMSNORM_ERR_VALUE;
    int rc = ws_checks(workspace, n_logical_rows, hidden);
    if (rc) return rc;
    if (!dweight) return RMSNORM_ERR_NULL;
    if (!aligned16(dweight)) return RMSNORM_ERR_ALIGN;
    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    WsView ws = ws_view(workspace, n_logical_rows, hidden);
    if (ws.n_blocks == 0) {
        zero_f32_kernel<<<1, 256, 0, s>>>(dweight, hidden);
        if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
        g_launches.fetch_add(1, std::memory_order_relaxed);
        return RMSNORM_OK;
    }
    return finalize_blocks(ws, 0, ws.n_blocks, dweight, grad_scale, s);
}

extern "C" int dweight_finalize_range(void *workspace, int64_t n_logical_rows, int64_t hidden, int64_t block_lo,
                                      int64_t block_count, float *root, rmsnorm_stream_t stream) {
    int rc = ws_checks(workspace, n_logical_rows, hidden);
    if (rc) return rc;
    if (!root) return RMSNORM_ERR_NULL;
    if (!aligned16(root)) return RMSNORM_ERR_ALIGN;
    const int64_t nb = (n_logical_rows + kBlockRows - 1) / kBlockRows;
    if (block_count < 1 || (block_count & (block_count - 1)) != 0 || block_lo < 0 || block_lo % block_count != 0 ||
        block_lo >= nb)
        return RMSNORM_ERR_LAYOUT;
    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    const int64_t count = block_lo + block_count > nb ? nb - block_lo : block_count;
    return finalize_blocks(ws_view(workspace, n_logical_rows, hidden), block_lo, count, root, 1.f,
                           reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int dweight_combine(const float *roots, int64_t n_roots, int64_t hidden, float grad_scale,
                               float *dweight, rmsnorm_stream_t stream) {
    if (!std::isfinite(grad_scale)) return RMSNORM_ERR_VALUE;
    Shape sh;
    if (!hidden_shape(hidden, &sh)) return RMSNORM_ERR_HIDDEN;
    if (!roots || !dweight) return RMSNORM_ERR_NULL;
    if (!aligned16(roots) || !aligned16(dweight)) return RMSNORM_ERR_ALIGN;
    if (n_roots < 1 || n_roots >= 2048) return RMSNORM_ERR_LAYOUT;
    DeviceInfo *d = nullptr;
    int rc = device_info(&d);
    if (rc) return rc;
    const int V = int(hidden / 8);
    combine_kernel<<<unsigned((V + 127) / 128), 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        roots, n_roots, int(hidden), grad_scale, dweight);
    if (cudaGetLastError() != cudaSuccess) return RMSNORM_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return RMSNORM_OK;
}

extern "C" int rmsnorm_dweight_status(const void *workspace, rmsnorm_stream_t stream, int32_t *status) {
    if (!workspace || !status) return RMSNORM_ERR_NULL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const WsHeader *h = static_cast<const WsHeader *>(workspace);
    if (cudaMemcpyAsync(status, &h->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

extern "C" const char *rmsnorm_strerror(int code) {
    switch (code) {
        case RMSNORM_OK: return "ok";
        case RMSNORM_ERR_NULL: return "a required pointer is NULL";
        case RMSNORM_ERR_HIDDEN: return "hidden size not supported";
        case RMSNORM_ERR_ALIGN: return "pointer not 16-byte aligned or stride not a multiple of 8";
        case RMSNORM_ERR_STRIDE: return "token_stride smaller than rows_per_token * hidden";
        case RMSNORM_ERR_LAYOUT: return "invalid layout sizes";
        case RMSNORM_ERR_WORKSPACE: return "workspace too small";
        case RMSNORM_ERR_PLAN: return "dweight contribution needs a plan";
        case RMSNORM_ERR_ID: return "token id out of range";
        case RMSNORM_ERR_DUPLICATE: return "logical token appears twice in one call";
        case RMSNORM_ERR_CAPACITY: return "plan buffer too small";
        case RMSNORM_ERR_CUDA: return "CUDA runtime error";
        case RMSNORM_ERR_DEVICE: return "device is not sm_103";
        case RMSNORM_ERR_VALUE: return "grad_scale is not finite";
        default: return "unknown error";
    }
}

extern "C" int64_t rmsnorm_kernel_launches(void) { return g_launches.load(); }

// ==================================================================== allocation-free backward
//
// The workspace of rmsnorm_bwd_noalloc lives in this file-scope device array.
// In host code the symbol is only a stand-in; its device address is looked up
// once per device with cudaGetSymbolAddress and passed to the kernels.

static __device__ __align__(256) uint8_t g_noalloc_scratch[RMSNORM_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_addr[64] = {nullptr};

int noalloc_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RMSNORM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return RMSNORM_ERR_CUDA;
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return RMSNORM_OK;
}
}  // namespace

extern "C" int rmsnorm_bwd_noalloc(const uint16_t *x, const uint16_t *weight, const uint16_t *dy, int64_t hidden,
                                   float eps, const rmsnorm_layout_t *layout, uint16_t *dx, float *dweight,
                                   int32_t *status, rmsnorm_stream_t stream) {
    Shape sh;
    if (!hidden_shape(hidden, &sh)) return RMSNORM_ERR_HIDDEN;
    int rc = check_layout(layout, hidden);
    if (rc) return rc;
    if (!dweight) return RMSNORM_ERR_NULL;
    if (!aligned16(dweight)) return RMSNORM_ERR_ALIGN;
    // every argument error returns before anything is enqueued (the scratch
    // is cleared by the first launch)
    if (layout->n_tokens > 0) {
        if (!x || !weight || !dy) return RMSNORM_ERR_NULL;
        if (!aligned16(x) || !aligned16(weight) || !aligned16(dy) || (dx && !aligned16(dx)))
            return RMSNORM_ERR_ALIGN;
    }
    const int64_t N = layout->n_logical_tokens * layout->rows_per_token;
    const size_t need = rmsnorm_dweight_workspace_bytes(N, hidden);
    if (need == 0) return RMSNORM_ERR_LAYOUT;
    if (need > RMSNORM_NOALLOC_SCRATCH_BYTES) return RMSNORM_ERR_WORKSPACE;
    if (layout->n_tokens > 0 && !layout->plan) return RMSNORM_ERR_PLAN;
    DeviceInfo *d = nullptr;
    if ((rc = device_info(&d))) return rc;
    void *ws = nullptr;
    if ((rc = noalloc_address(&ws))) return rc;
    if ((rc = rmsnorm_dweight_begin(ws, RMSNORM_NOALLOC_SCRATCH_BYTES, N, hidden, stream))) return rc;
    if (layout->n_tokens > 0 && (rc = rmsnorm_bwd_dx(x, weight, dy, hidden, eps, layout, dx, ws, stream))) return rc;
    if ((rc = dweight_finalize(ws, N, hidden, dweight, stream))) return rc;
    if (status) {
        const WsHeader *h = static_cast<const WsHeader *>(ws);
        if (cudaMemcpyAsync(status, &h->status, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
    }
    return RMSNORM_OK;
}
