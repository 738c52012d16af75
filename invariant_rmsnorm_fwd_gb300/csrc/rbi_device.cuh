// Device helpers for the batch-invariant RMSNorm kernels (sm_103a).
//
// Every floating-point operation on the numeric path is an explicit
// round-to-nearest intrinsic (__fadd_rn, __fmul_rn, __fmaf_rn, ...), and the
// library is compiled with -fmad=false, so the compiler can neither contract
// nor reassociate: a value depends only on the operands and the fixed order
// written here, never on which kernel, launch shape or layout produced it.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace rbi {

constexpr int kBlockRows = 64;       // logical block of the dweight reduction
constexpr int kBlockLevels = 6;      // log2(kBlockRows)
constexpr unsigned kFull = 0xffffffffu;

// Longest wait of any pipeline role before it gives up and reports a timeout
// (1 s).  A test-only build of the library sets RBI_WAIT_LIMIT_NS lower.
#ifndef RBI_WAIT_LIMIT_NS
#define RBI_WAIT_LIMIT_NS 1000000000ull
#endif
constexpr uint64_t kWaitLimitNs = RBI_WAIT_LIMIT_NS;

// Status bits (mirror RMSNORM_STATUS_* in the public header).
constexpr int kStDouble = 1, kStMissing = 2, kStHeader = 4, kStPlan = 8, kStTimeout = 16;

// ----------------------------------------------------------------- workspace

constexpr uint64_t kWsMagic = 0x3149422d4d524e52ull;   // "RNMR-BI1"

struct WsHeader {
    uint64_t magic;
    int64_t n_rows;
    int64_t hidden;
    int64_t n_blocks;
    int32_t status;
    int32_t pad[55];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

struct WsView {                      // device addresses of the workspace regions
    WsHeader *hdr;
    uint8_t *block_state;            // [nb][4] per quarter: 0 none, 1 quarter partial, 2 whole-block partial,
                                     //   4 / 8 / 12 first / second / both eighth partials
    uint8_t *leaf_flag;              // [N]    1 = row spilled
    float *block_partial;            // [nb][4][H] quarter partials (slot 0 holds a whole-block partial;
                                     //   a quarter split in two eighths holds the first one)
    float *eighth;                   // [nb][4][H] second eighth partials of split quarters
    float *scratch_a;                // [ceil(nb/32)][H]
    float *scratch_b;                // [ceil(nb/32)][H]
    float *spill;                    // [N][H]
    int64_t n_rows, hidden, n_blocks;
};

__host__ __device__ inline int64_t align256(int64_t v) { return (v + 255) & ~int64_t(255); }

// Region offsets depend only on (N, H); host and device compute them alike.
struct WsLayout {
    int64_t off_state, off_flag, off_partial, off_eighth, off_sa, off_sb, off_spill, total;
    __host__ __device__ WsLayout(int64_t N, int64_t H) {
        int64_t nb = (N + kBlockRows - 1) / kBlockRows;
        int64_t ng = (nb + 31) / 32;                     // first-pass groups of 32 blocks
        off_state = 256;
        off_flag = align256(off_state + nb * 4);
        off_partial = align256(off_flag + N);
        off_eighth = align256(off_partial + nb * 4 * H * 4);
        off_sa = align256(off_eighth + nb * 4 * H * 4);
        off_sb = align256(off_sa + ng * H * 4);
        off_spill = align256(off_sb + ng * H * 4);
        total = align256(off_spill + N * H * 4);
    }
};

inline WsView ws_view(void *base, int64_t N, int64_t H) {
    WsLayout L(N, H);
    uint8_t *b = static_cast<uint8_t *>(base);
    WsView v;
    v.hdr = reinterpret_cast<WsHeader *>(b);
    v.block_state = b + L.off_state;
    v.leaf_flag = b + L.off_flag;
    v.block_partial = reinterpret_cast<float *>(b + L.off_partial);
    v.eighth = reinterpret_cast<float *>(b + L.off_eighth);
    v.scratch_a = reinterpret_cast<float *>(b + L.off_sa);
    v.scratch_b = reinterpret_cast<float *>(b + L.off_sb);
    v.spill = reinterpret_cast<float *>(b + L.off_spill);
    v.n_rows = N;
    v.hidden = H;
    v.n_blocks = (N + kBlockRows - 1) / kBlockRows;
    return v;
}

__device__ __forceinline__ void set_status(WsHeader *h, int bit) {
    // Error reporting only: a plain store of the OR of what this thread saw.
    // Concurrent writers can only lose a bit if two different errors race,
    // and any non-zero word already reports failure.
    volatile int32_t *s = &h->status;
    *s = *s | bit;
}

__device__ __forceinline__ bool header_ok(const WsView &ws) {
    const WsHeader *h = ws.hdr;
    return h->magic == kWsMagic && h->n_rows == ws.n_rows && h->hidden == ws.hidden;
}

// ----------------------------------------------------------------- plan items

struct PlanItem {                    // written by the host planner
    int32_t kind;                    // 0 = whole logical block, 1 = rows of cut blocks,
                                     // 2 = complete quarters of a cut block
    int32_t block;                   // block id for kinds 0 and 2, -1 otherwise
    int32_t count;                   // used slots
    int32_t quarters;                // kind 2: bit q set = quarter q present (slots 16q..16q+15)
    int32_t prow[kBlockRows];        // physical row within the call, -1 = empty slot
    int32_t lrow[kBlockRows];        // logical row id, -1 = empty slot
};

// Item kinds as staged for the kernels: the low byte is the kind, bits 8-11
// the quarter mask of a kind-2 item; kBadItem marks a malformed item, which
// contributes nothing.
constexpr int kItemWhole = 0, kItemSpill = 1, kItemQuarters = 2, kBadItem = 3;
__device__ __forceinline__ int32_t staged_kind(const PlanItem &it) {
    return it.kind == kItemQuarters ? (kItemQuarters | ((it.quarters & 15) << 8)) : it.kind;
}
static_assert(sizeof(PlanItem) == 528, "plan item layout is part of the ABI");

// ----------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity; gives up after kWaitLimitNs of wall time.
// Between polls the warp sleeps (32 ns, doubling to 256 ns) so that waiting
// warps leave the issue slots to the warps that have work.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t ns = 32;
#pragma unroll 1
    while (true) {
        __nanosleep(ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (ns < 256) ns <<= 1;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// The same bounded wait without sleeping between polls, for the few threads
// whose latency sets the pace (the MMA issuer and the producer of a tensor-core
// pipeline): try_wait itself suspends the thread for a short hardware time
// window, and the clock is read only every 256 polls.
__device__ __forceinline__ bool mbar_wait_spin_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// The spinning wait with cluster-scope acquire, for an mbarrier that threads
// of another CTA of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_spin_bounded_cluster(uint64_t *bar, uint32_t parity);

// One-dimensional bulk copy global -> this CTA's shared memory, completion
// counted in bytes on `bar`.  Both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// cp.async groups: each thread waits only for its own copies.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Cluster-scope variants used by the cross-CTA exchange of row-sum partials.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_spin_bounded_cluster(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t ns = 32;
#pragma unroll 1
    while (true) {
        __nanosleep(ns);
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (ns < 256) ns <<= 1;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Asynchronous store of two floats to shared::cluster address `addr` (another
// CTA's shared memory, or this CTA's); its completion decrements the
// transaction count of the mbarrier at shared::cluster address `bar` (in the
// same CTA as `addr`) by 8 bytes.
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
                 "f"(a), "f"(b), "r"(bar)
                 : "memory");
}

// Arrive on the mbarrier at shared::cluster address `addr` (possibly another
// CTA's), releasing this thread's earlier shared-memory stores at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// Arrival with an expected transaction count on the mbarrier at shared::cluster
// address `addr` (possibly another CTA's).  CTA-scope release: the arriving
// thread publishes no data of its own (the bytes counted are asynchronous
// copies, which complete on the barrier themselves).
__device__ __forceinline__ void mbar_arrive_expect_tx_remote(uint32_t addr, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(addr), "r"(bytes) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}


__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ uint4 ld_shared_v4(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

__device__ __forceinline__ void st_global_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_global_f32x4(float *p, float a, float b, float c, float d) {
    asm volatile("st.global.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ float4 ld_global_f32x4(const float *p) {
    float4 v;
    asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// ----------------------------------------------------------------- f2: FP32 pairs in 64-bit registers
//
// sm_100-class GPUs execute two FP32 lanes per instruction (add/mul/fma
// .rn.f32x2).  Each lane is an ordinary IEEE binary32 round-to-nearest-even
// operation, so values are the same as with scalar __fadd_rn/__fmul_rn/
// __fmaf_rn; only the instruction count halves.  The pair lives in one
// 64-bit register from the bf16 unpack (exact: the bf16 bits are the top
// half of the binary32) to the bf16 pack.

typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
    f2_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
    f2_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
    f2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2_t f2_make(float lo, float hi) {
    f2_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ float f2_lo(f2_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo;
}
__device__ __forceinline__ float f2_hi(f2_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return hi;
}
// two bf16 (low half = even column) -> FP32 pair, exact
__device__ __forceinline__ f2_t f2_from_bf16x2(uint32_t w) {
    f2_t d;
    asm("{\n\t.reg .b32 lo, hi;\n\tshl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xffff0000;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(d)
        : "r"(w));
    return d;
}
// FP32 pair -> two bf16, round-to-nearest-even (even column in the low half)
__device__ __forceinline__ uint32_t f2_to_bf16x2(f2_t v) {
    uint32_t r;
    asm("{\n\t.reg .f32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\tcvt.rn.bf16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(r)
        : "l"(v));
    return r;
}
__device__ __forceinline__ void f2_unpack8(const uint4 &v, f2_t (&f)[4]) {
    f[0] = f2_from_bf16x2(v.x);
    f[1] = f2_from_bf16x2(v.y);
    f[2] = f2_from_bf16x2(v.z);
    f[3] = f2_from_bf16x2(v.w);
}
// The same unpacking as a volatile sequence: the compiler may not merge it
// with an earlier unpacking of the same registers, so the unpacked values
// need not stay live in between (used where packed data is kept across phases).
__device__ __forceinline__ f2_t f2_from_bf16x2_v(uint32_t w) {
    f2_t d;
    asm volatile("{\n\t.reg .b32 lo, hi;\n\tshl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xffff0000;\n\t"
                 "mov.b64 %0, {lo, hi};\n\t}"
                 : "=l"(d)
                 : "r"(w));
    return d;
}
__device__ __forceinline__ void f2_unpack8_v(const uint4 &v, f2_t (&f)[4]) {
    f[0] = f2_from_bf16x2_v(v.x);
    f[1] = f2_from_bf16x2_v(v.y);
    f[2] = f2_from_bf16x2_v(v.z);
    f[3] = f2_from_bf16x2_v(v.w);
}
__device__ __forceinline__ uint4 f2_pack8(const f2_t (&f)[4]) {
    return make_uint4(f2_to_bf16x2(f[0]), f2_to_bf16x2(f[1]), f2_to_bf16x2(f[2]), f2_to_bf16x2(f[3]));
}
__device__ __forceinline__ void st_global_f2x4(float *p, const f2_t (&f)[4]) {
    asm volatile("st.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(f[0]), "l"(f[1]) : "memory");
    asm volatile("st.global.v2.b64 [%0], {%1, %2};" ::"l"(p + 4), "l"(f[2]), "l"(f[3]) : "memory");
}

// ----------------------------------------------------------------- lane vectors of 8 bf16 columns

__device__ __forceinline__ void vec_unpack(const uint4 &v, f2_t (&f)[4]) { f2_unpack8(v, f); }
__device__ __forceinline__ void vec_unpack_v(const uint4 &v, f2_t (&f)[4]) { f2_unpack8_v(v, f); }
__device__ __forceinline__ void vec_pack(const f2_t (&f)[4], uint4 &r) { r = f2_pack8(f); }
__device__ __forceinline__ void vec_zero(uint4 &r) { r = make_uint4(0, 0, 0, 0); }

// Asynchronous 16-byte copy of one lane vector global -> shared (L2 only), of
// which the first src_bytes are read and the rest written as zeros
// (src_bytes = 0: nothing is read; src must still be a valid address);
// completion through the cp.async groups.  dst is a shared-memory address.
__device__ __forceinline__ void cp_async_zfill(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void ld_shared_vec(uint32_t addr, uint4 &v) {
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
}
// Stores that take effect only when pred != 0 (no branch).
__device__ __forceinline__ void st_global_vec_if(void *p, const uint4 &v, uint32_t pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t@q st.global.v4.u32 [%0], {%1,%2,%3,%4};\n\t}" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(pred)
                 : "memory");
}
__device__ __forceinline__ void st_global_f2_if(float *p, const f2_t (&f)[4], uint32_t pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q st.global.v2.b64 [%0], {%1, %2};\n\t}" ::"l"(p),
                 "l"(f[0]), "l"(f[1]), "r"(pred)
                 : "memory");
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q st.global.v2.b64 [%0], {%1, %2};\n\t}" ::"l"(p + 4),
                 "l"(f[2]), "l"(f[3]), "r"(pred)
                 : "memory");
}
__device__ __forceinline__ void st_global_f32_if(float *p, float v, uint32_t pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.global.f32 [%0], %1;\n\t}" ::"l"(p), "f"(v),
                 "r"(pred)
                 : "memory");
}

// ----------------------------------------------------------------- 64-leaf tree
//
// Streaming form of the complete pairwise tree over the 64 leaves of a
// logical block: leaf n (0..63) is combined with the pending partials whose
// bits are set in n (binary counter), earlier leaves always on the left.
// After leaf 63 the returned value is the block partial.  Any subtree of 2^k
// aligned leaves can be pushed as one item at level k.
//
// TreeStackF2 holds the pending partials of NC FP32 column pairs per lane in
// registers, for compile-time item indices (push_static);
// push_group_subtree keeps them in shared memory for a run-time index that is
// uniform across the warp.
template <int NC, int LEVELS>
struct TreeStackF2 {
    f2_t s[LEVELS][NC];

    template <int LEVEL>
    __device__ __forceinline__ void push_static(f2_t (&v)[NC], int idx) {
#pragma unroll
        for (int l = LEVEL; l < LEVELS; ++l) {
            if ((idx >> (l - LEVEL)) & 1) {
#pragma unroll
                for (int c = 0; c < NC; ++c) v[c] = f2_add(s[l][c], v[c]);
            } else {
#pragma unroll
                for (int c = 0; c < NC; ++c) s[l][c] = v[c];
                break;
            }
        }
    }
};

// The same push for a run-time index uniform across the warp, with the
// pending partials in shared memory (level l at base + l * stride, NC pairs
// per lane): only the levels that the item closes are read.
template <int NC, int LEVELS>
__device__ __forceinline__ void push_group_subtree(f2_t (&v)[NC], int idx, uint32_t base, uint32_t stride) {
    bool carry = true;
#pragma unroll
    for (int l = 0; l < LEVELS; ++l) {
        if (carry) {
            const uint32_t a = base + l * stride;
            if ((idx >> l) & 1) {
#pragma unroll
                for (int c = 0; c < NC; c += 2) {
                    f2_t s0, s1;
                    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(s0), "=l"(s1) : "r"(a + c * 8));
                    v[c] = f2_add(s0, v[c]);
                    v[c + 1] = f2_add(s1, v[c + 1]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < NC; c += 2)
                    asm volatile("st.shared.v2.b64 [%0], {%1, %2};" ::"r"(a + c * 8), "l"(v[c]), "l"(v[c + 1])
                                 : "memory");
                carry = false;
            }
        }
    }
}

// ----------------------------------------------------------------- row sums
//
// Canonical row-sum trees.  The sum of squares (and, in the backward, the
// sum of dy*w*x) of a row is formed by a tree that depends on H only:
//
//  hidden <= 256 (small_row_kernel): each 8-column vector is folded as two
//   FMA chains (columns 0,2,4,6 and 1,3,5,7) that are then added, and the
//   V = H/8 vector sums, zero-padded to P = next_pow2(V), are added by a
//   complete tree with adjacent pairing: (0,1), (2,3), ... (xor butterflies
//   1, 2, 4, ...).
//  hidden > 256 (split_kernel): see the description above split_kernel in
//   rmsnorm_kernels.cuh (lane folds within each column slice, a lane tree
//   pairing 16 apart first, then the slice sums in a fixed order).
//
// The forward and the backward use the same kernel family for a given H, so
// rstd is bitwise the same in both.

// v / H, correctly rounded.  For a power-of-two H it is the product with the
// exact reciprocal 2^-k: both operations round the same real number, so the
// result is the same bit pattern and the division's longer sequence is
// skipped.  inv_h is 1/H for a power-of-two H and 0 otherwise (row_inv_h).
__device__ __forceinline__ float div_h(float v, float Hf, float inv_h) {
    return inv_h != 0.f ? __fmul_rn(v, inv_h) : __fdiv_rn(v, Hf);
}
__device__ __forceinline__ float row_inv_h(int H) {
    return (H & (H - 1)) == 0 ? __frcp_rn(float(H)) : 0.f;
}

// rstd = 1 / sqrt(ss / H + eps), each step correctly rounded.
__device__ __forceinline__ float row_rstd(float ss, float Hf, float inv_h, float eps) {
    return __frcp_rn(__fsqrt_rn(__fadd_rn(div_h(ss, Hf, inv_h), eps)));
}

// m = mean(g * xhat) = (rstd * sum(g * x)) / H.
__device__ __forceinline__ float row_mean_gxhat(float gx, float rstd, float Hf, float inv_h) {
    return div_h(__fmul_rn(gx, rstd), Hf, inv_h);
}

}  // namespace rbi
