// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarriers with bounded waits, TMA tile
// loads, and the tcgen05 tensor-core / tensor-memory instructions.
//
// Every wait on an mbarrier is bounded in wall-clock time (GQA_WAIT_LIMIT_NS).  A wait
// that expires returns false; the caller records GQA_ERR_DEVICE_TIMEOUT in the status
// word and unwinds, so a lost arrival can never hang the GPU.
#pragma once
#include <cstdint>
#include <cuda.h>

#ifndef GQA_WAIT_LIMIT_NS
#define GQA_WAIT_LIMIT_NS 2000000000ull   // 2 s
#endif

namespace gqa {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Records the first device-side error (later ones are dropped).
__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Diagnostic code of the first bounded wait that expired, stored next to the status word:
// (kernel << 24) | (role << 20) | (barrier << 16) | (tile index & 0xffff).
enum DiagKernel {
    kDiagPrefill = 1,
    kDiagPrefillWide = 2,
    kDiagDecode = 3,
    kDiagWatchdog = 4,
    kDiagPrefillPair = 5,
    kDiagCache = 6   // cache append, chunk gather, RoPE pass, Q/K normalisation
};
__device__ __forceinline__ void set_timeout(int *status, int kernel, int role, int barrier,
                                            int tile) {
    if (!status) return;
    const int code = (kernel << 24) | (role << 20) | (barrier << 16) | (tile & 0xffff);
    atomicCAS(status, 0, -6 /* GQA_ERR_DEVICE_TIMEOUT */);
    atomicCAS(status + 1, 0, code);                // first expired wait overall
    atomicCAS(status + 2 + (role & 3), 0, code);   // first expired wait of this role
}

// ---- index checks of the debug build ----------------------------------------------------
// Built with -DGQA_DEBUG_BOUNDS, GQA_IN_BOUNDS(i, n, status, site) checks 0 <= i < n before
// a global access whose index comes from device-side data (a cache slot, a table row, a
// workspace record).  A failing check records GQA_ERR_DEVICE_BOUNDS (the first device
// error wins) and the site's code in the diagnostic word, (kernel << 24) | (1 << 23) |
// site, and evaluates to false: the caller skips the access or uses a safe index.  It
// never traps.  In other builds it is the constant true.
#ifdef GQA_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(long i, long n, int *status, int site) {
    if (i >= 0 && i < n) return true;
    if (status) {
        atomicCAS(status, 0, -9 /* GQA_ERR_DEVICE_BOUNDS */);
        atomicCAS(status + 1, 0, site | (1 << 23));
    }
    return false;
}
#define GQA_IN_BOUNDS(i, n, status, site) \
    ::gqa::in_bounds(static_cast<long>(i), static_cast<long>(n), (status), (site))
#else
#define GQA_IN_BOUNDS(i, n, status, site) ((void)(n), true)
#endif

// ---- mbarrier ---------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if it did not
// complete within limit_ns nanoseconds.
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity,
                                              uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// mbar_wait_for with the library-wide limit, GQA_WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, GQA_WAIT_LIMIT_NS);
}

// ---- TMA ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load: box at coordinates (c0 innermost, c1, c2) into shared memory, completing
// `bytes` on the mbarrier.  c0 * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// tma_load_3d multicast to the CTAs of the cluster in `mask`: the box lands at the same
// shared-memory offset in each, and each one's mbarrier at the offset of `bar` receives
// the bytes.  Only for this GPU's own memory.
__device__ __forceinline__ void tma_load_3d_mc(void *dst, const CUtensorMap *map, uint64_t *bar,
                                               int c0, int c1, int c2, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "h"(mask)
        : "memory");
}

// 1-D bulk copy global -> shared (TMA engine), completing `bytes` on the mbarrier.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
        "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled store shared -> global of the box at (c0, c1, c2) (bulk-group completion);
// elements outside the tensor are not written.  c0 * element size must be a multiple of
// 16 bytes and no coordinate may be negative.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until the shared memory of every committed bulk store has been read.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- cluster launch control (dynamic work for persistent CTAs) ------------------------
// Asks the hardware to cancel one CTA of this grid that has not been launched yet; the
// 16-byte response is written to `resp` and completes 16 bytes of transaction on `bar`
// (arm it with mbar_arrive_expect_tx(bar, 16) first).  Never issue another request after
// a response that reported no cancellation.
__device__ __forceinline__ void clc_try_cancel(void *resp, uint64_t *bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
        "[%0], [%1];" ::"r"(smem_u32(resp)),
        "r"(smem_u32(bar))
        : "memory");
}
// The x index of the cancelled CTA in a response, or -1 if nothing was cancelled.
__device__ __forceinline__ int clc_decode(const void *resp) {
    uint32_t canceled, x = 0;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b128 r;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(canceled), "+r"(x)
        : "r"(smem_u32(resp))
        : "memory");
    return canceled ? static_cast<int>(x) : -1;
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05: tensor memory ------------------------------------------------------------
// Allocation is warp-collective; the TMEM address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- tcgen05: descriptors ----------------------------------------------------------------
// Shared-memory matrix descriptor (sm_100 format): start address, leading and stride
// byte offsets (16-byte units), descriptor version 1 (bits 46-47), 128-byte swizzle
// (layout type 2 in bits 61-63).  Atoms are 1024-byte aligned, so the base offset is 0.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A and B and an fp32 accumulator.
// a_mn / b_mn: 1 if that operand is MN-major (transposed), 0 if K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- tcgen05: MMA --------------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T, one elected thread issues.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on the mbarrier when every tcgen05 operation this thread issued before
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// umma_commit to the mbarrier at the offset of `bar` in each CTA of the cluster in `mask`.
__device__ __forceinline__ void umma_commit_mc(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// ---- tcgen05: TMEM <-> registers (warp-collective, 32 lanes x 32-bit, 32 columns) ---------
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- register split between warpgroups (all warps of a warpgroup execute the same one) ----
template <uint32_t N>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---- programmatic dependent launch ----------------------------------------------------------
// A kernel launched with programmatic stream serialization may start before the previous
// kernel on its stream has finished: griddep_wait() returns once that kernel has completed
// and its writes are visible (at once when there is no such dependency), and
// griddep_launch_dependents() lets the next kernel start launching.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- thread-block clusters (distributed shared memory) ------------------------------------
// This CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the variable at shared::cta address `addr` in the CTA of
// the cluster with rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Every thread of every CTA of the cluster arrives, then waits for all of them (release /
// acquire at cluster scope).  Every thread of the cluster must execute it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// 1-D bulk copy from this CTA's shared memory to the shared memory of a CTA of the cluster
// (dst and bar are shared::cluster addresses in that CTA); completes `bytes` of
// transaction on that CTA's mbarrier.  Addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_s2c(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(dst),
        "r"(smem_u32(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Arrives once on an mbarrier of another CTA of the cluster (shared::cluster address),
// ordering this thread's earlier memory accesses before the arrival at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}

// mbar_wait for a phase completed from another CTA of the cluster (acquire at cluster
// scope): an arrival or a transaction count from a remote thread or copy.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer_ns() - t0 > GQA_WAIT_LIMIT_NS) return false;
    }
}

// ---- misc ----------------------------------------------------------------------------------
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Three-input maximum (one instruction on sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed fp32x2 a * b + c with scalar b and c, round to nearest (sm_100+).
__device__ __forceinline__ float2 ffma2(float2 a, float b, float c) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\tmov.b64 rc, {%5, %5};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b), "f"(c));
    return r;
}

// Packed fp32x2 a + b, round to nearest (sm_100+).
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// Packed fp32x2 a - b, round to nearest (sm_100+).
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// Packed fp32x2 a * b, round to nearest (sm_100+).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// Packed fp32x2 a * b + c, all operands pairs, round to nearest (sm_100+).
__device__ __forceinline__ float2 ffma2v(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// 2^x for two values on the FMA and integer pipes, so that part of a softmax's
// exponentials can bypass the special-function unit (which the softmax saturates).
// Cody-Waite style reduction: x = n + f with n = rint(x) (the add of 1.5 * 2^23 rounds
// to an integer and leaves n in the low mantissa bits), f in [-1/2, 1/2];
// 2^f = 1 + f * (a0 + f * (a1 + f * a2)), the Chebyshev interpolant written out by
// exp2_poly.py (relative error below 2.5e-4 over the range); n is then added into the
// exponent field.  x is clamped below at -127, where f = 0 and the result is exactly
// +0.0, so -inf (a masked score) maps to 0.  Valid for x <= 127.
constexpr float kExp2A0 = 0x1.62e43p-1f;
constexpr float kExp2A1 = 0x1.efb038p-3f;
constexpr float kExp2A2 = 0x1.c8bdfap-5f;
__device__ __forceinline__ float2 ex2_fma2(float2 x) {
    constexpr float kMagic = 12582912.0f;
    x.x = fmaxf(x.x, -127.0f);
    x.y = fmaxf(x.y, -127.0f);
    const float2 t = fadd2(x, make_float2(kMagic, kMagic));
    const float2 f = fsub2(x, fsub2(t, make_float2(kMagic, kMagic)));
    float2 u = ffma2v(make_float2(kExp2A2, kExp2A2), f, make_float2(kExp2A1, kExp2A1));
    u = ffma2v(u, f, make_float2(kExp2A0, kExp2A0));
    const float2 pw = ffma2v(u, f, make_float2(1.0f, 1.0f));
    return make_float2(__uint_as_float(__float_as_uint(pw.x) + (__float_as_uint(t.x) << 23)),
                       __uint_as_float(__float_as_uint(pw.y) + (__float_as_uint(t.y) << 23)));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace gqa
