// prefill.cu -- flash-style causal / sliding-window GQA prefill on tcgen05 tensor cores.
//
// Computes, for one layer ("PLaMo 3アーキテクチャ徹底解析" §4.5, §5.1):
//   O[b,h,t] = sum_s softmax_s(scale <Q'[b,h,t], K'[b,g(h),s]> masked) V[b,g(h),s]
// without materialising the score matrix: S = Q K^T and O += P V run as 128x128 tiles
// on the tensor cores with fp32 accumulators in tensor memory, and the softmax is an
// online (running max / running sum) fp32 pass over each S tile.
//
// Work item = (batch b, KV head g, pair of query heads of that group, block of 128 query
// rows).  Both query tiles of an item sit at the same positions and read the same KV
// head, so they share every K and V tile load and the same mask.  Only key tiles that
// intersect [q_pos - W + 1, q_pos] for some row of the block are loaded (window tile
// skipping, §1 and §5.3: local prefill costs O(T W)); the per-element mask is applied on
// the tiles that straddle the diagonal or the window's lower edge only.
//
// The kernel is persistent: the grid has one CTA per item, but the CTAs that get an SM
// claim the items of CTAs not launched yet (cluster launch control), so each SM keeps one
// CTA that walks items in launch order (longest rows first) and the load balances itself.
// The per-item fixed work overlaps the previous item: the next item's Q tiles are loaded
// into the second of two Q buffers and rotated while the current item runs, and the
// current item's epilogue overlaps the next item's first score products.
//
// Warp roles (12 warps, 3 warpgroups; 3 warps per SM sub-partition cap every thread at
// 168 registers at launch, and warpgroup 0 then hands registers to the two softmax
// warpgroups: 96 and 200 per thread):
//   warp 0      TMA producer: Q tiles of each item into Q buffer (item & 1), K and V
//               tiles into a 3-slot ring in the order they are consumed:
//               K(0), V(0), K(1), V(1), ...
//   warp 1      tensor-memory allocator and the single MMA-issuing thread.
//   warps 2-3   RoPE (§6.1) on each item's Q tiles in shared memory, ahead of use (and,
//               in the fused-K form, on every K tile as it lands in the ring); warp 2 also
//               issues the TMA stores of each item's O once the epilogue has staged it.
//   warps 4-7   softmax + epilogue for query tile 0, warps 8-11 for query tile 1: one
//               thread per query row; warp w reads TMEM lanes 32*(w%4).. (its quarter).
// K normally arrives already rotated (the caller-side pass rotates each key once).  The
// fused-K form (KROT) takes K before RoPE and rotates each K tile in shared memory, at
// positions n0 .. n0 + 127, between its landing and its score products: no workspace and
// no pass over K, but every reload of a K tile is rotated again (each tile is reloaded
// once per query block whose window reaches it).
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512).
// P (bf16) overwrites the first 64 columns of its S tile and feeds the PV product
// directly from tensor memory.  The tensor pipe does not order an MMA's reads of its
// TMEM operand before a later MMA's writes to the same columns, so S_i(j+1) is issued
// only after PV_i(j) has completed.  Rescaling of O is lazy: it happens only when a row's
// maximum grows by more than 2^8, otherwise the stale maximum is kept (exact, since O and
// the running sum always share one reference maximum).
//
// Barrier phases run across items: every role counts the completions it has consumed
// (per query tile) and waits on the parity of that count.  No barrier can run two phases
// ahead of a waiter, because each producer of a phase first waits on a consequence of
// the previous one.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kSlots = 3;                     // K/V ring depth
constexpr int kBoxBytes = 128 * 128;          // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kTileBytes = 2 * kBoxBytes;     // 128 rows x 128 bf16
constexpr int kSmemQ = 0;                     // 2 buffers x 2 query tiles
constexpr int kSmemRing = 4 * kTileBytes;
constexpr int kSmemBar = kSmemRing + kSlots * kTileBytes;
constexpr int kSmemBytes = kSmemBar + 512 + 1024;  // + barriers + alignment slack
constexpr int kThreads = 384;
constexpr int kRotThreads = 64;               // warps 2-3
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;     // log2 units
// Items with at least this many key tiles on average go to the one-CTA-per-item kernel:
// their per-item fixed work is small next to the item, and the hardware balances uneven
// causal item lengths better than the static persistent schedule (GB300 measurements:
// persistent 0.56 vs 0.51 of peak at ~17 tiles per item, 0.68 vs 0.74 at ~128).
constexpr int kStreamMinTiles = 48;
// Column pairs (bit i: pair i of each 32-column chunk) whose exponentials run on the FMA
// pipe (ex2_fma2) instead of the special-function unit.  Off by default: the softmax is
// bound by instruction issue and latency, not by the special-function unit, so the
// extra instructions cost more than the offload saves (measured on GB300).
#ifndef GQA_PREFILL_POLY_PAIRS
#define GQA_PREFILL_POLY_PAIRS 0x0000u
#endif
constexpr uint32_t kPolyPairs = GQA_PREFILL_POLY_PAIRS;

constexpr int kItemSlots = 4;                 // responses of the work-claiming ring
constexpr int kItemReaders = 11;              // MMA thread + 2 RoPE warps + 8 softmax warps

struct Bars {
    uint4 clc_resp[kItemSlots];                   // cluster-launch-control responses
    uint64_t clc_full[kItemSlots];                // response for item k landed (slot k & 3)
    uint64_t item_free[kItemSlots];               // every role has read that response
    uint64_t q_full[2], q_ready[2];               // per Q buffer
    uint64_t epi_done[2];                         // the buffer's O staging has been stored
    uint64_t staged[2][2];                        // [buffer][query tile]: O rows in smem
    uint64_t full[kSlots], empty[kSlots];         // K/V ring
    uint64_t s_full[2], p_full[2], o_done[2];     // per query tile
    uint64_t o_final[2];                          // an item's last PV product of the tile
    uint64_t o_free[2];                           // the epilogue has read O out of TMEM
    uint64_t krot[2];                             // fused-K form: K tile rotated (alternate)
    uint64_t mma_done;
    uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct Params {
    __nv_bfloat16 *o;
    float *lse;
    const float2 *table;
    int *status;
    int T, S, Hq, Hkv, G, window;
    int n_mblocks, n_pairs, n_items;
    float scale_log2;
};

struct Item {
    int mb, g, b, h0, kt_first, n_tiles;
    bool two;
};

// Item index -> its coordinates; query blocks with the most keys first.
__device__ __forceinline__ Item make_item(const Params &p, int idx) {
    Item it;
    const int pair = idx % p.n_pairs;
    idx /= p.n_pairs;
    it.mb = p.n_mblocks - 1 - (idx % p.n_mblocks);
    idx /= p.n_mblocks;
    it.g = idx % p.Hkv;
    it.b = idx / p.Hkv;
    it.h0 = it.g * p.G + 2 * pair;
    it.two = (2 * pair + 1) < p.G;
    const int q_lo = p.S - p.T + it.mb * kBM;                 // position of row 0
    const int q_hi = min(q_lo + kBM - 1, p.S - 1);            // position of the last row
    it.kt_first = p.window > 0 ? max(0, q_lo - p.window + 1) / kBN : 0;
    it.n_tiles = q_hi / kBN - it.kt_first + 1;
    return it;
}

// Work items are claimed dynamically: item 0 of a CTA is its own blockIdx.x (the grid has
// one CTA per item), and during item k the producer asks the hardware to cancel one CTA
// that has not been launched yet and takes over its item as item k + 1 (cluster launch
// control).  CTAs that finish early thus take more items, in launch order (longest rows
// first), without any counter in memory.  The responses go through a 4-slot ring that
// every role reads.

// Item j >= 1 of a CTA has its response in slot (j - 1) % 4, the ((j - 1) / 4)-th use of
// that slot (item 0 is the CTA's own index and has no response).
__device__ __forceinline__ int item_slot(int j) { return (j - 1) & (kItemSlots - 1); }
__device__ __forceinline__ int item_use(int j) { return (j - 1) / kItemSlots; }

// Item k (k >= 1) of this CTA for a reader role: waits for the response, decodes it.
// Returns -1 when nothing was left to claim (or the wait expired: *ok is cleared).
__device__ __forceinline__ int read_item(Bars *bars, int k, int n_items, bool &ok) {
    const int slot = item_slot(k);
    if (!mbar_wait(&bars->clc_full[slot], item_use(k) & 1)) {
        ok = false;
        return -1;
    }
    const int x = clc_decode(&bars->clc_resp[slot]);
    return x < n_items ? x : -1;
}

// A bounded wait whose outcome every lane of the warp agrees on, so the warp-collective
// tcgen05.ld/st that follow are never reached by only part of a warp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// Roles for the diagnostic code of an expired wait.
enum Role { kRoleProducer = 0, kRoleMma = 1, kRoleSoftmax = 2, kRoleRope = 3 };

template <bool KROT>   // K before RoPE, rotated tile by tile in shared memory
__global__ void __launch_bounds__(kThreads, 1)
    prefill_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const Params p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    Bars *bars = reinterpret_cast<Bars *>(smem + kSmemBar);
    auto sQ = [&](int buf, int i) { return smem + kSmemQ + (2 * buf + i) * kTileBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->q_full[i], 1);
            mbar_init(&bars->q_ready[i], kRotThreads);
            mbar_init(&bars->epi_done[i], 2);
            mbar_init(&bars->staged[i][0], 128);
            mbar_init(&bars->staged[i][1], 128);
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->p_full[i], 128);
            mbar_init(&bars->o_done[i], 1);
            mbar_init(&bars->o_final[i], 1);
            mbar_init(&bars->o_free[i], 128);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(&bars->clc_full[i], 1);
            mbar_init(&bars->item_free[i], kItemReaders);
        }
        mbar_init(&bars->krot[0], kRotThreads);
        mbar_init(&bars->krot[1], kRotThreads);
        mbar_init(&bars->mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // Register split (launch: 384 threads x 168): the producer, MMA and RoPE warps
    // (warpgroup 0) give registers to the two softmax warpgroups, which hold a whole
    // 128-column S row per thread: 128 x 96 + 256 x 200 <= 384 x 168, and neither side
    // spills.
    if (warp < 4) {
    reg_dealloc<96>();
    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmO);
            bool ok = true;
            int u = 0;          // ring loads issued
            int q_issued = 0;   // items whose Q tiles have been issued
            // claims item k (k >= 1) of this CTA: one cancellation request into its slot, once
            // every role has read the slot's previous response (item k - 4)
            auto claim = [&](int k) {
                const int slot = item_slot(k);
                if (k > kItemSlots &&
                    !(ok = mbar_wait(&bars->item_free[slot], (item_use(k) - 1) & 1))) {
                    set_timeout(p.status, kDiagPrefill, kRoleProducer, 2, k);
                    return;
                }
                mbar_arrive_expect_tx(&bars->clc_full[slot], 16);
                clc_try_cancel(&bars->clc_resp[slot], &bars->clc_full[slot]);
            };
            auto load_q = [&](int k, int idx) {
                const Item it = make_item(p, idx);
                const int buf = k & 1;
                // buffer reuse: item k - 2 is finished and its O, staged in this buffer,
                // has been read out by the TMA stores
                if (k >= 2 && !(ok = mbar_wait(&bars->epi_done[buf], ((k - 2) >> 1) & 1))) {
                    set_timeout(p.status, kDiagPrefill, kRoleProducer, 0, k);
                    return;
                }
                const int zq = it.b * p.Hq + it.h0;
                mbar_arrive_expect_tx(&bars->q_full[buf], (it.two ? 2 : 1) * kTileBytes);
                for (int i = 0; i < (it.two ? 2 : 1); ++i) {
                    tma_load_3d(sQ(buf, i), &tmQ, &bars->q_full[buf], 0, it.mb * kBM, zq + i);
                    tma_load_3d(sQ(buf, i) + kBoxBytes, &tmQ, &bars->q_full[buf], 64,
                                it.mb * kBM, zq + i);
                }
                q_issued = k + 1;
            };
            auto put = [&](const CUtensorMap *map, int n0, int zk) {
                const int st = u % kSlots;
                if (u >= kSlots && !(ok = mbar_wait(&bars->empty[st], ((u / kSlots) - 1) & 1))) {
                    set_timeout(p.status, kDiagPrefill, kRoleProducer, 1, u);
                    return;
                }
                uint8_t *dst = smem + kSmemRing + st * kTileBytes;
                mbar_arrive_expect_tx(&bars->full[st], kTileBytes);
                tma_load_3d(dst, map, &bars->full[st], 0, n0, zk);
                tma_load_3d(dst + kBoxBytes, map, &bars->full[st], 64, n0, zk);
                ++u;
            };
            int idx = blockIdx.x;
            load_q(0, idx);
            for (int k = 0; ok && idx >= 0; ++k) {
                const Item it = make_item(p, idx);
                claim(k + 1);   // one item ahead: its Q is loaded during this one
                int next = -1;
                const int zk = it.b * p.Hkv + it.g;
                // K(0), V(0), K(1), V(1), ...; the next item's Q after the fourth load, by
                // which time the MMA thread has moved on to this item
                const int n_loads = 2 * it.n_tiles;
                const int q_at = min(3, n_loads - 1);
                for (int l = 0; l < n_loads && ok; ++l) {
                    const int n0 = (it.kt_first + (l >> 1)) * kBN;
                    put((l & 1) ? &tmV : &tmK, n0, zk);
                    if (l == q_at && ok) {
                        next = read_item(bars, k + 1, p.n_items, ok);
                        if (!ok) set_timeout(p.status, kDiagPrefill, kRoleProducer, 3, k + 1);
                        if (next >= 0) load_q(k + 1, next);
                    }
                }
                idx = next;
            }
            if (!ok) {
                // never leave the CTA with copies in flight
                for (int w = max(0, u - kSlots); w < u; ++w)
                    mbar_wait(&bars->full[w % kSlots], (w / kSlots) & 1);
                for (int k = max(0, q_issued - 2); k < q_issued; ++k)
                    mbar_wait(&bars->q_full[k & 1], (k >> 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
            const uint32_t idesc_o = idesc_bf16_f32(kBM, kD, 0, 1);
            const uint32_t ring0 = smem_u32(smem + kSmemRing);
            bool ok = true;
            int u = 0;                 // ring slots consumed
            int cpv[2] = {0, 0};       // PV products issued, per query tile (all items)
            int nepi[2] = {0, 0};      // items finished, per query tile
            auto take = [&](int &st) {
                st = u % kSlots;
                if (!(ok = mbar_wait(&bars->full[st], (u / kSlots) & 1))) {
                    set_timeout(p.status, kDiagPrefill, kRoleMma, 1, u);
                    return;
                }
                ++u;
                tc_fence_after();
            };
            // a K tile: landed (or, fused-K form, rotated by warps 2-3: K tile kc of this
            // CTA signals krot[kc & 1])
            int kc = 0;
            auto take_k = [&](int &st) {
                if constexpr (!KROT) {
                    take(st);
                } else {
                    st = u % kSlots;
                    if (!(ok = mbar_wait(&bars->krot[kc & 1], (kc >> 1) & 1))) {
                        set_timeout(p.status, kDiagPrefill, kRoleMma, 7, kc);
                        return;
                    }
                    ++u;
                    ++kc;
                    tc_fence_after();
                }
            };
            auto issue_s = [&](uint32_t qaddr, int i, int st) {
                const uint32_t ka = ring0 + st * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    umma_ss(tmem + i * 128, sdesc_sw128(qaddr + off, 16, 1024),
                            sdesc_sw128(ka + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bars->s_full[i]);
            };
            auto issue_pv = [&](int i, int st, bool acc) {
                const uint32_t va = ring0 + st * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    umma_ts(tmem + 256 + i * 128, tmem + i * 128 + kk * 8,
                            sdesc_sw128(va + kk * 16 * 128, kBoxBytes, 1024), idesc_o,
                            (acc || kk > 0) ? 1u : 0u);
                }
                umma_commit(&bars->o_done[i]);
                ++cpv[i];
            };
            // waits until PV product number cpv[i] - 1 of tile i has completed
            auto wait_last_pv = [&](int i, int where) {
                if (cpv[i] > 0 && !(ok = mbar_wait(&bars->o_done[i], (cpv[i] - 1) & 1)))
                    set_timeout(p.status, kDiagPrefill, kRoleMma, where, cpv[i]);
                tc_fence_after();
            };
            for (int k = 0, idx = blockIdx.x; ok && idx >= 0; ++k) {
                const Item it = make_item(p, idx);
                const int buf = k & 1, ntile = it.two ? 2 : 1, n = it.n_tiles;
                const uint32_t qaddr[2] = {smem_u32(sQ(buf, 0)), smem_u32(sQ(buf, 1))};
                if (!(ok = mbar_wait(&bars->q_ready[buf], (k >> 1) & 1))) {
                    set_timeout(p.status, kDiagPrefill, kRoleMma, 0, k);
                    break;
                }
                tc_fence_after();
                int kst = 0, vst = 0;
                take_k(kst);
                for (int i = 0; i < ntile && ok; ++i) {
                    // S_i(0) overwrites the columns the previous item's last P_i sits in
                    wait_last_pv(i, 2);
                    if (ok) issue_s(qaddr[i], i, kst);
                }
                if (!ok) break;
                umma_commit(&bars->empty[kst]);
                int kprev = kst;   // K slot of the last score products issued
                for (int j = 0; j < n && ok; ++j) {
                    take(vst);
                    for (int i = 0; i < ntile && ok; ++i) {
                        if (!(ok = mbar_wait(&bars->p_full[i], cpv[i] & 1))) {
                            set_timeout(p.status, kDiagPrefill, kRoleMma, 3, cpv[i]);
                            break;
                        }
                        // the first PV of an item overwrites O_i: the previous item's
                        // epilogue must have read it out
                        if (j == 0 && nepi[i] > 0 &&
                            !(ok = mbar_wait(&bars->o_free[i], (nepi[i] - 1) & 1))) {
                            set_timeout(p.status, kDiagPrefill, kRoleMma, 4, nepi[i]);
                            break;
                        }
                        tc_fence_after();
                        issue_pv(i, vst, j > 0);
                        if (j == n - 1) umma_commit(&bars->o_final[i]);
                        if (j + 1 < n) {
                            if (i == 0) take_k(kst);
                            if (!ok) break;
                            // S_i(j+1) overwrites the columns P_i(j) sits in
                            wait_last_pv(i, 5);
                            // PV_i(j) has completed, and with it every earlier product of
                            // this thread: K(j) (read by S_0(j) and S_1(j)) is free once
                            // PV_0(j) is, V(j) once the last tile's PV(j) is.  Plain arrivals
                            // here cost the issuing thread less than commits.
                            if (i == 0 && j > 0) mbar_arrive(&bars->empty[kprev]);
                            if (i == ntile - 1) mbar_arrive(&bars->empty[vst]);
                            if (ok) issue_s(qaddr[i], i, kst);
                        } else {
                            // the item's last key tile: K and V go free when its products do
                            if (i == 0 && j > 0) umma_commit(&bars->empty[kprev]);
                            if (i == ntile - 1) umma_commit(&bars->empty[vst]);
                        }
                    }
                    kprev = kst;
                }
                if (!ok) break;
                for (int i = 0; i < ntile; ++i) ++nepi[i];
                idx = read_item(bars, k + 1, p.n_items, ok);
                if (!ok) {
                    set_timeout(p.status, kDiagPrefill, kRoleMma, 6, k + 1);
                    break;
                }
                mbar_arrive(&bars->item_free[item_slot(k + 1)]);
            }
            if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            // every tcgen05 operation issued above completes before TMEM is released
            umma_commit(&bars->mma_done);
            mbar_wait(&bars->mma_done, 0);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ================= RoPE on Q tiles (and fused-K K tiles); O stores =================
        // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7); the pair
        // (j, j + 64) is the same offset in box 0 and box 1
        const int rt = threadIdx.x - 64;   // 0..63
        // rotates the 128 rows of a tile in shared memory, row r at position pos0 + r (rows
        // at or past position S hold the load's zero fill and are left alone)
        auto rotate_tile = [&](uint8_t *tile, int pos0) {
            for (int rr = 0; rr < kBM / kRotThreads; ++rr) {
                const int r = rt + kRotThreads * rr;
                const int pos = pos0 + r;
                if (pos >= p.S) continue;
                const float4 *t4 = reinterpret_cast<const float4 *>(p.table + (size_t)pos * (kD / 2));
                uint8_t *row0 = tile + r * 128;
                uint8_t *row1 = row0 + kBoxBytes;
#pragma unroll 2
                for (int c = 0; c < 8; ++c) {
                    const int pc = (c ^ (r & 7)) * 16;
                    const uint4 a = *reinterpret_cast<uint4 *>(row0 + pc);
                    const uint4 bq = *reinterpret_cast<uint4 *>(row1 + pc);
                    float cs[16];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const float4 tv = __ldg(t4 + 4 * c + qq);
                        cs[4 * qq] = tv.x;
                        cs[4 * qq + 1] = tv.y;
                        cs[4 * qq + 2] = tv.z;
                        cs[4 * qq + 3] = tv.w;
                    }
                    uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {bq.x, bq.y, bq.z, bq.w};
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const float a0 = bf16lo(aw[qq]), a1 = bf16hi(aw[qq]);
                        const float b0 = bf16lo(bw[qq]), b1 = bf16hi(bw[qq]);
                        const float c0 = cs[4 * qq], s0 = cs[4 * qq + 1];
                        const float c1 = cs[4 * qq + 2], s1 = cs[4 * qq + 3];
                        aw[qq] = pack_bf16x2(fmaf(a0, c0, -b0 * s0), fmaf(a1, c1, -b1 * s1));
                        bw[qq] = pack_bf16x2(fmaf(a0, s0, b0 * c0), fmaf(a1, s1, b1 * c1));
                    }
                    *reinterpret_cast<uint4 *>(row0 + pc) = make_uint4(aw[0], aw[1], aw[2], aw[3]);
                    *reinterpret_cast<uint4 *>(row1 + pc) = make_uint4(bw[0], bw[1], bw[2], bw[3]);
                }
            }
        };
        int ku = 0;   // fused-K form: ring loads of the items so far
        int kc = 0;   // fused-K form: K tiles rotated
        int nst[2][2] = {{0, 0}, {0, 0}};   // staged completions consumed, [buffer][tile]
        // stores item kk's O (the plain form; the fused-K form stores from the epilogue):
        // waits until the epilogue has staged its tiles in Q buffer kk & 1, one TMA store
        // per 64-column box, and frees the buffer once the stores have read it
        auto store_o = [&](int kk, const Item &itp) {
            const int nt = itp.two ? 2 : 1;
            for (int t = 0; t < nt; ++t) {
                if (!warp_wait(&bars->staged[kk & 1][t], nst[kk & 1][t] & 1)) {
                    set_timeout(p.status, kDiagPrefill, kRoleRope, 3, kk);
                    return false;
                }
                ++nst[kk & 1][t];
            }
            if (lane == 0) {
                for (int t = 0; t < nt; ++t) {
                    const int zo = itp.b * p.Hq + itp.h0 + t;
                    tma_store_3d(&tmO, sQ(kk & 1, t), 0, itp.mb * kBM, zo);
                    tma_store_3d(&tmO, sQ(kk & 1, t) + kBoxBytes, 64, itp.mb * kBM, zo);
                }
                bulk_commit_group();
                bulk_wait_read_all();
                mbar_arrive_cnt(&bars->epi_done[kk & 1], 2);
            }
            __syncwarp();
            return true;
        };
        Item prev{};
        int k = 0;
        bool rok = true;
        for (int idx = blockIdx.x; rok && idx >= 0; ++k) {
            const Item it = make_item(p, idx);
            const int buf = k & 1;
            if (!warp_wait(&bars->q_full[buf], (k >> 1) & 1)) {
                set_timeout(p.status, kDiagPrefill, kRoleRope, 0, k);
                rok = false;
                break;
            }
            for (int i = 0; i < (it.two ? 2 : 1); ++i)
                rotate_tile(sQ(buf, i), p.S - p.T + it.mb * kBM);
            fence_proxy_async_smem();
            mbar_arrive(&bars->q_ready[buf]);
            if constexpr (KROT) {
                // this item's K tiles, ring loads ku, ku + 2, ... (K and V alternate), each
                // rotated at its keys' positions as soon as it lands
                for (int j = 0; j < it.n_tiles; ++j) {
                    const int u = ku + 2 * j, st = u % kSlots;
                    if (!warp_wait(&bars->full[st], (u / kSlots) & 1)) {
                        set_timeout(p.status, kDiagPrefill, kRoleRope, 2, kc);
                        rok = false;
                        break;
                    }
                    rotate_tile(smem + kSmemRing + st * kTileBytes, (it.kt_first + j) * kBN);
                    fence_proxy_async_smem();
                    mbar_arrive(&bars->krot[kc & 1]);
                    ++kc;
                }
                ku += 2 * it.n_tiles;
                if (!rok) break;
            } else if (warp == 2 && k >= 1 && !(rok = store_o(k - 1, prev))) {
                break;
            }
            prev = it;
            idx = __shfl_sync(0xffffffffu, read_item(bars, k + 1, p.n_items, rok), 0);
            if (!__all_sync(0xffffffffu, rok)) {
                set_timeout(p.status, kDiagPrefill, kRoleRope, 1, k + 1);
                rok = false;
                break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->item_free[item_slot(k + 1)]);
        }
        // the last item's O; every store completes before the CTA exits
        if (!KROT && warp == 2 && rok && k >= 1) store_o(k - 1, prev);
        if (warp == 2 && lane == 0) bulk_wait_all();
    }
    } else {
        reg_alloc<200>();
        // ================= softmax / epilogue =================
        const int wg = (warp - 4) >> 2;      // query tile
        const int r = (warp & 3) * 32 + lane;  // row in tile == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + wg * 128;
        const uint32_t tO = tmem + lane_off + 256 + wg * 128;
        int cs = 0;    // score tiles consumed (all items)
        int pvb = 0;   // PV products of the previous items
        int ne = 0;    // items finished
        int nsb[2] = {0, 0};   // items finished per Q buffer
        bool ok = true;
        for (int k = 0, idx = blockIdx.x; ok && idx >= 0; ++k) {
            // the item after this one (read at the end of the loop body)
            auto advance = [&]() {
                bool rok = true;
                const int nx = __shfl_sync(0xffffffffu, read_item(bars, k + 1, p.n_items, rok), 0);
                if (!__all_sync(0xffffffffu, rok)) {
                    set_timeout(p.status, kDiagPrefill, kRoleSoftmax, 4, k + 1);
                    ok = false;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->item_free[item_slot(k + 1)]);
                idx = nx;
            };
            int n_tiles, kt_first, qpos;
            {
                const Item it = make_item(p, idx);
                if (wg == 1 && !it.two) {
                    advance();
                    continue;
                }
                n_tiles = it.n_tiles;
                kt_first = it.kt_first;
                qpos = p.S - p.T + it.mb * kBM + r;
            }
            const bool valid = qpos < p.S;   // the row exists (t < T)
            float m = -CUDART_INF_F, l = 0.f;
            for (int j = 0; j < n_tiles; ++j) {
                if (!warp_wait(&bars->s_full[wg], cs & 1)) {
                    set_timeout(p.status, kDiagPrefill, kRoleSoftmax, 0, cs);
                    ok = false;
                    break;
                }
                ++cs;
                tc_fence_after();
                const int n0 = (kt_first + j) * kBN;
                const bool full = valid && (n0 + kBN - 1 <= qpos) &&
                                  (p.window <= 0 || n0 >= qpos - p.window + 1);
                // visible columns of this row in the tile: [c_lo, c_hi)
                int c_lo = 0, c_hi = kBN;
                if (!full) {
                    c_hi = valid ? min(kBN, qpos - n0 + 1) : 0;
                    c_lo = p.window > 0 ? max(0, qpos - p.window + 1 - n0) : 0;
                }
                // Masking, decided per warp and 32-column chunk, applied in tensor memory
                // before the row is loaded: a chunk visible in all 32 rows of the warp is
                // left alone; one hidden in all of them gets -inf and is skipped below (P = 0,
                // no exponentials); a mixed one is masked element by element.  The loop over
                // chunks is not unrolled (one copy of the code, taken on two tiles per item).
                uint32_t dead = 0;   // chunks hidden in every row of the warp
                if (!__all_sync(0xffffffffu, full)) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        const bool vis = c_lo <= 32 * c && 32 * c + 32 <= c_hi;
                        const bool hid = c_hi <= 32 * c || 32 * c + 32 <= c_lo || c_hi <= c_lo;
                        if (__all_sync(0xffffffffu, vis)) continue;
                        uint32_t rr[32];
                        if (__all_sync(0xffffffffu, hid)) {
                            dead |= 1u << c;
#pragma unroll
                            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(-CUDART_INF_F);
                        } else {
                            tmem_ld32(tS + 32 * c, rr);
                            tmem_wait_ld();
                            const int lo = c_lo - 32 * c, hi = c_hi - 32 * c;
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (i < lo || i >= hi) rr[i] = __float_as_uint(-CUDART_INF_F);
                        }
                        tmem_st32(tS + 32 * c, rr);
                    }
                    tmem_wait_st();
                }
                // the whole S row in registers: four loads in flight, one wait
                float x[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tS + 32 * c, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(rr[i]);
                }
                tmem_wait_ld();
                // row maximum of the raw scores: 3-input max, 8 independent chains of 16
                float mx8[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mx8[kk] = fmax3(x[kk], x[kk + 8], x[kk + 16]);
#pragma unroll
                    for (int tt = 3; tt < 15; tt += 2)
                        mx8[kk] = fmax3(mx8[kk], x[kk + 8 * tt], x[kk + 8 * tt + 8]);
                    mx8[kk] = fmaxf(mx8[kk], x[kk + 120]);
                }
                const float mraw = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                         fmaxf(mx8[6], mx8[7]));
                const float mx = mraw * p.scale_log2;   // scale > 0: max commutes with it
                const float m_new = fmaxf(m, mx);
                const bool grow = m_new > m + kRescaleThreshold;  // false while both -inf
                const bool need_o = grow && j > 0 && m != -CUDART_INF_F;
                const float f = grow ? ex2_approx(m - m_new) : 1.0f;  // 0 when m was -inf
                if (grow) {
                    l *= f;
                    m = m_new;
                }
                const float nmref = (m == -CUDART_INF_F) ? 0.f : -m;
                // P = 2^(s * scale * log2e - m) as bf16 over the first 64 columns of the S
                // tile, 16 columns at a time (each piece lands on columns already read);
                // packed fp32x2 FMA / add, row sum in 4 pairs of chains
                float2 ls[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
                    if (dead & (1u << c)) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[i] = 0u;
                        tmem_st16(tS + 16 * c, pk);
                        continue;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 a = ffma2(make_float2(x[32 * c + 2 * i], x[32 * c + 2 * i + 1]),
                                               p.scale_log2, nmref);
                        float e0, e1;
                        if ((kPolyPairs >> i) & 1) {
                            const float2 e = ex2_fma2(a);
                            e0 = e.x;
                            e1 = e.y;
                        } else {
                            e0 = ex2_approx(a.x);
                            e1 = ex2_approx(a.y);
                        }
                        ls[i & 3] = fadd2(ls[i & 3], make_float2(e0, e1));
                        pk[i] = pack_bf16x2(e0, e1);
                    }
                    tmem_st16(tS + 16 * c, pk);
                }
                l += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) +
                     ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
                if (__any_sync(0xffffffffu, need_o)) {
                    // O holds the product of tiles < j (already complete: S_i(j) was
                    // issued after PV_i(j-1) finished); rescale it in TMEM before this
                    // tile's PV is issued
                    if (!warp_wait(&bars->o_done[wg], (pvb + j - 1) & 1)) {
                        set_timeout(p.status, kDiagPrefill, kRoleSoftmax, 1, pvb + j);
                        ok = false;
                    }
                    tc_fence_after();
                    const float fo = need_o ? f : 1.0f;
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t rr[32];
                        tmem_ld32(tO + 32 * c, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            rr[i] = __float_as_uint(__uint_as_float(rr[i]) * fo);
                        tmem_st32(tO + 32 * c, rr);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars->p_full[wg]);
                if (!ok) break;
            }
            if (!ok) break;
            pvb += n_tiles;
            // ---- epilogue: O out of TMEM first (frees it for the next item); O / l as
            // bf16 into this item's Q buffer (every score product has completed, so the
            // buffer is free), in the 128-byte-swizzled layout of a Q tile; one TMA store
            // per 64-column box writes it out (rows past T are clipped by the tensor map)
            if (!warp_wait(&bars->o_final[wg], ne & 1)) {
                set_timeout(p.status, kDiagPrefill, kRoleSoftmax, 2, ne);
                ok = false;
                break;
            }
            tc_fence_after();
            {
                float x[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tO + 32 * c, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(rr[i]);
                }
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bars->o_free[wg]);
                const float inv_l = l > 0.f ? 1.0f / l : 0.f;
                uint8_t *stage = sQ(k & 1, wg) + r * 128;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<uint4 *>(stage + (c >> 3) * kBoxBytes +
                                               (((c & 7) ^ (r & 7)) << 4)) =
                        make_uint4(pack_bf16x2(x[8 * c] * inv_l, x[8 * c + 1] * inv_l),
                                   pack_bf16x2(x[8 * c + 2] * inv_l, x[8 * c + 3] * inv_l),
                                   pack_bf16x2(x[8 * c + 4] * inv_l, x[8 * c + 5] * inv_l),
                                   pack_bf16x2(x[8 * c + 6] * inv_l, x[8 * c + 7] * inv_l));
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->staged[k & 1][wg]);
            const Item it = make_item(p, idx);
            if (KROT && r == 0) {
                // fused-K form: the RoPE warp is busy with K tiles, the epilogue stores
                if (!mbar_wait(&bars->staged[k & 1][wg], nsb[k & 1] & 1)) {
                    set_timeout(p.status, kDiagPrefill, kRoleSoftmax, 3, ne);
                    ok = false;
                } else {
                    const int zo = it.b * p.Hq + it.h0 + wg;
                    tma_store_3d(&tmO, sQ(k & 1, wg), 0, it.mb * kBM, zo);
                    tma_store_3d(&tmO, sQ(k & 1, wg) + kBoxBytes, 64, it.mb * kBM, zo);
                    bulk_commit_group();
                    bulk_wait_read_all();
                    // the buffer's second arrival comes from tile 1, or from here if the
                    // item has no tile 1
                    mbar_arrive_cnt(&bars->epi_done[k & 1], it.two ? 1 : 2);
                }
            }
            ++ne;
            ++nsb[k & 1];
            if (valid && p.lse) {
                const int t = it.mb * kBM + r;
                p.lse[((size_t)it.b * p.Hq + it.h0 + wg) * p.T + t] =
                    (m + __log2f(l)) * 0.69314718055994531f;
            }
            advance();
        }
        // the O stores complete before the CTA exits
        if (r == 0) bulk_wait_all();
        if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against
// libcuda at build time).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [rows, inner] bf16 slabs: dims {d, rows, slabs}, box {64, 128, 1}, 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, int d, int rows, int slabs) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)slabs};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * rows};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_prefill(const void *q, const void *k_rot, const void *v, void *o, float *lse, int B,
                   int T, int S, int Hq, int Hkv, int d, int window, float scale,
                   const float *table, int table_len, int *status, cudaStream_t s, bool fuse_k) {
    (void)table_len;
    if (d != kD) return GQA_ERR_UNSUPPORTED;
    if (!fuse_k) {
        // long items (a causal sweep over a long sequence): one CTA per item
        const int n_mb = (T + kBM - 1) / kBM;
        long tiles = 0;
        for (int mb = 0; mb < n_mb; ++mb) {
            const int q_lo = S - T + mb * kBM, q_hi = (q_lo + kBM - 1 < S - 1) ? q_lo + kBM - 1 : S - 1;
            const int kt0 = window > 0 ? (q_lo - window + 1 > 0 ? q_lo - window + 1 : 0) / kBN : 0;
            tiles += q_hi / kBN - kt0 + 1;
        }
        if (tiles >= (long)kStreamMinTiles * n_mb)
            return launch_prefill_stream(q, k_rot, v, o, lse, B, T, S, Hq, Hkv, d, window, scale,
                                         table, status, s);
    }
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, q, d, T, B * Hq) || !make_map(&mk, k_rot, d, S, B * Hkv) ||
        !make_map(&mv, v, d, S, B * Hkv) || !make_map(&mo, o, d, T, B * Hq))
        return GQA_ERR_CUDA;
    auto kern = fuse_k ? prefill_persistent_kernel<true> : prefill_persistent_kernel<false>;
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), kSmemBytes) != cudaSuccess)
        return GQA_ERR_CUDA;   // the error stays readable with cudaGetLastError
    Params p;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.table = reinterpret_cast<const float2 *>(table);
    p.status = status;
    p.T = T;
    p.S = S;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.window = window;
    p.n_mblocks = (T + kBM - 1) / kBM;
    p.n_pairs = (p.G + 1) / 2;
    p.scale_log2 = scale * 1.4426950408889634f;
    const long n_items = (long)B * Hkv * p.n_pairs * p.n_mblocks;
    if (n_items > 0x7fffffffL) return GQA_ERR_UNSUPPORTED;
    p.n_items = static_cast<int>(n_items);
    // one CTA per item; the CTAs that get an SM first claim the rest (cluster launch control)
    kern<<<static_cast<unsigned>(n_items), kThreads, kSmemBytes, s>>>(mq, mk, mv, mo, p);
    const cudaError_t e = cudaPeekAtLastError();
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
