// prefill_stream.cu -- the d = 128 prefill as one CTA per work item, for long causal
// sweeps.
//
// Same computation, work item, warp roles and tensor-memory layout as the persistent
// kernel in prefill.cu ("PLaMo 3アーキテクチャ徹底解析" §4.5, §5.1), but every item is its
// own CTA and the hardware hands CTAs to SMs as they free up.  When items are long (a
// causal layer over a long sequence: up to T/128 key tiles per item) the per-item fixed
// work is negligible, and the hardware's dynamic assignment balances the very uneven
// item lengths better than a static persistent schedule; the deeper K/V buffering (two
// stages of K and V) also suits a K/V stream that no longer fits in L2.
//
// CTA = (batch b, KV head g, pair of query heads of that group, block of 128 query rows).
// Both query tiles of a CTA sit at the same positions and read the same KV head, so they
// share every K and V tile load and the same mask.  Only key tiles that intersect
// [q_pos - W + 1, q_pos] for some row of the block are loaded (window tile skipping,
// §1 and §5.3: local prefill costs O(T W)); the per-element mask is applied on the tiles
// that straddle the diagonal or the window's lower edge only.
//
// Warp roles (12 warps, 3 warpgroups):
//   warp 0      TMA producer: Q tiles once, then K/V tiles into a 2-stage ring.
//   warp 1      tensor-memory allocator and the single MMA-issuing thread.
//   warps 2-3   idle (with 12 warps, 3 per SM sub-partition, every thread gets 168
//               registers; fewer warps would not raise that cap).
//   warps 4-7   softmax for query tile 0, warps 8-11 for query tile 1: one thread per
//               query row; warp w reads TMEM lanes 32*(w%4).. (its lane quarter).
// Q is rotated (RoPE, §6.1) in shared memory by the softmax warps right after it lands;
// K arrives already rotated (the caller-side pass rotates each key once).
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512).
// P (bf16) overwrites the first 64 columns of its S tile and feeds the PV product
// directly from tensor memory.  Rescaling of O is lazy: it happens only when a row's
// maximum grows by more than 2^8, otherwise the stale maximum is kept (exact, since O
// and the running sum always share one reference maximum).
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
constexpr int kStages = 2;
constexpr int kBoxBytes = 128 * 128;          // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kTileBytes = 2 * kBoxBytes;     // 128 rows x 128 bf16
constexpr int kSmemQ = 0;                     // two query tiles
constexpr int kSmemK = 2 * kTileBytes;
constexpr int kSmemV = kSmemK + kStages * kTileBytes;
constexpr int kSmemBar = kSmemV + kStages * kTileBytes;
constexpr int kSmemBytes = kSmemBar + 256 + 1024;  // + barriers + alignment slack
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;     // log2 units
// Column pairs (bit i: pair i of each 32-column chunk) whose exponentials run on the FMA
// pipe (ex2_fma2) instead of the special-function unit.  Off by default: the softmax is
// bound by instruction issue and latency, not by the special-function unit, so the
// extra instructions cost more than the offload saves (measured on GB300).
#ifndef GQA_PREFILL_POLY_PAIRS
#define GQA_PREFILL_POLY_PAIRS 0x0000u
#endif
constexpr uint32_t kPolyPairs = GQA_PREFILL_POLY_PAIRS;

struct Bars {
    uint64_t q_full;
    uint64_t q_ready[2];
    uint64_t k_full[kStages];
    uint64_t v_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_done[2];
    uint64_t mma_done;
    uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Params {
    __nv_bfloat16 *o;
    float *lse;
    const float2 *table;
    int *status;
    int T, S, Hq, Hkv, G, window;
    int n_mblocks, n_pairs;
    float scale_log2;
};

// A bounded wait whose outcome every lane of the warp agrees on, so the warp-collective
// tcgen05.ld/st that follow are never reached by only part of a warp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    Bars *bars = reinterpret_cast<Bars *>(smem + kSmemBar);
    uint8_t *sQ[2] = {smem + kSmemQ, smem + kSmemQ + kTileBytes};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- work item ----
    int idx = blockIdx.x;
    const int pair = idx % p.n_pairs;
    idx /= p.n_pairs;
    const int mb = p.n_mblocks - 1 - (idx % p.n_mblocks);  // longest rows first
    idx /= p.n_mblocks;
    const int g = idx % p.Hkv;
    const int b = idx / p.Hkv;
    const int h0 = g * p.G + 2 * pair;
    const bool two = (2 * pair + 1) < p.G;
    const int q_lo = p.S - p.T + mb * kBM;                   // position of row 0
    const int q_hi = min(q_lo + kBM - 1, p.S - 1);           // position of the last row
    const int kt_first = p.window > 0 ? max(0, q_lo - p.window + 1) / kBN : 0;
    const int kt_last = q_hi / kBN;
    const int n_tiles = kt_last - kt_first + 1;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->q_ready[i], 128);
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->p_full[i], 128);
            mbar_init(&bars->o_done[i], 1);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
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

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const int zq = b * p.Hq + h0;
            mbar_arrive_expect_tx(&bars->q_full, (two ? 2 : 1) * kTileBytes);
            for (int i = 0; i < (two ? 2 : 1); ++i) {
                tma_load_3d(sQ[i], &tmQ, &bars->q_full, 0, mb * kBM, zq + i);
                tma_load_3d(sQ[i] + kBoxBytes, &tmQ, &bars->q_full, 64, mb * kBM, zq + i);
            }
            const int zk = b * p.Hkv + g;
            bool ok = true;
            int issued = 0;
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j % kStages;
                if (j >= kStages && !mbar_wait(&bars->kv_empty[s], ((j / kStages) - 1) & 1)) {
                    set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
                    ok = false;
                    break;
                }
                const int n0 = (kt_first + j) * kBN;
                uint8_t *sK = smem + kSmemK + s * kTileBytes;
                uint8_t *sV = smem + kSmemV + s * kTileBytes;
                mbar_arrive_expect_tx(&bars->k_full[s], kTileBytes);
                tma_load_3d(sK, &tmK, &bars->k_full[s], 0, n0, zk);
                tma_load_3d(sK + kBoxBytes, &tmK, &bars->k_full[s], 64, n0, zk);
                mbar_arrive_expect_tx(&bars->v_full[s], kTileBytes);
                tma_load_3d(sV, &tmV, &bars->v_full[s], 0, n0, zk);
                tma_load_3d(sV + kBoxBytes, &tmV, &bars->v_full[s], 64, n0, zk);
                issued = j + 1;
            }
            // never leave the CTA with copies in flight
            mbar_wait(&bars->q_full, 0);
            for (int j = max(0, issued - kStages); j < issued; ++j) {
                mbar_wait(&bars->k_full[j % kStages], (j / kStages) & 1);
                mbar_wait(&bars->v_full[j % kStages], (j / kStages) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
            const uint32_t idesc_o = idesc_bf16_f32(kBM, kD, 0, 1);
            const uint32_t qaddr[2] = {smem_u32(sQ[0]), smem_u32(sQ[1])};
            const uint32_t kaddr0 = smem_u32(smem + kSmemK), vaddr0 = smem_u32(smem + kSmemV);
            const int ntile = two ? 2 : 1;
            bool ok = true;
            auto issue_s = [&](int i, int s) {
                const uint32_t ka = kaddr0 + s * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    umma_ss(tmem + i * 128, sdesc_sw128(qaddr[i] + off, 16, 1024),
                            sdesc_sw128(ka + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bars->s_full[i]);
            };
            auto issue_pv = [&](int i, int s, bool acc) {
                const uint32_t va = vaddr0 + s * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    umma_ts(tmem + 256 + i * 128, tmem + i * 128 + kk * 8,
                            sdesc_sw128(va + kk * 16 * 128, kBoxBytes, 1024), idesc_o,
                            (acc || kk > 0) ? 1u : 0u);
                }
                umma_commit(&bars->o_done[i]);
            };
            for (int i = 0; i < ntile && ok; ++i) ok = mbar_wait(&bars->q_ready[i], 0);
            tc_fence_after();
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j % kStages;
                const uint32_t par = (j / kStages) & 1;
                if (j == 0) {
                    if (!(ok = mbar_wait(&bars->k_full[s], par))) break;
                    tc_fence_after();
                    for (int i = 0; i < ntile; ++i) issue_s(i, s);
                }
                if (!(ok = mbar_wait(&bars->v_full[s], par))) break;
                const int s1 = (j + 1) % kStages;
                const uint32_t par1 = ((j + 1) / kStages) & 1;
                for (int i = 0; i < ntile && ok; ++i) {
                    if (!(ok = mbar_wait(&bars->p_full[i], j & 1))) break;
                    tc_fence_after();
                    issue_pv(i, s, j > 0);
                    if (j + 1 < n_tiles) {
                        if (i == 0 && !(ok = mbar_wait(&bars->k_full[s1], par1))) break;
                        // S_i(j+1) overwrites the TMEM columns P_i(j) sits in; the tensor
                        // pipe does not order that write after PV_i(j)'s read, so wait for
                        // PV_i(j) to complete first
                        if (!(ok = mbar_wait(&bars->o_done[i], j & 1))) break;
                        // with the last tile's PV(j), every product that read stage s has
                        // completed: a plain arrival frees it (cheaper than a commit)
                        if (i == ntile - 1) mbar_arrive(&bars->kv_empty[s]);
                        tc_fence_after();
                        issue_s(i, s1);
                    } else if (i == ntile - 1) {
                        umma_commit(&bars->kv_empty[s]);
                    }
                }
            }
            if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            // every tcgen05 operation issued above completes before TMEM is released
            umma_commit(&bars->mma_done);
            mbar_wait(&bars->mma_done, 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ================= softmax / epilogue =================
        const int wg = (warp - 4) >> 2;      // query tile
        const int r = (warp & 3) * 32 + lane;  // row in tile == TMEM lane
        const bool tile_on = (wg == 0) || two;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + wg * 128;
        const uint32_t tO = tmem + lane_off + 256 + wg * 128;
        const int t = mb * kBM + r;
        const bool valid = t < p.T;
        const int qpos = p.S - p.T + t;
        const int h = h0 + wg;
        bool ok = true;

        if (tile_on) {
            // ---- RoPE on the Q row in shared memory (128-byte swizzle: 16-byte chunk c of
            // row r sits at chunk c ^ (r & 7); pair (j, j + 64) = same offset in box 0 / 1)
            // the row's table entries are fetched while the Q tile is still in flight
            float4 tq[32];
            {
                const float4 *t4 = reinterpret_cast<const float4 *>(
                    p.table + (size_t)(valid ? qpos : 0) * (kD / 2));
#pragma unroll
                for (int i = 0; i < 32; ++i) tq[i] = __ldg(t4 + i);
            }
            ok = warp_wait(&bars->q_full, 0);
            if (ok && valid) {
                uint8_t *row0 = sQ[wg] + r * 128;
                uint8_t *row1 = row0 + kBoxBytes;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int pc = (c ^ (r & 7)) * 16;
                    uint4 a = *reinterpret_cast<uint4 *>(row0 + pc);
                    uint4 bq = *reinterpret_cast<uint4 *>(row1 + pc);
                    float cs[16];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const float4 tv = tq[4 * c + qq];
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
            fence_proxy_async_smem();
            mbar_arrive(&bars->q_ready[wg]);
        }

        float m = -CUDART_INF_F, l = 0.f;
        if (tile_on && ok) {
            for (int j = 0; j < n_tiles; ++j) {
                if (!warp_wait(&bars->s_full[wg], j & 1)) { ok = false; break; }
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
                if (!full) {
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        x[i] = (i >= c_lo && i < c_hi) ? x[i] : -CUDART_INF_F;
                }
                // row maximum of the raw scores: 3-input max, 8 independent chains of 16
                float mx8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    mx8[k] = fmax3(x[k], x[k + 8], x[k + 16]);
#pragma unroll
                    for (int t = 3; t < 15; t += 2)
                        mx8[k] = fmax3(mx8[k], x[k + 8 * t], x[k + 8 * t + 8]);
                    mx8[k] = fmaxf(mx8[k], x[k + 120]);
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
                    // O still holds the product of tiles < j: wait for the last one, then
                    // rescale it in TMEM before this tile's PV is issued.
                    if (!warp_wait(&bars->o_done[wg], (j - 1) & 1)) ok = false;
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
            if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            // ---- epilogue: O / l -> bf16, lse
            if (ok && warp_wait(&bars->o_done[wg], (n_tiles - 1) & 1)) {
                tc_fence_after();
                const float inv_l = l > 0.f ? 1.0f / l : 0.f;
                __nv_bfloat16 *orow = p.o + (((size_t)b * p.Hq + h) * p.T + t) * kD;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tO + 32 * c, rr);
                    tmem_wait_ld();
                    if (valid) {
                        uint32_t pkd[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pkd[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv_l,
                                                 __uint_as_float(rr[2 * i + 1]) * inv_l);
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2],
                                                pkd[4 * i + 3]);
                    }
                }
                if (valid && p.lse)
                    p.lse[((size_t)b * p.Hq + h) * p.T + t] =
                        (m + __log2f(l)) * 0.69314718055994531f;
            } else if (ok) {
                set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            }
        }
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

int launch_prefill_stream(const void *q, const void *k_rot, const void *v, void *o, float *lse,
                          int B, int T, int S, int Hq, int Hkv, int d, int window, float scale,
                          const float *table, int *status, cudaStream_t s) {
    if (d != kD) return GQA_ERR_UNSUPPORTED;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, d, T, B * Hq) || !make_map(&mk, k_rot, d, S, B * Hkv) ||
        !make_map(&mv, v, d, S, B * Hkv))
        return GQA_ERR_CUDA;
    if (ensure_smem_attr(reinterpret_cast<const void *>(prefill_kernel), kSmemBytes) !=
        cudaSuccess)
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
    const long nblocks = (long)B * Hkv * p.n_pairs * p.n_mblocks;
    prefill_kernel<<<static_cast<unsigned>(nblocks), kThreads, kSmemBytes, s>>>(mq, mk, mv, p);
    const cudaError_t e = cudaPeekAtLastError();
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace gqa
