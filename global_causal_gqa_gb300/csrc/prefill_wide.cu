// prefill_wide.cu -- causal / sliding-window GQA prefill for d = 256 heads on tcgen05
// tensor cores (d = 512 runs on a pair of CTAs, prefill_pair.cu).
//
// Same computation as prefill.cu ("PLaMo 3アーキテクチャ徹底解析" §4.5, §5.1; the
// Gemma-4 local layers of the qiita.com Gemma-4-26B-A4B explainer, Attention block
// section), for heads too wide for two query tiles to share tensor memory: a 128 x 256
// fp32 output tile takes half of the 512 TMEM columns.
//
// CTA = (batch, query head, 128-row query block).  One query tile per CTA;
// its score tile S (128 keys) is double-buffered in TMEM so that S(j+2) = Q K(j+2)^T can
// run on the tensor core while the softmax warps work on S(j+1).  TMEM: S_a, S_b (128
// columns each) and O (the CTA's 256 output columns).  K (128-dim chunks of a key tile)
// and V (128-dim halves of the CTA's output columns) stream through one ring of 32 KB
// slots, loaded by TMA (128-byte swizzle) in exactly the order the MMA thread uses them:
// K(0), K(1), then V(j), K(j + 2) for j = 0, 1, ...; Q 64 KB + 5 ring slots.
// (The kernel is written for a head of D dims with DV output columns per CTA; it is
// instantiated for D = DV = 256 only.)
// Warps: 0 TMA producer, 1 TMEM owner + MMA issuer, 2-3 idle, 4-7 softmax/epilogue (one
// thread per query row).  Q is rotated (RoPE) in shared memory after it lands, by all 8
// warps, while the first K tiles load; pairs (j, j + d/2) sit at the same offset of boxes
// k and k + d/128.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kBM = 128;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct Wide;

template <>
struct Wide<256> {
    static constexpr int BN = 128, DV = 256, NS = 5;
};
constexpr int kSlotBytes = 128 * 256;   // 128 rows x 128 bf16 (two 64-column TMA boxes)
constexpr int kMaxSlots = 5;

struct WBars {
    uint64_t q_full, q_ready;
    uint64_t t_full;          // the Q rows' RoPE table rows, staged in ring slots 1..4
    uint64_t full[kMaxSlots], empty[kMaxSlots];
    uint64_t s_full[2], p_full[2], o_done, mma_done;
    // the last PV product: S(j+2) waits only for PV(j), so when the softmax finishes the
    // last tile PV(n-2) may still run and o_done can be two phases behind -- its parity
    // would then already read as "done" for PV(n-1)
    uint64_t o_final;
    uint64_t staged;          // O rows written to the shared-memory staging area
    uint32_t tmem_base;
};
static_assert(sizeof(WBars) <= 256, "barrier block");

struct WParams {
    __nv_bfloat16 *o;
    float *lse;
    const float2 *table;
    int *status;
    int T, S, Hq, Hkv, G, window;
    int n_mblocks, n_slices;
    float scale_log2;
};

__device__ __forceinline__ bool warp_wait_w(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, const WParams p) {
    constexpr int BN = Wide<D>::BN, DV = Wide<D>::DV, NS = Wide<D>::NS;
    constexpr int NKC = D / 128;                  // 128-dim K chunks per key tile
    constexpr int NVH = DV / 128;                 // 128-dim V halves per key tile
    constexpr int QBOX = kBM * 128;               // 128 rows x 64 bf16
    constexpr int QBYTES = (D / 64) * QBOX;
    constexpr int BOX = BN * 128;                 // BN rows x 64 bf16
    constexpr int OFF_RING = QBYTES;
    constexpr int OFF_BAR = OFF_RING + NS * kSlotBytes;
    constexpr uint32_t TS0 = 0, TS1 = BN, TO = 2 * BN;
    static_assert(BN == 128 && 2 * BOX == kSlotBytes && NS <= kMaxSlots, "ring layout");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    WBars *bars = reinterpret_cast<WBars *>(smem + OFF_BAR);
    uint8_t *sQ = smem;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int idx = blockIdx.x;
    const int slice = idx % p.n_slices;
    idx /= p.n_slices;
    const int h = idx % p.Hq;
    idx /= p.Hq;
    const int mb = p.n_mblocks - 1 - (idx % p.n_mblocks);   // longest rows first
    const int b = idx / p.n_mblocks;
    const int g = h / p.G;
    const int q_lo = p.S - p.T + mb * kBM;
    const int q_hi = min(q_lo + kBM - 1, p.S - 1);
    const int kt_first = p.window > 0 ? max(0, q_lo - p.window + 1) / BN : 0;
    const int n_tiles = q_hi / BN - kt_first + 1;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->t_full, 1);
        mbar_init(&bars->q_ready, kThreads);
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bars->full[i], 1);
            mbar_init(&bars->empty[i], 1);
        }
        mbar_init(&bars->s_full[0], 1);
        mbar_init(&bars->s_full[1], 1);
        mbar_init(&bars->p_full[0], 128);
        mbar_init(&bars->p_full[1], 128);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->o_final, 1);
        mbar_init(&bars->staged, 128);
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

    // The ring sequence, shared by the producer and the MMA thread: K(0), K(1), then for
    // j = 0 .. n-1: V(j), and K(j + 2) if it exists; each K is NKC slots, each V is NVH.
    // Slot load u of the sequence: its tensor, its key tile and its 128 columns.
    const int n_k0 = NKC * min(2, n_tiles);      // the loads of K(0), K(1)
    const int n_pair = max(0, n_tiles - 2);      // tiles j with a K(j + 2) after V(j)
    const int n_loads = (NKC + NVH) * n_tiles;
    auto slot_load = [&](int u, const CUtensorMap *&map, int &jt, int &c0) {
        if (u < n_k0) {
            map = &tmK;
            jt = u / NKC;
            c0 = 128 * (u % NKC);
            return;
        }
        int v = u - n_k0, j, w;
        if (v < n_pair * (NKC + NVH)) {
            j = v / (NKC + NVH);
            w = v % (NKC + NVH);
        } else {
            v -= n_pair * (NKC + NVH);
            j = n_pair + v / NVH;
            w = v % NVH;
        }
        if (w < NVH) {
            map = &tmV;
            jt = j;
            c0 = slice * DV + 128 * w;
        } else {
            map = &tmK;
            jt = j + 2;
            c0 = 128 * (w - NVH);
        }
    };
    // producer state (warp 0, lane 0)
    int pu = 0;
    bool pok = true;
    // one 32 KB slot: rows of key tile jt, columns c0 .. c0 + 127 of K or V
    auto put = [&]() {
        const int st = pu % NS;
        if (pu >= NS && !(pok = mbar_wait(&bars->empty[st], ((pu / NS) - 1) & 1))) {
            set_timeout(p.status, kDiagPrefillWide, 0, 1, pu);
            return;
        }
        const CUtensorMap *map;
        int jt, c0;
        slot_load(pu, map, jt, c0);
        const int n0 = (kt_first + jt) * BN, zk = b * p.Hkv + g;
        uint8_t *dst = smem + OFF_RING + st * kSlotBytes;
        mbar_arrive_expect_tx(&bars->full[st], kSlotBytes);
        tma_load_3d(dst, map, &bars->full[st], c0, n0, zk);
        tma_load_3d(dst + BOX, map, &bars->full[st], c0 + 64, n0, zk);
        ++pu;
    };
    // The Q rows' table rows (positions q_lo .. q_hi, D/2 (cos, sin) pairs each: 128 KB at
    // D = 256) are staged by bulk copies in ring slots 1..4, which the K/V stream only
    // needs after the rotation: the rotation then reads them from shared memory instead of
    // waiting on L2 row by row.
    constexpr int kTabRowBytes = D * 4;
    static_assert(kBM * kTabRowBytes <= (NS - 1) * kSlotBytes, "table rows fit in the ring");
    const int n_tab_rows = q_hi - q_lo + 1;
    uint8_t *stab = smem + OFF_RING + kSlotBytes;
    if (warp == 0 && lane == 0) {
        // Q, the table rows and the first ring load, before the rotation below
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_arrive_expect_tx(&bars->q_full, QBYTES);
        for (int i = 0; i < D / 64; ++i)
            tma_load_3d(sQ + i * QBOX, &tmQ, &bars->q_full, 64 * i, mb * kBM, b * p.Hq + h);
        mbar_arrive_expect_tx(&bars->t_full, n_tab_rows * kTabRowBytes);
        for (int r0 = 0; r0 < n_tab_rows; r0 += 32)
            bulk_copy_g2s(stab + r0 * kTabRowBytes,
                          p.table + (size_t)(q_lo + r0) * (D / 2),
                          min(32, n_tab_rows - r0) * kTabRowBytes, &bars->t_full);
        if (n_loads > 0) put();   // slot 0; slots 1..4 once the rotation is done
    }

    // ================= RoPE on the Q tile, by every warp =================
    // Warp w takes rows QR w .. QR w + QR - 1, one row at a time: lane l rotates pairs
    // 64 bb + 2l, 64 bb + 2l + 1 of every 64-pair box bb against their partners D/2 later
    // (the same swizzled word of box bb + NB).  The table row is read from its staging in
    // the ring as NB 512-byte pieces, RIF rows at a time.
    {
        constexpr int NB = D / 128;               // 64-pair boxes in each half of a row
        constexpr int QR = kBM / (kThreads / 32);   // rows per warp
        constexpr int RIF = QR < 32 / NB ? QR : 32 / NB;   // rows whose table loads are in flight
        bool qok = warp_wait_w(&bars->q_full, 0) && warp_wait_w(&bars->t_full, 0);
        if (!qok) set_timeout(p.status, kDiagPrefillWide, 3, 8, 0);
        if (qok) {
            const float4 *t4 = reinterpret_cast<const float4 *>(stab);
            for (int r0 = 0; r0 < QR; r0 += RIF) {
                float4 tv[RIF][NB];
#pragma unroll
                for (int i = 0; i < RIF; ++i) {
                    const int row = QR * warp + r0 + i;
                    // rows past T hold zeros (the load's out-of-range fill): any table row
                    const int pos = min(p.S - p.T + mb * kBM + row, p.S - 1);
#pragma unroll
                    for (int bb = 0; bb < NB; ++bb)
                        tv[i][bb] = t4[(size_t)(pos - q_lo) * (D / 4) + 32 * bb + lane];
                }
#pragma unroll
                for (int i = 0; i < RIF; ++i) {
                    const int row = QR * warp + r0 + i;
                    const int off =
                        row * 128 + ((((lane >> 2) ^ (row & 7)) << 4) | ((lane & 3) << 2));
#pragma unroll
                    for (int bb = 0; bb < NB; ++bb) {
                        uint32_t *pa = reinterpret_cast<uint32_t *>(sQ + bb * QBOX + off);
                        uint32_t *pb = reinterpret_cast<uint32_t *>(sQ + (bb + NB) * QBOX + off);
                        const float4 t = tv[i][bb];   // (cos, sin) of the two pairs
                        const uint32_t aw = *pa, bw = *pb;
                        const float a0 = bf16lo(aw), a1 = bf16hi(aw);
                        const float b0 = bf16lo(bw), b1 = bf16hi(bw);
                        *pa = pack_bf16x2(fmaf(a0, t.x, -b0 * t.y), fmaf(a1, t.z, -b1 * t.w));
                        *pb = pack_bf16x2(fmaf(a0, t.y, b0 * t.x), fmaf(a1, t.w, b1 * t.z));
                    }
                }
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->q_ready);
    }

    if (warp == 0) {
        // ================= TMA producer: the rest of the ring =================
        if (lane == 0) {
            // the table rows in slots 1..4 have been read once every thread has arrived
            pok = mbar_wait(&bars->q_ready, 0);
            if (!pok) set_timeout(p.status, kDiagPrefillWide, 0, 2, 0);
            while (pok && pu < n_loads) put();
            if (!pok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            // never leave the CTA with copies in flight
            mbar_wait(&bars->q_full, 0);
            mbar_wait(&bars->t_full, 0);
            for (int w = max(0, pu - NS); w < pu; ++w) mbar_wait(&bars->full[w % NS], (w / NS) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(kBM, BN, 0, 0);
            const uint32_t idesc_o = idesc_bf16_f32(kBM, 128, 0, 1);
            const uint32_t qaddr = smem_u32(sQ);
            const uint32_t ring = smem_u32(smem + OFF_RING);
            bool ok = mbar_wait(&bars->q_ready, 0);
            if (!ok) set_timeout(p.status, kDiagPrefillWide, 1, 4, 0);
            tc_fence_after();
            int u = 0;
            // waits for the next ring slot; returns its shared-memory address
            auto take = [&](uint32_t &addr) {
                const int st = u % NS;
                if (!(ok = mbar_wait(&bars->full[st], (u / NS) & 1))) {
                    set_timeout(p.status, kDiagPrefillWide, 1, 0, u);
                    return -1;
                }
                tc_fence_after();
                addr = ring + st * kSlotBytes;
                return st;
            };
            auto issue_s = [&](int j) {
                const uint32_t dst = tmem + ((j & 1) ? TS1 : TS0);
                for (int c = 0; c < NKC && ok; ++c) {
                    uint32_t ka;
                    const int st = take(ka);
                    if (st < 0) break;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const int dk = 8 * c + kk;   // 16-dim step over the whole head
                        const uint64_t ad = sdesc_sw128(
                            qaddr + (dk >> 2) * QBOX + (dk & 3) * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(
                            ka + (kk >> 2) * BOX + (kk & 3) * 32, 16, 1024);
                        umma_ss(dst, ad, bd, idesc_s, (c > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(&bars->empty[st]);
                    ++u;
                }
                if (ok) umma_commit(&bars->s_full[j & 1]);
            };
            if (ok) issue_s(0);
            if (ok && n_tiles > 1) issue_s(1);
            for (int j = 0; j < n_tiles && ok; ++j) {
                // one barrier per S buffer: the softmax may finish S(j+1) before this wait,
                // never S(j+2) (issued below, after PV(j)), so no phase is skipped
                if (!(ok = mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1))) {
                    set_timeout(p.status, kDiagPrefillWide, 1, 5, j);
                    break;
                }
                tc_fence_after();
                const uint32_t pcol = tmem + ((j & 1) ? TS1 : TS0);
                for (int hh = 0; hh < NVH && ok; ++hh) {
                    uint32_t va;
                    const int st = take(va);
                    if (st < 0) break;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        umma_ts(tmem + TO + 128 * hh, pcol + kk * 8,
                                sdesc_sw128(va + kk * 2048, BOX, 1024), idesc_o,
                                (j > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&bars->empty[st]);
                    ++u;
                }
                if (!ok) break;
                umma_commit(&bars->o_done);
                if (j == n_tiles - 1) umma_commit(&bars->o_final);
                // S(j+2) reuses the TMEM buffer P(j) sits in: PV(j) must have finished
                // reading P(j) before the first S(j+2) product is written there
                if (j + 2 < n_tiles) {
                    if (!(ok = mbar_wait(&bars->o_done, j & 1))) {
                        set_timeout(p.status, kDiagPrefillWide, 1, 7, j);
                        break;
                    }
                    tc_fence_after();
                    issue_s(j + 2);
                }
            }
            if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            umma_commit(&bars->mma_done);
            mbar_wait(&bars->mma_done, 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ================= softmax / epilogue =================
        const int r = (warp & 3) * 32 + lane;   // row in tile == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int t = mb * kBM + r;
        const bool valid = t < p.T;
        const int qpos = p.S - p.T + t;
        bool ok = true;

        float m = -CUDART_INF_F, l = 0.f;
        for (int j = 0; j < n_tiles && ok; ++j) {
            if (!warp_wait_w(&bars->s_full[j & 1], (j >> 1) & 1)) {
                set_timeout(p.status, kDiagPrefillWide, 3, 6, j);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tS = tmem + lane_off + ((j & 1) ? TS1 : TS0);
            const int n0 = (kt_first + j) * BN;
            const bool full = valid && (n0 + BN - 1 <= qpos) &&
                              (p.window <= 0 || n0 >= qpos - p.window + 1);
            int c_lo = 0, c_hi = BN;
            if (!full) {
                c_hi = valid ? min(BN, qpos - n0 + 1) : 0;
                c_lo = p.window > 0 ? max(0, qpos - p.window + 1 - n0) : 0;
            }
            // Masking, decided per warp and 32-column chunk, applied in tensor memory
            // before the row is loaded: a chunk visible in all 32 rows of the warp is left
            // alone; one hidden in all of them gets -inf and is skipped below (P = 0, no
            // exponentials); a mixed one is masked element by element.  The chunk loop is
            // not unrolled (one copy of the code, taken on the window-edge and diagonal
            // tiles only).
            uint32_t dead = 0;   // chunks hidden in every row of the warp
            if (!__all_sync(0xffffffffu, full)) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
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
            float x[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t rr[32];
                tmem_ld32(tS + 32 * c, rr);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(rr[i]);
            }
            tmem_wait_ld();
            constexpr int CH = BN / 8;   // values per max chain
            float mx8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                mx8[k] = x[k];
#pragma unroll
                for (int tt = 1; tt < CH; ++tt) mx8[k] = fmaxf(mx8[k], x[k + 8 * tt]);
            }
            const float mraw = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                     fmaxf(mx8[6], mx8[7]));
            const float mx = mraw * p.scale_log2;
            const float m_new = fmaxf(m, mx);
            const bool grow = m_new > m + kRescaleThreshold;
            const bool need_o = grow && j > 0 && m != -CUDART_INF_F;
            const float f = grow ? ex2_approx(m - m_new) : 1.0f;
            if (grow) {
                l *= f;
                m = m_new;
            }
            const float nmref = (m == -CUDART_INF_F) ? 0.f : -m;
            float2 ls[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
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
                    const float e0 = ex2_approx(a.x), e1 = ex2_approx(a.y);
                    ls[i & 3] = fadd2(ls[i & 3], make_float2(e0, e1));
                    pk[i] = pack_bf16x2(e0, e1);
                }
                tmem_st16(tS + 16 * c, pk);
            }
            l += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) +
                 ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
            if (__any_sync(0xffffffffu, need_o)) {
                // O holds the product of tiles < j: wait for the last one, rescale in TMEM
                if (!warp_wait_w(&bars->o_done, (j - 1) & 1)) {
                    set_timeout(p.status, kDiagPrefillWide, 3, 7, j);
                    ok = false;
                }
                tc_fence_after();
                const float fo = need_o ? f : 1.0f;
#pragma unroll 1
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tmem + lane_off + TO + 32 * c, rr);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        rr[i] = __float_as_uint(__uint_as_float(rr[i]) * fo);
                    tmem_st32(tmem + lane_off + TO + 32 * c, rr);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full[j & 1]);
        }
        if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
        if (ok && warp_wait_w(&bars->o_final, 0)) {
            // O / l as bf16 into the Q buffer (every score product has completed), in the
            // 128-byte-swizzled layout of 64-column boxes; TMA stores write it out (rows
            // past T are clipped by the tensor map)
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_off + TO + 32 * c, rr);
                tmem_wait_ld();
                uint8_t *box = sQ + (c >> 1) * QBOX + r * 128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int cc = 4 * (c & 1) + q4;   // 16-byte chunk within the box row
                    *reinterpret_cast<uint4 *>(box + ((cc ^ (r & 7)) << 4)) = make_uint4(
                        pack_bf16x2(__uint_as_float(rr[8 * q4]) * inv_l,
                                    __uint_as_float(rr[8 * q4 + 1]) * inv_l),
                        pack_bf16x2(__uint_as_float(rr[8 * q4 + 2]) * inv_l,
                                    __uint_as_float(rr[8 * q4 + 3]) * inv_l),
                        pack_bf16x2(__uint_as_float(rr[8 * q4 + 4]) * inv_l,
                                    __uint_as_float(rr[8 * q4 + 5]) * inv_l),
                        pack_bf16x2(__uint_as_float(rr[8 * q4 + 6]) * inv_l,
                                    __uint_as_float(rr[8 * q4 + 7]) * inv_l));
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->staged);
            if (r == 0) {
                if (!mbar_wait(&bars->staged, 0)) {
                    set_timeout(p.status, kDiagPrefillWide, 3, 10, n_tiles);
                } else {
                    for (int bx = 0; bx < DV / 64; ++bx)
                        tma_store_3d(&tmO, sQ + bx * QBOX, slice * DV + 64 * bx, mb * kBM,
                                     b * p.Hq + h);
                    bulk_commit_group();
                    // the stores have read the staging area before the CTA (and its
                    // shared memory) ends; their writes complete on their own
                    bulk_wait_read_all();
                }
            }
            if (valid && p.lse && slice == 0)
                p.lse[((size_t)b * p.Hq + h) * p.T + t] = (m + __log2f(l)) * 0.69314718055994531f;
        } else if (ok) {
            set_timeout(p.status, kDiagPrefillWide, 3, 9, n_tiles);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
constexpr int wide_smem_bytes() {
    return (D / 64) * kBM * 128 + Wide<D>::NS * kSlotBytes + 256 + 1024;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_wide() {
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

// dims {d, rows, slabs}, box {64, box_rows, 1}, 128-byte swizzle
bool make_map_wide(CUtensorMap *map, const void *base, int d, int rows, int slabs, int box_rows) {
    EncodeTiledFn fn = encode_fn_wide();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)slabs};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * rows};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_wide(const void *q, const void *k_rot, const void *v, void *o, float *lse, int B,
                int T, int S, int Hq, int Hkv, int window, float scale, const float *table,
                int *status, cudaStream_t s) {
    constexpr int BN = Wide<D>::BN, DV = Wide<D>::DV;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map_wide(&mq, q, D, T, B * Hq, kBM) || !make_map_wide(&mk, k_rot, D, S, B * Hkv, BN) ||
        !make_map_wide(&mv, v, D, S, B * Hkv, BN) || !make_map_wide(&mo, o, D, T, B * Hq, kBM))
        return GQA_ERR_CUDA;
    constexpr int smem = wide_smem_bytes<D>();
    if (ensure_smem_attr(reinterpret_cast<const void *>(prefill_wide_kernel<D>), smem) !=
        cudaSuccess)
        return GQA_ERR_CUDA;
    WParams p;
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
    p.n_slices = D / DV;
    p.scale_log2 = scale * 1.4426950408889634f;
    const long nblocks = (long)B * Hq * p.n_mblocks * p.n_slices;
    prefill_wide_kernel<D><<<static_cast<unsigned>(nblocks), kThreads, smem, s>>>(mq, mk, mv, mo, p);
    return cudaPeekAtLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace

int launch_prefill_wide(const void *q, const void *k_rot, const void *v, void *o, float *lse,
                        int B, int T, int S, int Hq, int Hkv, int d, int window, float scale,
                        const float *table, int *status, cudaStream_t s) {
    // d = 512: a 128 x 512 fp32 output tile fills TMEM, so a pair of CTAs splits the
    // score and output roles (prefill_pair.cu)
    if (d == 256)
        return launch_wide<256>(q, k_rot, v, o, lse, B, T, S, Hq, Hkv, window, scale, table,
                                status, s);
    if (d == 512)
        return launch_prefill_pair(q, k_rot, v, o, lse, B, T, S, Hq, Hkv, window, scale, table,
                                   status, s);
    return GQA_ERR_UNSUPPORTED;
}

}  // namespace gqa
