// prefill_pair.cu -- causal / sliding-window GQA prefill for d = 512 heads on pairs of CTAs
// (two pairs per thread-block cluster), each score tile computed once.
//
// Same computation as prefill_wide.cu ("PLaMo 3アーキテクチャ徹底解析" §4.5, §5.1; the
// Gemma-4 global layer of the qiita.com Gemma-4-26B-A4B explainer, with the p-RoPE of
// §6.4).  A 128 x 512 fp32 output tile fills all 512 TMEM columns of an SM, so one CTA
// cannot hold it next to a score tile.  The pair splits the work by role:
//   S-CTA (cluster rank 0): the rotated Q tile lives in its TMEM (bf16, 256 columns) as the
//     A operand of S = Q K^T; K streams through a 5-slot ring of 32 KB (128 keys x 128
//     dims); S is double-buffered in TMEM (2 x 128 columns).  Its softmax warps turn S(j)
//     into P(j) (bf16, 128 x 128) plus one rescale factor per row, store them in one of two
//     local staging buffers in the layout the tensor core reads, and one bulk copy carries
//     the packet into one of the O-CTA's three receive buffers.  It owns the running max
//     and sum (and writes the log-sum-exp); at the end it sends the row sums.
//   O-CTA (cluster rank 1): the whole 128 x 512 fp32 O in TMEM; V streams through a 4-slot
//     ring of 32 KB (64 keys x 256 dims); O += P(j) V(j) with both operands in shared
//     memory, 256 output columns per MMA so that each P element is read once per 256
//     dims.  Four warps apply the rare lazy rescale of O rows before a PV product and
//     write O / l at the end.
// Per key tile each CTA issues the same tensor work (S: 32 MMAs of 128 x 128 x 16 over the
// 512 dims; PV: 16 of 128 x 256 x 16), so the pair executes exactly the counted work,
// where two CTAs that each own half of O would both compute the whole score tile.
//
// Two acknowledgements flow back to the S-CTA as remote mbarrier arrivals: "packet j
// received" (the O-CTA's warp 3, as soon as the copy has landed: staging buffer j & 1 is
// free for P(j + 2)) and "PV(j) finished" (the O-CTA's warp 2, forwarding the tensor
// core's completion: receive buffer j % 3 is free for packet j + 3).  Three receive
// buffers keep the loop packet -> PV -> acknowledgement -> next packet off the tensor
// pipe's critical path.
// A cluster holds two such pairs, for two query heads of one KV group (ranks 0, 1: their
// S-CTAs; 2, 3: their O-CTAs).  The two S-CTAs read the same K tiles and the two O-CTAs the
// same V tiles, so each chunk is loaded once and multicast to both: each CTA issues every
// other chunk of its ring, arms its own "full" barrier for every chunk, and a slot is
// reloaded once both CTAs' MMAs have released it (their completions are multicast onto
// both "empty" barriers).  This halves the L2-to-SM traffic of a key tile; a CTA alone
// could not keep its tensor pipe fed from 5 slots in flight.  With an odd group size the
// last pair computes its group's last head a second time and stores nothing.
// Every wait is bounded; the four CTAs meet at a cluster barrier before any exits, so no
// copy, multicast load or remote arrival targets the shared memory of a CTA that has
// finished.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kD = 512;
constexpr int kBM = 128;                  // query rows per pair
constexpr int kBN = 128;                  // keys per tile
constexpr int kThreads = 256;
constexpr int kNS_S = 5;                  // S-CTA ring slots
constexpr int kNS_O = 4;                  // O-CTA ring slots
constexpr int kBox = 128 * 128;           // 128 rows x 64 bf16 (one 128-byte-swizzled TMA box)
constexpr int kVBox = 64 * 128;           // 64 keys x 64 bf16
constexpr int kSlot = 2 * kBox;           // 32 KB: K 128 keys x 128 dims, V 64 keys x 256 dims
constexpr int kChunks = 4;                // ring loads per key tile (K or V)
constexpr int kPBytes = kBM * kBN * 2;    // P tile, bf16
constexpr int kFBytes = kBM * 4;          // rescale factors (or the final row sums), fp32
constexpr int kNR = 3;                    // O-CTA receive buffers
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// shared memory of the S-CTA: ring, 2 staging buffers (P, f), the row sums
constexpr int S_OFF_P = kNS_S * kSlot;
constexpr int S_OFF_F = S_OFF_P + 2 * kPBytes;
constexpr int S_OFF_L = S_OFF_F + 2 * kFBytes;
// shared memory of the O-CTA: ring, 3 receive buffers (P, f; the row sums land in the f
// slot of the buffer after the last packet)
constexpr int O_OFF_P = kNS_O * kSlot;
constexpr int O_OFF_F = O_OFF_P + kNR * kPBytes;
// the barrier block sits at the same offset in both
constexpr int OFF_BAR = 230912;
constexpr int kBarBytes = 320;
constexpr int kSmemBytes = OFF_BAR + kBarBytes + 1024;
static_assert(S_OFF_L + kFBytes <= OFF_BAR && O_OFF_F + kNR * kFBytes <= OFF_BAR, "layout");
static_assert(S_OFF_P % 1024 == 0 && O_OFF_P % 1024 == 0 && kPBytes % 1024 == 0,
              "P boxes are 1024-byte aligned");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// TMEM columns: S-CTA Q (bf16 pairs) and two score buffers; O-CTA all of O
constexpr uint32_t TQ = 0, TS0 = 256, TS1 = 384, TO = 0;

struct PBars {
    uint64_t full[kNS_S], empty[kNS_S];   // ring (both; the O-CTA uses kNS_O); empty: 2
    uint64_t q_rot;                   // S: Q rotated in shared memory (256 arrivals)
    uint64_t q_ready;                 // S: Q in TMEM (128)
    uint64_t s_full[2], s_free[2];    // S: score buffer written / read out (128)
    uint64_t p_staged[2];             // S: packet j stored in staging buffer j & 1 (128)
    uint64_t rack[2];                 // S: packet j landed in the O-CTA (remote)
    uint64_t pfree[kNR];              // S: PV(j) of receive buffer j % 3 done (remote)
    uint64_t l_staged;                // S: row sums stored (128)
    uint64_t p_full[kNR];             // O: packet (or the row sums) landed (transaction bytes)
    uint64_t o_ok[kNR];               // O: rows rescaled (or not needed) for packet j (128)
    uint64_t pv_done[kNR];            // O: PV(j) complete
    uint64_t o_final;                 // O: last PV complete
    uint64_t staged;                  // O: output rows staged for the TMA store (128)
    uint64_t mma_done;
    uint32_t tmem_base;
};
static_assert(sizeof(PBars) <= kBarBytes, "barrier block");

struct PairParams {
    float *lse;
    const float2 *table;
    int *status;
    int T, S, Hq, Hkv, G, window;
    int n_mblocks, n_hpairs;   // query blocks; head pairs per KV group, ceil(G / 2)
    float scale_log2;
};

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity));
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, const PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    PBars *bars = reinterpret_cast<PBars *>(smem + OFF_BAR);
    uint8_t *ring = smem;   // the ring starts the layout in both CTAs
    const uint32_t rank = cluster_ctarank();
    const bool is_s = rank < 2;
    const int sub = static_cast<int>(rank & 1);          // which head of the cluster's pair
    const uint16_t role_mask = is_s ? 0x3 : 0xC;           // the CTAs sharing this ring
    const uint32_t sibling = rank ^ 1u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int idx = blockIdx.x >> 2;
    const int hpi = idx % (p.Hkv * p.n_hpairs);
    idx /= p.Hkv * p.n_hpairs;
    const int mb = p.n_mblocks - 1 - (idx % p.n_mblocks);   // longest rows first
    const int b = idx / p.n_mblocks;
    const int g = hpi / p.n_hpairs;
    const int hg = 2 * (hpi % p.n_hpairs) + sub;           // head within the group
    const bool dup = hg >= p.G;                              // odd group: a repeat, not stored
    const int h = g * p.G + (dup ? p.G - 1 : hg);
    const int q_lo = p.S - p.T + mb * kBM;
    const int q_hi = min(q_lo + kBM - 1, p.S - 1);
    const int kt_first = p.window > 0 ? max(0, q_lo - p.window + 1) / kBN : 0;
    const int n_tiles = q_hi / kBN - kt_first + 1;
    // S-CTA: Q (4 slot loads), then K(0) chunks 0..3, K(1) ...; O-CTA: V(0) as (dims 0-255,
    // keys 0-63), (0-255, 64-127), (256-511, 0-63), (256-511, 64-127), V(1) ...
    const int kNS = is_s ? kNS_S : kNS_O;
    const int n_q = is_s ? 4 : 0;
    const int n_loads = n_q + kChunks * n_tiles;
    // bytes landing on the O-CTA's p_full phase i: packet i, then the row sums as "packet" n
    auto rx_bytes = [&](int i) {
        return i < n_tiles ? kPBytes + kFBytes : (i == n_tiles ? kFBytes : 0);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNS_S; ++i) {
            mbar_init(&bars->full[i], 1);
            mbar_init(&bars->empty[i], 2);   // this CTA's MMA and its sibling's
        }
        mbar_init(&bars->q_rot, kThreads);
        mbar_init(&bars->q_ready, 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_free[i], 128);
            mbar_init(&bars->p_staged[i], 128);
            mbar_init(&bars->rack[i], 1);
        }
        for (int i = 0; i < kNR; ++i) {
            mbar_init(&bars->pfree[i], 1);
            mbar_init(&bars->p_full[i], 1);
            mbar_init(&bars->o_ok[i], 128);
            mbar_init(&bars->pv_done[i], 1);
        }
        mbar_init(&bars->l_staged, 128);
        mbar_init(&bars->o_final, 1);
        mbar_init(&bars->staged, 128);
        mbar_init(&bars->mma_done, 1);
        if (!is_s) {
            // the first three receptions, before the S-CTA may send anything
            for (int i = 0; i < kNR; ++i)
                if (rx_bytes(i)) mbar_arrive_expect_tx(&bars->p_full[i], rx_bytes(i));
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers exist before any remote copy or arrival
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t peer = rank ^ 2u;   // the other role of this head's pair

    // ---- ring producer state (warp 0, lane 0) ----
    int pu = 0;
    bool pok = true;
    auto put = [&]() {
        const int st = pu % kNS;
        if (pu >= kNS && !(pok = mbar_wait(&bars->empty[st], ((pu / kNS) - 1) & 1))) {
            set_timeout(p.status, kDiagPrefillPair, 0, 1, pu);
            return;
        }
        const CUtensorMap *map;
        int c0, c1, c2;
        if (pu < n_q) {
            map = &tmQ;
            c0 = 128 * pu;
            c1 = mb * kBM;
            c2 = b * p.Hq + h;
        } else if (is_s) {
            // K chunk v of the shared stream: armed here, loaded by one of the two S-CTAs
            const int v = pu - n_q;
            uint8_t *dst = ring + st * kSlot;
            mbar_arrive_expect_tx(&bars->full[st], kSlot);
            if ((v & 1) == sub) {
                const int k0 = 128 * (v % kChunks), r0 = (kt_first + v / kChunks) * kBN;
                tma_load_3d_mc(dst, &tmK, &bars->full[st], k0, r0, b * p.Hkv + g, role_mask);
                tma_load_3d_mc(dst + kBox, &tmK, &bars->full[st], k0 + 64, r0, b * p.Hkv + g,
                               role_mask);
            }
            ++pu;
            return;
        } else {
            // V chunk pu, four 64 x 64 boxes: dims 256 dh + 64 i, keys 64 kh .. 64 kh + 63;
            // armed here, loaded by one of the two O-CTAs
            const int w = pu % kChunks;
            uint8_t *dst = ring + st * kSlot;
            const int d0 = 256 * (w >> 1), r0 = (kt_first + pu / kChunks) * kBN + 64 * (w & 1);
            mbar_arrive_expect_tx(&bars->full[st], kSlot);
            if ((pu & 1) == sub)
                for (int i = 0; i < 4; ++i)
                    tma_load_3d_mc(dst + i * kVBox, &tmV, &bars->full[st], d0 + 64 * i, r0,
                                   b * p.Hkv + g, role_mask);
            ++pu;
            return;
        }
        uint8_t *dst = ring + st * kSlot;
        mbar_arrive_expect_tx(&bars->full[st], kSlot);
        tma_load_3d(dst, map, &bars->full[st], c0, c1, c2);
        tma_load_3d(dst + kBox, map, &bars->full[st], c0 + 64, c1, c2);
        ++pu;
    };
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(is_s ? &tmQ : &tmV);
        if (is_s) tma_prefetch_desc(&tmK);
        while (pu < min(kNS, n_loads)) put();
    }

    if (is_s) {
        // ================= S-CTA: RoPE on the Q tile, by every warp =================
        // Q box i (dims 64 i .. 64 i + 63) sits at ring + i * kBox.  Warp w rotates rows
        // 16 w .. 16 w + 15, one at a time: lane l takes pairs 64 bb + 2l, + 1 of every
        // 64-pair box bb against their partners 256 dims later (box bb + 4); the table row
        // is read as 4 coalesced 512-byte pieces, 2 rows in flight.
        {
            constexpr int NB = kD / 128, QR = kBM / (kThreads / 32);
            constexpr int RIF = QR < 32 / NB ? QR : 32 / NB;   // rows in flight
            bool qok = true;
            for (int i = 0; i < 4; ++i) qok = qok && warp_wait(&bars->full[i], 0);
            if (!qok) set_timeout(p.status, kDiagPrefillPair, 3, 8, 0);
            if (qok) {
                const float4 *t4 = reinterpret_cast<const float4 *>(p.table);
                for (int r0 = 0; r0 < QR; r0 += RIF) {
                    float4 tv[RIF][NB];
#pragma unroll
                    for (int i = 0; i < RIF; ++i) {
                        const int row = QR * warp + r0 + i;
                        // rows past T hold zeros (the load's out-of-range fill): any row
                        const int pos = min(p.S - p.T + mb * kBM + row, p.S - 1);
#pragma unroll
                        for (int bb = 0; bb < NB; ++bb)
                            tv[i][bb] = __ldg(t4 + (size_t)pos * (kD / 4) + 32 * bb + lane);
                    }
#pragma unroll
                    for (int i = 0; i < RIF; ++i) {
                        const int row = QR * warp + r0 + i;
                        const int off =
                            row * 128 + ((((lane >> 2) ^ (row & 7)) << 4) | ((lane & 3) << 2));
#pragma unroll
                        for (int bb = 0; bb < NB; ++bb) {
                            uint32_t *pa = reinterpret_cast<uint32_t *>(ring + bb * kBox + off);
                            uint32_t *pb =
                                reinterpret_cast<uint32_t *>(ring + (bb + NB) * kBox + off);
                            const float4 t = tv[i][bb];
                            const uint32_t aw = *pa, bw = *pb;
                            const float a0 = bf16lo(aw), a1 = bf16hi(aw);
                            const float b0 = bf16lo(bw), b1 = bf16hi(bw);
                            *pa = pack_bf16x2(fmaf(a0, t.x, -b0 * t.y), fmaf(a1, t.z, -b1 * t.w));
                            *pb = pack_bf16x2(fmaf(a0, t.y, b0 * t.x), fmaf(a1, t.w, b1 * t.z));
                        }
                    }
                }
            }
            fence_proxy_async_smem();   // the slots are refilled by TMA afterwards
            mbar_arrive(&bars->q_rot);
        }

        if (warp == 0) {
            // ================= S-CTA: TMA producer, the rest of the ring =================
            if (lane == 0) {
                while (pok && pu < n_loads) put();
                if (!pok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
                for (int w = max(0, pu - kNS_S); w < pu; ++w)
                    mbar_wait(&bars->full[w % kNS_S], (w / kNS_S) & 1);
            }
            __syncwarp();
        } else if (warp == 1) {
            // ================= S-CTA: MMA issuer, S(j) = Q K(j)^T =================
            if (lane == 0) {
                const uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
                const uint32_t rbase = smem_u32(ring);
                bool ok = mbar_wait(&bars->q_ready, 0);
                if (!ok) set_timeout(p.status, kDiagPrefillPair, 1, 4, 0);
                tc_fence_after();
                // the Q slots are free for K once Q has been copied into TMEM (here and,
                // for the sibling's loads into them, there)
                const uint32_t empty_sib = mapa_shared(smem_u32(&bars->empty[0]), sibling);
                for (int i = 0; i < 4; ++i) {
                    mbar_arrive(&bars->empty[i]);
                    mbar_arrive_remote(empty_sib + 8 * i);
                }
                int u = n_q;
                for (int j = 0; j < n_tiles && ok; ++j) {
                    if (j >= 2) {
                        // the softmax has read S(j - 2) out of this buffer
                        if (!(ok = mbar_wait(&bars->s_free[j & 1], ((j >> 1) + 1) & 1))) {
                            set_timeout(p.status, kDiagPrefillPair, 1, 7, j);
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint32_t dst = tmem + ((j & 1) ? TS1 : TS0);
                    for (int c = 0; c < kChunks && ok; ++c) {
                        const int st = u % kNS_S;
                        if (!(ok = mbar_wait(&bars->full[st], (u / kNS_S) & 1))) {
                            set_timeout(p.status, kDiagPrefillPair, 1, 0, u);
                            break;
                        }
                        tc_fence_after();
                        const uint32_t ka = rbase + st * kSlot;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const int dk = 8 * c + kk;   // 16-dim step over the whole head
                            const uint64_t bd =
                                sdesc_sw128(ka + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
                            umma_ts(dst, tmem + TQ + 8 * dk, bd, idesc_s,
                                    (c > 0 || kk > 0) ? 1u : 0u);
                        }
                        umma_commit_mc(&bars->empty[st], role_mask);
                        ++u;
                    }
                    if (ok) umma_commit(&bars->s_full[j & 1]);
                }
                if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
                umma_commit(&bars->mma_done);
                mbar_wait(&bars->mma_done, 0);
            }
            __syncwarp();
        } else if (warp >= 4) {
            // ================= S-CTA: Q into TMEM, softmax, packets =================
            const int r = (warp & 3) * 32 + lane;   // row in tile == TMEM lane
            const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const int t = mb * kBM + r;
            const bool valid = t < p.T;
            const int qpos = p.S - p.T + t;
            bool ok = warp_wait(&bars->q_rot, 0);
            if (!ok) set_timeout(p.status, kDiagPrefillPair, 3, 9, 0);
            if (ok) {
                // row r of box bb: 8 swizzled 16-byte chunks = TMEM columns 32 bb .. + 31
                // (column c holds dims 2c, 2c + 1: the A-operand layout)
#pragma unroll 1
                for (int bb = 0; bb < 2 * kChunks; ++bb) {
                    uint32_t rr[32];
                    const uint8_t *row = ring + bb * kBox + r * 128;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint4 v =
                            *reinterpret_cast<const uint4 *>(row + ((cc ^ (r & 7)) << 4));
                        rr[4 * cc] = v.x;
                        rr[4 * cc + 1] = v.y;
                        rr[4 * cc + 2] = v.z;
                        rr[4 * cc + 3] = v.w;
                    }
                    tmem_st32(tmem + lane_off + TQ + 32 * bb, rr);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&bars->q_ready);

            const uint32_t p_full_remote = mapa_shared(smem_u32(&bars->p_full[0]), peer);
            const uint32_t p_remote = mapa_shared(smem_u32(smem + O_OFF_P), peer);
            const uint32_t f_remote = mapa_shared(smem_u32(smem + O_OFF_F), peer);
            float *fst = reinterpret_cast<float *>(smem + S_OFF_F);
            float m = -CUDART_INF_F, l = 0.f;
            for (int j = 0; j < n_tiles && ok; ++j) {
                if (!warp_wait(&bars->s_full[j & 1], (j >> 1) & 1)) {
                    set_timeout(p.status, kDiagPrefillPair, 3, 6, j);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tS = tmem + lane_off + ((j & 1) ? TS1 : TS0);
                const int n0 = (kt_first + j) * kBN;
                const bool full = valid && (n0 + kBN - 1 <= qpos) &&
                                  (p.window <= 0 || n0 >= qpos - p.window + 1);
                int c_lo = 0, c_hi = kBN;
                if (!full) {
                    c_hi = valid ? min(kBN, qpos - n0 + 1) : 0;
                    c_lo = p.window > 0 ? max(0, qpos - p.window + 1 - n0) : 0;
                }
                float x[kBN];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tS + 32 * c, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(rr[i]);
                }
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bars->s_free[j & 1]);   // the MMA may overwrite it with S(j + 2)
                if (!full) {
#pragma unroll
                    for (int i = 0; i < kBN; ++i)
                        x[i] = (i >= c_lo && i < c_hi) ? x[i] : -CUDART_INF_F;
                }
                float mx8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    mx8[k] = x[k];
#pragma unroll
                    for (int tt = 1; tt < kBN / 8; ++tt) mx8[k] = fmaxf(mx8[k], x[k + 8 * tt]);
                }
                // scale > 0, so the maximum commutes with it
                const float mraw = fmax3(fmax3(mx8[0], mx8[1], mx8[2]),
                                         fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
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
                // staging buffer j & 1 is free once packet j - 2 has landed in the O-CTA
                if (j >= 2 && !warp_wait_cluster(&bars->rack[j & 1], ((j >> 1) + 1) & 1)) {
                    set_timeout(p.status, kDiagPrefillPair, 3, 11, j);
                    ok = false;
                    break;
                }
                uint8_t *pbuf = smem + S_OFF_P + (j & 1) * kPBytes;
                float2 ls[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 a = ffma2(make_float2(x[32 * c + 2 * i], x[32 * c + 2 * i + 1]),
                                               p.scale_log2, nmref);
                        const float e0 = ex2_approx(a.x), e1 = ex2_approx(a.y);
                        ls[i & 3] = fadd2(ls[i & 3], make_float2(e0, e1));
                        pk[i] = pack_bf16x2(e0, e1);
                    }
                    // keys 32c .. 32c + 31: chunks 4c .. 4c + 3 of the row, in the
                    // 128-byte-swizzled K-major layout of two 64-key boxes
                    uint8_t *box = pbuf + (c >> 1) * kBox + r * 128;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int cc = 4 * (c & 1) + q4;
                        *reinterpret_cast<uint4 *>(box + ((cc ^ (r & 7)) << 4)) =
                            make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    }
                }
                l += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) +
                     ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
                fst[(j & 1) * kBM + r] = need_o ? f : 1.0f;
                fence_proxy_async_smem();   // the bulk copy reads the packet
                mbar_arrive(&bars->p_staged[j & 1]);
                if (r == 0) {
                    // receive buffer j % 3 is free once PV(j - 3) has finished
                    const int rb = j % kNR;
                    if (!mbar_wait(&bars->p_staged[j & 1], (j >> 1) & 1)) {
                        set_timeout(p.status, kDiagPrefillPair, 3, 12, j);
                        ok = false;
                    } else if (j >= kNR &&
                               !mbar_wait_cluster(&bars->pfree[rb], ((j / kNR) + 1) & 1)) {
                        set_timeout(p.status, kDiagPrefillPair, 3, 13, j);
                        ok = false;
                    } else {
                        const uint32_t bar = p_full_remote + rb * 8;
                        bulk_copy_s2c(p_remote + rb * kPBytes, pbuf, kPBytes, bar);
                        bulk_copy_s2c(f_remote + rb * kFBytes, fst + (j & 1) * kBM, kFBytes,
                                      bar);
                    }
                }
                ok = __all_sync(0xffffffffu, ok);   // the elected lane's wait decides for its warp
            }
            if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            // the row sums (into the f slot of receive buffer n % 3, as reception n), then
            // the log-sum-exp
            float *lst = reinterpret_cast<float *>(smem + S_OFF_L);
            lst[r] = l;
            fence_proxy_async_smem();
            mbar_arrive(&bars->l_staged);
            if (valid && p.lse && !dup)
                p.lse[((size_t)b * p.Hq + h) * p.T + t] = (m + __log2f(l)) * 0.69314718055994531f;
            if (r == 0 && ok) {
                const int rb = n_tiles % kNR;
                if (!mbar_wait(&bars->l_staged, 0) ||
                    (n_tiles >= kNR &&
                     !mbar_wait_cluster(&bars->pfree[rb], ((n_tiles / kNR) + 1) & 1))) {
                    set_timeout(p.status, kDiagPrefillPair, 3, 14, n_tiles);
                    ok = false;
                } else {
                    bulk_copy_s2c(f_remote + rb * kFBytes, lst, kFBytes, p_full_remote + rb * 8);
                }
                // the O-CTA's last acknowledgements land before this CTA may finish
                for (int jj = max(0, n_tiles - kNR); jj < n_tiles && ok; ++jj)
                    if (!mbar_wait_cluster(&bars->pfree[jj % kNR], (jj / kNR) & 1)) {
                        set_timeout(p.status, kDiagPrefillPair, 3, 15, jj);
                        ok = false;
                    }
                for (int jj = max(0, n_tiles - 2); jj < n_tiles && ok; ++jj)
                    if (!mbar_wait_cluster(&bars->rack[jj & 1], (jj >> 1) & 1)) {
                        set_timeout(p.status, kDiagPrefillPair, 3, 15, jj);
                        ok = false;
                    }
                if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            }
        }
    } else {
        if (warp == 0) {
            // ================= O-CTA: TMA producer (V) =================
            if (lane == 0) {
                while (pok && pu < n_loads) put();
                if (!pok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
                for (int w = max(0, pu - kNS_O); w < pu; ++w)
                    mbar_wait(&bars->full[w % kNS_O], (w / kNS_O) & 1);
            }
            __syncwarp();
        } else if (warp == 1) {
            // ================= O-CTA: MMA issuer, O += P(j) V(j) =================
            if (lane == 0) {
                const uint32_t idesc_o = idesc_bf16_f32(kBM, 256, 0, 1);
                const uint32_t rbase = smem_u32(ring);
                const uint32_t pbase = smem_u32(smem + O_OFF_P);
                bool ok = true;
                int u = 0;
                for (int j = 0; j < n_tiles && ok; ++j) {
                    const int rb = j % kNR;
                    if (!(ok = mbar_wait_cluster(&bars->p_full[rb], (j / kNR) & 1))) {
                        set_timeout(p.status, kDiagPrefillPair, 1, 2, j);
                        break;
                    }
                    // arm this buffer for reception j + 3
                    if (rx_bytes(j + kNR)) mbar_arrive_expect_tx(&bars->p_full[rb], rx_bytes(j + kNR));
                    if (!(ok = mbar_wait(&bars->o_ok[rb], (j / kNR) & 1))) {
                        set_timeout(p.status, kDiagPrefillPair, 1, 3, j);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t pa = pbase + rb * kPBytes;
                    // chunk w = 2 dh + kh: output columns 256 dh .., keys 64 kh ..
                    for (int w = 0; w < kChunks && ok; ++w) {
                        const int st = u % kNS_O, dh = w >> 1, kh = w & 1;
                        if (!(ok = mbar_wait(&bars->full[st], (u / kNS_O) & 1))) {
                            set_timeout(p.status, kDiagPrefillPair, 1, 0, u);
                            break;
                        }
                        tc_fence_after();
                        const uint32_t va = rbase + st * kSlot;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = sdesc_sw128(pa + kh * kBox + kk * 32, 16, 1024);
                            umma_ss(tmem + TO + 256 * dh, ad,
                                    sdesc_sw128(va + kk * 2048, kVBox, 1024), idesc_o,
                                    (j > 0 || kh > 0 || kk > 0) ? 1u : 0u);
                        }
                        umma_commit_mc(&bars->empty[st], role_mask);
                        ++u;
                    }
                    if (!ok) break;
                    umma_commit(&bars->pv_done[rb]);
                    if (j == n_tiles - 1) umma_commit(&bars->o_final);
                }
                if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
                umma_commit(&bars->mma_done);
                mbar_wait(&bars->mma_done, 0);
            }
            __syncwarp();
        } else if (warp == 2) {
            // ================= O-CTA: forwards "PV(j) done" to the S-CTA =================
            if (lane == 0) {
                const uint32_t pfree_remote = mapa_shared(smem_u32(&bars->pfree[0]), peer);
                for (int j = 0; j < n_tiles; ++j) {
                    if (!mbar_wait(&bars->pv_done[j % kNR], (j / kNR) & 1)) {
                        set_timeout(p.status, kDiagPrefillPair, 2, 14, j);
                        set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
                        break;
                    }
                    mbar_arrive_remote(pfree_remote + (j % kNR) * 8);
                }
            }
            __syncwarp();
        } else if (warp == 3) {
            // ======== O-CTA: tells the S-CTA that packet j has landed (staging j & 1 free) ========
            if (lane == 0) {
                const uint32_t rack_remote = mapa_shared(smem_u32(&bars->rack[0]), peer);
                for (int j = 0; j < n_tiles; ++j) {
                    if (!mbar_wait_cluster(&bars->p_full[j % kNR], (j / kNR) & 1)) {
                        set_timeout(p.status, kDiagPrefillPair, 2, 15, j);
                        set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
                        break;
                    }
                    mbar_arrive_remote(rack_remote + (j & 1) * 8);
                }
            }
            __syncwarp();
        } else if (warp >= 4) {
            // ================= O-CTA: lazy rescale of O rows, epilogue =================
            const int r = (warp & 3) * 32 + lane;
            const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const float *frcv = reinterpret_cast<const float *>(smem + O_OFF_F);
            bool ok = true;
            for (int j = 0; j < n_tiles && ok; ++j) {
                if (!warp_wait_cluster(&bars->p_full[j % kNR], (j / kNR) & 1)) {
                    set_timeout(p.status, kDiagPrefillPair, 3, 2, j);
                    ok = false;
                    break;
                }
                const float f = frcv[(j % kNR) * kBM + r];
                if (__any_sync(0xffffffffu, f != 1.0f)) {
                    // O holds the products of tiles < j: wait for the last one (j > 0: the
                    // factor of the first tile is always 1)
                    if (!warp_wait(&bars->pv_done[(j - 1) % kNR], ((j - 1) / kNR) & 1)) {
                        set_timeout(p.status, kDiagPrefillPair, 3, 7, j);
                        ok = false;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < kD / 32 && ok; ++c) {
                        uint32_t rr[32];
                        tmem_ld32(tmem + lane_off + TO + 32 * c, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            rr[i] = __float_as_uint(__uint_as_float(rr[i]) * f);
                        tmem_st32(tmem + lane_off + TO + 32 * c, rr);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(&bars->o_ok[j % kNR]);
            }
            if (!ok) set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            if (ok && warp_wait(&bars->o_final, 0) &&
                warp_wait_cluster(&bars->p_full[n_tiles % kNR], (n_tiles / kNR) & 1)) {
                // O / l as bf16 into the ring (every PV product has completed, so no V tile
                // is still read), as eight 128-byte-swizzled 64-column boxes; TMA stores
                // write them out (rows past T are clipped by the tensor map)
                tc_fence_after();
                const float l = frcv[(n_tiles % kNR) * kBM + r];   // the row sums
                const float inv_l = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll 1
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t rr[32];
                    tmem_ld32(tmem + lane_off + TO + 32 * c, rr);
                    tmem_wait_ld();
                    uint8_t *box = ring + (c >> 1) * kBox + r * 128;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int cc = 4 * (c & 1) + q4;
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
                if (r == 0 && !dup) {
                    if (!mbar_wait(&bars->staged, 0)) {
                        set_timeout(p.status, kDiagPrefillPair, 3, 10, n_tiles);
                    } else {
                        for (int bx = 0; bx < kD / 64; ++bx)
                            tma_store_3d(&tmO, ring + bx * kBox, 64 * bx, mb * kBM, b * p.Hq + h);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                }
            } else if (ok) {
                set_timeout(p.status, kDiagPrefillPair, 3, 9, n_tiles);
                set_status(p.status, GQA_ERR_DEVICE_TIMEOUT);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no copy or remote arrival may target a CTA that has finished
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_pair() {
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
bool make_map_pair(CUtensorMap *map, const void *base, int rows, int slabs, int box_rows) {
    EncodeTiledFn fn = encode_fn_pair();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)rows, (cuuint64_t)slabs};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * 2 * rows};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_prefill_pair(const void *q, const void *k_rot, const void *v, void *o, float *lse,
                        int B, int T, int S, int Hq, int Hkv, int window, float scale,
                        const float *table, int *status, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_map_pair(&mq, q, T, B * Hq, 128) || !make_map_pair(&mk, k_rot, S, B * Hkv, 128) ||
        !make_map_pair(&mv, v, S, B * Hkv, 64) || !make_map_pair(&mo, o, T, B * Hq, 128))
        return GQA_ERR_CUDA;
    if (ensure_smem_attr(reinterpret_cast<const void *>(prefill_pair_kernel), kSmemBytes) !=
        cudaSuccess)
        return GQA_ERR_CUDA;
    PairParams p;
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
    p.n_hpairs = (p.G + 1) / 2;
    p.scale_log2 = scale * 1.4426950408889634f;
    const long clusters = (long)B * Hkv * p.n_hpairs * p.n_mblocks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(4 * clusters));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, prefill_pair_kernel, mq, mk, mv, mo, p) != cudaSuccess)
        return GQA_ERR_CUDA;
    return GQA_OK;
}

}  // namespace gqa
