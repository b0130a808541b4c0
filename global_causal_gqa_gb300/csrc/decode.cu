// decode.cu -- split-KV decode over a linear or ring KV cache, then an LSE combine.
//
// "PLaMo 3アーキテクチャ徹底解析": §4.4 (K cached before RoPE and rotated at every step,
// keys at positions 0..R-1, query at R-1; the local ring keeps the newest W tokens),
// §4.5 (attention equation), §2.3 (decode reads every cached K and V once per step:
// 4 Hkv d bytes per token and layer -- the bound this kernel is written against).
//
// Work split: one CTA per (split of `chunk` keys, sequence, block of KV heads; the split
// rule is decode_split below); each KV head is streamed by d/128 warps (d = 128, 256, 512), each of which owns
// 64 pairs of the split-half RoPE in two groups of 32 -- [64 p, 64 p + 64) at d <= 256;
// [32 p, +32) and [d/4 + 32 p, +32) at d = 512, so that the pairs p-RoPE rotates are
// spread over two warps -- with the head-dim elements j and d/2 + j of each pair j, so
// every warp sees a 128-element vector whose RoPE pairs are (l, l + 64), the d = 128
// layout.  Keys go in blocks of 16 with 16-byte read-only loads, double-buffered in
// registers so the next block's loads are in flight during the math; the warps of a
// head add their partial scores through shared memory (one named barrier per block)
// and each accumulates the output for its own elements.
// The query group of G <= 8 heads shares every K and V element, so the per-block math
// is two warp-level bf16 MMAs (m16n8k16): S^T = K' Q'^T and O^T += V^T P^T, fp32
// accumulate.  The head dimension is permuted (identically on both operands of each
// product) so that every 16-byte load lands directly in MMA fragment order and each
// RoPE pair (j, j + 64) sits in one thread.  K is rotated in registers from the fp32
// table at its logical position.  Each warp writes an unnormalised partial (m, l, O) for
// its G heads; the combine kernel merges the splits by their log-sum-exp.
//
// Shared K/V projection (Gemma 4 global layers, attention_k_eq_v, §5.2 and §8 of the same
// page): the cache holds one row Zn = N_1(Z) per token; the values are Zn and the keys
// RoPE(gamma_k * Zn), the fp32 gain multiplied into each loaded K element of a rotating
// pair in fp32 and rotated in fp32, with one rounding to bf16 for the MMA (pairs that
// never rotate carry the gain on the query instead).  Each row is loaded once, in the
// K layout; the V fragments are the 8x8 transposes (movmatrix) of those registers taken
// before the gain and the rotation, so every byte of the cache crosses L1 once: half the
// traffic of separate K and V.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 8;
// two 8 KB table stages per warp, then the partial-score exchange (8 KB)
constexpr int kDecodeSmem = kWarps * 2 * 512 * 16 + kWarps * 2 * 32 * 4 * 4;

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte asynchronous copy global -> shared, cached in L1 (the 8 warps of a CTA read
// the same table rows).
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t word(const uint4 &u, int i) {
    return i == 0 ? u.x : i == 1 ? u.y : i == 2 ? u.z : u.w;
}

// Rotates the two pairs in 32-bit word q of chunks a and b by t = (cos0, sin0, cos1, sin1)
// (amplitude included).
__device__ __forceinline__ void rotate_word(uint4 &a, uint4 &b, int q, const float4 &t) {
    uint32_t &aw = q == 0 ? a.x : q == 1 ? a.y : q == 2 ? a.z : a.w;
    uint32_t &bw = q == 0 ? b.x : q == 1 ? b.y : q == 2 ? b.z : b.w;
    const float a0 = bf16lo(aw), a1 = bf16hi(aw), b0 = bf16lo(bw), b1 = bf16hi(bw);
    aw = pack_bf16x2(fmaf(a0, t.x, -b0 * t.y), fmaf(a1, t.z, -b1 * t.w));
    bw = pack_bf16x2(fmaf(a0, t.y, b0 * t.x), fmaf(a1, t.w, b1 * t.z));
}

// Shared K/V keys: multiplies the two pairs in word q of chunks a and b by the key gain in
// fp32 (ga: a's two elements, gb: b's), rotates them by t and rounds once to bf16.
__device__ __forceinline__ void gain_rotate_word(uint4 &a, uint4 &b, int q, const float4 &t,
                                                 const float2 &ga, const float2 &gb) {
    uint32_t &aw = q == 0 ? a.x : q == 1 ? a.y : q == 2 ? a.z : a.w;
    uint32_t &bw = q == 0 ? b.x : q == 1 ? b.y : q == 2 ? b.z : b.w;
    // packed over the word's two pairs: (a0, a1) and (b0, b1)
    const float2 av = fmul2(make_float2(bf16lo(aw), bf16hi(aw)), ga);
    const float2 bv = fmul2(make_float2(bf16lo(bw), bf16hi(bw)), gb);
    const float2 c = make_float2(t.x, t.z), s = make_float2(t.y, t.w);
    const float2 ra = fsub2(fmul2(av, c), fmul2(bv, s));
    const float2 rb = ffma2v(av, s, fmul2(bv, c));
    aw = pack_bf16x2(ra.x, ra.y);
    bw = pack_bf16x2(rb.x, rb.y);
}

// Gain pair qq (elements 2 qq, 2 qq + 1) of a chunk whose 8 gains are g[0], g[1].
__device__ __forceinline__ float2 gain_pair(const float4 (&g)[2], int qq) {
    const float4 &h = g[qq >> 1];
    return (qq & 1) ? make_float2(h.z, h.w) : make_float2(h.x, h.y);
}

// Rotates the 8 pairs (a[e], b[e]) held in two 16-byte chunks by the table entries
// starting at `tab` (8 consecutive float2 = (amp cos, amp sin)).
__device__ __forceinline__ void rotate8(uint4 &a, uint4 &b, const float2 *tab) {
    const float4 *t4 = reinterpret_cast<const float4 *>(tab);
    float cs[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 t = __ldg(t4 + q);
        cs[4 * q] = t.x;
        cs[4 * q + 1] = t.y;
        cs[4 * q + 2] = t.z;
        cs[4 * q + 3] = t.w;
    }
    uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float a0 = bf16lo(aw[q]), a1 = bf16hi(aw[q]);
        const float b0 = bf16lo(bw[q]), b1 = bf16hi(bw[q]);
        const float c0 = cs[4 * q], s0 = cs[4 * q + 1], c1 = cs[4 * q + 2], s1 = cs[4 * q + 3];
        aw[q] = pack_bf16x2(fmaf(a0, c0, -b0 * s0), fmaf(a1, c1, -b1 * s1));
        bw[q] = pack_bf16x2(fmaf(a0, s0, b0 * c0), fmaf(a1, s1, b1 * c1));
    }
    a = make_uint4(aw[0], aw[1], aw[2], aw[3]);
    b = make_uint4(bw[0], bw[1], bw[2], bw[3]);
}

struct SeqView {
    int R;        // logical keys attended
    int first;    // ring slot of logical key 0
    int cap;
    bool ok;
};

__device__ __forceinline__ SeqView seq_view(const gqa_kv_desc &desc, int max_len) {
    SeqView v;
    v.cap = desc.cap;
    v.R = desc.is_ring ? min(desc.count, desc.cap) : desc.count;
    v.first = desc.is_ring ? (desc.count - v.R) % max(desc.cap, 1) : 0;
    v.ok = v.R > 0 && v.R <= max_len && v.R <= desc.rope_len && v.R <= desc.cap;
    return v;
}

// Shared memory after the table stages and the exchange: the key gain, fp32 [d].
constexpr int kDecodeSmemShared = kDecodeSmem + kMaxHeadDim * 4;

template <int PARTS, bool SHARED>   // warps per KV head: d = 128 PARTS; shared K/V rows
__global__ void __launch_bounds__(kWarps * 32, 1)
    decode_partial_kernel(const __nv_bfloat16 *__restrict__ q,
                          const gqa_kv_desc *__restrict__ descs, int Hq, int Hkv,
                          float scale_log2, int max_len, int chunk, int nsplit,
                          float *__restrict__ ws_ml,
                          float *__restrict__ ws_o, int *status,
                          const float *__restrict__ k_gamma) {
    constexpr int d = kD * PARTS, parts = PARTS;
    griddep_wait();               // the appended token, counts and partials of earlier kernels
    griddep_launch_dependents();  // the combine kernel may start launching
    extern __shared__ float4 dsmem[];
    // the key gain as float pairs: entry i holds elements 2i, 2i + 1
    float2 *sgain = reinterpret_cast<float2 *>(reinterpret_cast<uint8_t *>(dsmem) + kDecodeSmem);
    if constexpr (SHARED) {
        // before any warp may leave: every thread takes part in the barrier
        for (int i = threadIdx.x; i < d / 2; i += blockDim.x)
            sgain[i] = reinterpret_cast<const float2 *>(k_gamma)[i];
        __syncthreads();
    }
    const int split = blockIdx.x, seq = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = warp % parts;               // this warp's 64 RoPE pairs (pb below)
    const int hg = warp / parts;                 // head group within the CTA
    const int g = blockIdx.z * (kWarps / parts) + hg;
    // This warp's RoPE pairs for the K/Q layout's chunk group c (c = 0, 1): 32 pairs from
    // pb(c).  d = 512 spreads them, [32 part, +32) and [d/4 + 32 part, +32), so that the 64
    // pairs p-RoPE rotates fall to two warps, half each; otherwise [64 part + 32 c, +32).
    constexpr bool kSpread = PARTS == 4;
    auto pb = [&](int c) { return kSpread ? 32 * part + c * (d / 4) : 64 * part + 32 * c; };
    // global 16-byte chunk of the row for local chunk lc (8 elements) of this warp: K and Q
    // (gchunk), and V of separate caches (vchunk, whose 8 first-half chunks are one
    // 128-byte line)
    auto vchunk = [&](int lc) {
        return lc < 8 ? 8 * part + lc : d / 16 + 8 * part + (lc - 8);
    };
    auto gchunk = [&](int lc) {
        if constexpr (kSpread) {
            const int l = lc & 7;
            return (lc >> 3) * (d / 16) + pb(l >> 2) / 8 + (l & 3);
        } else {
            return vchunk(lc);
        }
    };
    const gqa_kv_desc desc = descs[seq];
    const SeqView sv = seq_view(desc, max_len);
    if (!sv.ok) {
        if (split == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            set_status(status, sv.R > max_len || sv.R > desc.cap ? GQA_ERR_CAPACITY
                                                                   : GQA_ERR_RANGE);
        return;
    }
    // the host passes a multiple of 64 (decode_split); the mask states that to the
    // compiler, which then fits the kernel in 255 registers without spilling
    chunk &= ~63;
    const int k_start = split * chunk;
    if (k_start >= sv.R || g >= Hkv) return;
    const int k_end = min(sv.R, k_start + chunk);
    const int G = Hq / Hkv;
    const int qpos = sv.R - 1;
    const int gq = lane >> 2, tq = lane & 3;
    const float2 *table = reinterpret_cast<const float2 *>(desc.rope);
    // p-RoPE (§6.4), d = 512: a group of 32 pairs that never rotate -- table rows 0 and 1
    // both exactly (1, 0), as gqa_rope_table_build writes for omega = 0 at amplitude 1 --
    // neither copies table rows nor rotates its keys (the rotation would multiply them by
    // 1 and add 0: the same keys).  With 64 of 256 pairs rotating this drops 3/4 of the
    // table traffic, which at 2 KB per position otherwise overflows L2, and the rotation
    // left falls to two warps.  rot_c: group c rotates (warp-uniform); lanes 16c .. 16c + 15
    // read its rows 0 and 1 here, and the vote follows the query load so the loads
    // overlap.  Not at d = 256, where the branches cost the register-bound kernel 5% on
    // fully rotating rings.
    bool rot0 = true, rot1 = true;
    float4 r0 = make_float4(0.f, 0.f, 0.f, 0.f), r1 = r0;
    if constexpr (PARTS == 4) {
        if (sv.R > 1) {
            const float2 *t0 = table + pb(lane >> 4) + 2 * (lane & 15);
            r0 = __ldg(reinterpret_cast<const float4 *>(t0));
            r1 = __ldg(reinterpret_cast<const float4 *>(t0 + d / 2));
        }
    }

    // Q' as the B operand of S^T = K' Q'^T: thread (gq, tq) holds head gq, elements
    // 32c + 8tq + e (c = 0..3, e = 0..7) of this warp's 128 (global chunk gchunk(4c + tq));
    // k-chunk kc = 2c + (e >> 2).
    uint32_t qb[8][2];
    {
        uint4 qc[4];
        if (gq < G && GQA_IN_BOUNDS((size_t)seq * Hq + (size_t)g * G + gq,
                                    (size_t)gridDim.y * Hq, status, (kDiagDecode << 24) | 1) &&
            GQA_IN_BOUNDS(qpos, desc.rope_len, status, (kDiagDecode << 24) | 5)) {
            const uint4 *qr = reinterpret_cast<const uint4 *>(
                q + ((size_t)seq * Hq + (size_t)g * G + gq) * d);
#pragma unroll
            for (int c = 0; c < 4; ++c) qc[c] = qr[gchunk(4 * c + tq)];
#pragma unroll
            for (int c = 0; c < 2; ++c)
                rotate8(qc[c], qc[c + 2],
                        table + (size_t)qpos * (d / 2) +
                            (kSpread ? pb(c) : 64 * part + 32 * c) + 8 * tq);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) qc[c] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            qb[2 * c][0] = qc[c].x;
            qb[2 * c][1] = qc[c].y;
            qb[2 * c + 1][0] = qc[c].z;
            qb[2 * c + 1][1] = qc[c].w;
        }
    }

    if constexpr (PARTS == 4) {
        const bool id = r0.x == 1.f && r0.y == 0.f && r0.z == 1.f && r0.w == 0.f &&
                        r1.x == 1.f && r1.y == 0.f && r1.z == 1.f && r1.w == 0.f;
        const unsigned b = __ballot_sync(0xffffffffu, id);
        rot0 = (b & 0xFFFFu) != 0xFFFFu;
        rot1 = (b >> 16) != 0xFFFFu;
        if constexpr (SHARED) {
            // A group of pairs that never rotates takes the key gain on the query instead:
            // sum_e q_e (gamma_e z_e) = sum_e (gamma_e q_e) z_e, so its keys are the raw
            // rows and the per-key gain work is gone; gamma_e q_e is formed in fp32 and
            // rounded once, as gamma_e z_e is for the rotating pairs.
            const float4 *sg4 = reinterpret_cast<const float4 *>(sgain);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (c == 0 ? rot0 : rot1) continue;
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // chunks c and c + 2
                    const int lc = 4 * (c + 2 * h) + tq;
                    const float4 gv[2] = {sg4[2 * gchunk(lc)], sg4[2 * gchunk(lc) + 1]};
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        uint32_t &w = qb[2 * (c + 2 * h) + (qq >> 1)][qq & 1];
                        const float2 v = fmul2(make_float2(bf16lo(w), bf16hi(w)), gain_pair(gv, qq));
                        w = pack_bf16x2(v.x, v.y);
                    }
                }
            }
        }
    }

    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run0 = -CUDART_INF_F, m_run1 = -CUDART_INF_F, l_run0 = 0.f, l_run1 = 0.f;

    // This warp's two table stages: the 16 table rows of a key block, 16-byte entry
    // (k, lane) at k * 32 + (lane ^ 2 (k & 3)) holding what lane (gq, tq) needs for
    // k = 8 rs + 4 c + qq: pairs pb(c) + 8tq + 2qq and the next one at position
    // kb + gq + 8 rs.
    // The XOR keeps both the copies in and the reads out free of bank conflicts.
    float4 *stage_base = dsmem + (size_t)warp * 2 * 512;
    float *xchg = reinterpret_cast<float *>(dsmem + (size_t)kWarps * 2 * 512) +
                  (size_t)hg * (2 * parts * 32 * 4);

    const __nv_bfloat16 *kbase = static_cast<const __nv_bfloat16 *>(desc.k) + (size_t)g * sv.cap * d;
    const __nv_bfloat16 *vbase =
        SHARED ? kbase : static_cast<const __nv_bfloat16 *>(desc.v) + (size_t)g * sv.cap * d;
    auto slot_of = [&](int key) {
        int s = sv.first + key;
        s = s >= sv.cap ? s - sv.cap : s;
        if (!GQA_IN_BOUNDS(s, sv.cap, status, (kDiagDecode << 24) | 2)) s = 0;
        return s;
    };

    // One block = 16 keys: K rows kb + gq and kb + gq + 8, V rows kb + 2tq + {0, 1, 8, 9}
    // (16-byte chunks vchunk(gq) and vchunk(8 + gq) of each, so every load instruction
    // reads whole 128-byte lines), and the block's table rows copied to shared memory;
    // rows at or past k_end are clamped in range and get weight 0.  Two register buffers
    // and two table stages: the next block's loads are in flight while the current block
    // is computed.
    struct Block {
        uint4 k0[4], k1[4], vv[4][2];
        int kb;
    };
    auto load = [&](Block &bl, int kb) {
        bl.kb = kb;
        const int kk0 = min(kb + gq, k_end - 1), kk1 = min(kb + gq + 8, k_end - 1);
        const uint4 *kr0 = reinterpret_cast<const uint4 *>(kbase + (size_t)slot_of(kk0) * d);
        const uint4 *kr1 = reinterpret_cast<const uint4 *>(kbase + (size_t)slot_of(kk1) * d);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            bl.k0[c] = ld_stream(kr0 + gchunk(4 * c + tq));
            bl.k1[c] = ld_stream(kr1 + gchunk(4 * c + tq));
        }
        if constexpr (!SHARED) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int key = min(kb + 2 * tq + (i & 1) + ((i >> 1) << 3), k_end - 1);
                const uint4 *vr =
                    reinterpret_cast<const uint4 *>(vbase + (size_t)slot_of(key) * d);
                bl.vv[i][0] = ld_stream(vr + vchunk(gq));
                bl.vv[i][1] = ld_stream(vr + vchunk(8 + gq));
            }
        }
        // table rows kb .. kb + 15: instruction i copies row i (clamped); lane l copies the
        // 16-byte piece l & 15 of chunk group c = l >> 4 -- pairs pb(c) + 2 (l & 15) and the
        // next one, i.e. pb(c) + 8tq + 2qq -- skipped for a group that never rotates
        __syncwarp();   // every lane is done reading this stage's previous block
        float4 *stg = stage_base + (((kb - k_start) >> 4) & 1) * 512;
        const int kq = ((lane >> 4) << 2) | (lane & 3);   // 4c + qq
        const int lp_lo = (lane >> 2) & 3;                  // tq
        if constexpr (kSpread) {
            if (lane < 16 ? rot0 : rot1) {
                const float4 *src =
                    reinterpret_cast<const float4 *>(table + pb(lane >> 4)) + (lane & 15);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    int row = min(kb + i, k_end - 1);
                    if (!GQA_IN_BOUNDS(row, desc.rope_len, status, (kDiagDecode << 24) | 4)) row = 0;
                    const int k = ((i >> 3) << 3) | kq;
                    const int lp = ((i & 7) << 2) | lp_lo;
                    cp_async16(stg + k * 32 + (lp ^ ((k & 3) << 1)), src + (size_t)row * (d / 4));
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                int row = min(kb + i, k_end - 1);
                if (!GQA_IN_BOUNDS(row, desc.rope_len, status, (kDiagDecode << 24) | 4)) row = 0;
                const int k = ((i >> 3) << 3) | kq;
                const int lp = ((i & 7) << 2) | lp_lo;
                cp_async16(stg + k * 32 + (lp ^ ((k & 3) << 1)),
                           reinterpret_cast<const float4 *>(table + (size_t)row * (d / 2) +
                                                            64 * part) + lane);
            }
        }
        cp_async_commit();
    };
    auto compute = [&](Block &bl, bool next_pending) {
        const int kb = bl.kb;
        const int key0 = kb + gq, key1 = kb + gq + 8;
        const bool ok0 = key0 < k_end, ok1 = key1 < k_end;
        // this block's table stage has landed (the next block's copies may still run)
        if (next_pending) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncwarp();
        const float4 *stg = stage_base + (((kb - k_start) >> 4) & 1) * 512;
        // Shared rows: the V^T fragments are the transposes of the raw K-layout words.
        // Word q of chunk c of key row kb + gq (k0; kb + gq + 8 for k1) is element
        // 8 gchunk(4c + tq) + 2q + {0, 1}; seen as an 8x8 matrix (row = key gq, column =
        // 2tq + j), its transpose gives this thread keys 2tq, 2tq + 1 (+8 for k1) of dim
        // 8 gchunk(4c + (gq >> 1)) + 2q + (gq & 1).
        uint32_t vt0[4][4], vt1[4][4];
        if constexpr (SHARED) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    vt0[c][qq] = transpose8x8(word(bl.k0[c], qq));
                    vt1[c][qq] = transpose8x8(word(bl.k1[c], qq));
                }
        }
        // rotate K at logical positions kb + gq, kb + gq + 8 (clamped rows: k_end - 1).
        // Shared rows: keys = gamma_k * Zn, formed in fp32 inside the rotation; word qq of
        // chunk lc holds elements 8 gchunk(lc) + 2 qq, + 1, gain pair 4 gchunk(lc) + qq.
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            // the 8 gains of chunks c and c + 2 (shared rows only)
            float4 gA[2], gB[2];
            if constexpr (SHARED) {
                const float4 *sg4 = reinterpret_cast<const float4 *>(sgain);
                gA[0] = sg4[2 * gchunk(4 * c + tq)];
                gA[1] = sg4[2 * gchunk(4 * c + tq) + 1];
                gB[0] = sg4[2 * gchunk(4 * (c + 2) + tq)];
                gB[1] = sg4[2 * gchunk(4 * (c + 2) + tq) + 1];
            }
            if (c == 0 ? rot0 : rot1) {
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int sw = lane ^ (qq << 1);
                    if constexpr (SHARED) {
                        const float2 ga = gain_pair(gA, qq), gb = gain_pair(gB, qq);
                        gain_rotate_word(bl.k0[c], bl.k0[c + 2], qq, stg[(4 * c + qq) * 32 + sw],
                                         ga, gb);
                        gain_rotate_word(bl.k1[c], bl.k1[c + 2], qq,
                                         stg[(8 + 4 * c + qq) * 32 + sw], ga, gb);
                    } else {
                        rotate_word(bl.k0[c], bl.k0[c + 2], qq, stg[(4 * c + qq) * 32 + sw]);
                        rotate_word(bl.k1[c], bl.k1[c + 2], qq, stg[(8 + 4 * c + qq) * 32 + sw]);
                    }
                }
            }
            // (a group that never rotates has its gain on the query: raw keys)
        }
        // S^T (16 keys x 8 heads) in two independent accumulation chains
        float s[4] = {0.f, 0.f, 0.f, 0.f}, t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            mma16816(s, bl.k0[c].x, bl.k1[c].x, bl.k0[c].y, bl.k1[c].y, qb[2 * c][0], qb[2 * c][1]);
            mma16816(t, bl.k0[c].z, bl.k1[c].z, bl.k0[c].w, bl.k1[c].w, qb[2 * c + 1][0],
                     qb[2 * c + 1][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] += t[i];
        if constexpr (PARTS > 1) {
            // add the other warps' partial scores for the same (key, head) fragment
            float *xb = xchg + (size_t)(((kb - k_start) >> 4) & 1) * (parts * 128);
            reinterpret_cast<float4 *>(xb + part * 128)[lane] = make_float4(s[0], s[1], s[2], s[3]);
            named_bar_sync(1 + hg, 32 * parts);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int pp = 0; pp < parts; ++pp) {
                const float4 v = reinterpret_cast<const float4 *>(xb + pp * 128)[lane];
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            s[0] = acc.x;
            s[1] = acc.y;
            s[2] = acc.z;
            s[3] = acc.w;
        }
        // online softmax per head column (heads 2tq, 2tq+1), log2 domain
        const float x0 = ok0 ? s[0] * scale_log2 : -CUDART_INF_F;
        const float x1 = ok0 ? s[1] * scale_log2 : -CUDART_INF_F;
        const float x2 = ok1 ? s[2] * scale_log2 : -CUDART_INF_F;
        const float x3 = ok1 ? s[3] * scale_log2 : -CUDART_INF_F;
        float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
        }
        const float mn0 = fmaxf(m_run0, bm0), mn1 = fmaxf(m_run1, bm1);
        const float f0 = ex2_approx(m_run0 - mn0), f1 = ex2_approx(m_run1 - mn1);
        const float p0 = ex2_approx(x0 - mn0), p1 = ex2_approx(x1 - mn1);
        const float p2 = ex2_approx(x2 - mn0), p3 = ex2_approx(x3 - mn1);
        l_run0 = l_run0 * f0 + p0 + p2;
        l_run1 = l_run1 * f1 + p1 + p3;
        m_run0 = mn0;
        m_run1 = mn1;
        const uint32_t pb0 = transpose8x8(pack_bf16x2(p0, p1));
        const uint32_t pb1 = transpose8x8(pack_bf16x2(p2, p3));
        // O^T (128 dims x 8 heads) += V^T P^T; dims permuted.  Separate V: row g of m-tile
        // mt is dim 64 (mt >> 2) + 8g + 2 (mt & 3), row g + 8 the dim after it.  Shared
        // rows: m-tile mt = 2c + (q >> 1) takes words q (rows 0..7) and q + 1 (rows 8..15)
        // of chunk c, q even.
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            o[mt][0] *= f0;
            o[mt][1] *= f1;
            o[mt][2] *= f0;
            o[mt][3] *= f1;
            if constexpr (SHARED) {
                const int c = mt >> 1, qq = 2 * (mt & 1);
                mma16816(o[mt], vt0[c][qq], vt0[c][qq + 1], vt1[c][qq], vt1[c][qq + 1], pb0,
                         pb1);
            } else {
                const uint32_t w0 = word(bl.vv[0][mt >> 2], mt & 3);
                const uint32_t w1 = word(bl.vv[1][mt >> 2], mt & 3);
                const uint32_t w2 = word(bl.vv[2][mt >> 2], mt & 3);
                const uint32_t w3 = word(bl.vv[3][mt >> 2], mt & 3);
                mma16816(o[mt], __byte_perm(w0, w1, 0x5410), __byte_perm(w0, w1, 0x7632),
                         __byte_perm(w2, w3, 0x5410), __byte_perm(w2, w3, 0x7632), pb0, pb1);
            }
        }
    };

    Block ba, bb;
    load(ba, k_start);
    for (int kb = k_start; kb < k_end; kb += 32) {
        const bool more1 = kb + 16 < k_end;
        if (more1) load(bb, kb + 16);
        compute(ba, more1);
        if (!more1) break;
        const bool more2 = kb + 32 < k_end;
        if (more2) load(ba, kb + 32);
        compute(bb, more2);
    }

    // partial sums of l over the 8 key rows held across gq
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, off);
        l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, off);
    }
    const int h0 = 2 * tq, h1 = 2 * tq + 1;  // heads within the group
    const size_t rec0 = ((size_t)seq * Hq + (size_t)g * G + h0) * nsplit + split;
    const size_t rec1 = ((size_t)seq * Hq + (size_t)g * G + h1) * nsplit + split;
    const size_t n_rec = (size_t)gridDim.y * Hq * nsplit;   // partial records in the workspace
    const bool rec0_ok = h0 >= G || GQA_IN_BOUNDS(rec0, n_rec, status, (kDiagDecode << 24) | 6);
    const bool rec1_ok = h1 >= G || GQA_IN_BOUNDS(rec1, n_rec, status, (kDiagDecode << 24) | 6);
    // this warp's output elements: local 64 (i >> 1) + 8 gq + 4 (i & 1) + 0..3, i.e.
    // global 64 part + 8 gq + ... in the first half and d/2 + 64 part + ... in the second
    auto out_off = [&](int i) {
        return (i >> 1) * (d / 2) + 64 * part + 8 * gq + 4 * (i & 1);
    };
    if constexpr (SHARED) {
        // This thread holds, for chunk c, dims b + 2q + par (q = 0..3, par = gq & 1,
        // b = 8 gchunk(4c + (gq >> 1))): o[2c][0, 2] for q = 0, 1 and o[2c + 1][0, 2] for
        // q = 2, 3 (head h0; columns 1, 3 for h1).  The lane with the other parity
        // (lane ^ 4) holds the rest; after one exchange the even lane writes b .. b + 3 and
        // the odd lane b + 4 .. b + 7.
        const int par = gq & 1;
        float4 out0[4], out1[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float *lo = o[2 * c], *hi = o[2 * c + 1];
            const float s0 = par ? lo[0] : hi[0], s1 = par ? lo[2] : hi[2];
            const float s2 = par ? lo[1] : hi[1], s3 = par ? lo[3] : hi[3];
            const float r0 = __shfl_xor_sync(0xffffffffu, s0, 4);
            const float r1 = __shfl_xor_sync(0xffffffffu, s1, 4);
            const float r2 = __shfl_xor_sync(0xffffffffu, s2, 4);
            const float r3 = __shfl_xor_sync(0xffffffffu, s3, 4);
            out0[c] = par ? make_float4(r0, hi[0], r1, hi[2]) : make_float4(lo[0], r0, lo[2], r1);
            out1[c] = par ? make_float4(r2, hi[1], r3, hi[3]) : make_float4(lo[1], r2, lo[3], r3);
        }
        auto sh_off = [&](int c) { return 8 * gchunk(4 * c + (gq >> 1)) + 4 * par; };
        if (h0 < G && rec0_ok) {
            if (gq == 0 && part == 0) {
                ws_ml[2 * rec0] = m_run0;
                ws_ml[2 * rec0 + 1] = l_run0;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<float4 *>(ws_o + rec0 * d + sh_off(c)) = out0[c];
        }
        if (h1 < G && rec1_ok) {
            if (gq == 0 && part == 0) {
                ws_ml[2 * rec1] = m_run1;
                ws_ml[2 * rec1 + 1] = l_run1;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<float4 *>(ws_o + rec1 * d + sh_off(c)) = out1[c];
        }
        return;
    }
    if (h0 < G && rec0_ok) {
        if (gq == 0 && part == 0) {
            ws_ml[2 * rec0] = m_run0;
            ws_ml[2 * rec0 + 1] = l_run0;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4 *>(ws_o + rec0 * d + out_off(i)) =
                make_float4(o[2 * i][0], o[2 * i][2], o[2 * i + 1][0], o[2 * i + 1][2]);
    }
    if (h1 < G && rec1_ok) {
        if (gq == 0 && part == 0) {
            ws_ml[2 * rec1] = m_run1;
            ws_ml[2 * rec1 + 1] = l_run1;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4 *>(ws_o + rec1 * d + out_off(i)) =
                make_float4(o[2 * i][1], o[2 * i][3], o[2 * i + 1][1], o[2 * i + 1][3]);
    }
}

// One block per (query head, sequence), one thread per head-dim element.
__global__ void __launch_bounds__(kMaxHeadDim)
    decode_combine_kernel(const gqa_kv_desc *__restrict__ descs, int Hq, int d, int max_len,
                          int chunk, int nsplit, const float *__restrict__ ws_ml,
                          const float *__restrict__ ws_o, __nv_bfloat16 *__restrict__ out,
                          float *__restrict__ lse, int *status) {
    const int h = blockIdx.x, seq = blockIdx.y, dd = threadIdx.x;
    griddep_wait();               // this step's partials
    griddep_launch_dependents();
    const SeqView sv = seq_view(descs[seq], max_len);
    if (!sv.ok) return;
    int ns = (sv.R + chunk - 1) / chunk;
    const size_t rec = ((size_t)seq * Hq + h) * nsplit;
    if (!GQA_IN_BOUNDS(ns - 1, nsplit, status, (kDiagDecode << 24) | 7)) ns = 0;
    float M = -CUDART_INF_F;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, ws_ml[2 * (rec + s)]);
    float L = 0.f, acc = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float f = ex2_approx(ws_ml[2 * (rec + s)] - M);
        L += ws_ml[2 * (rec + s) + 1] * f;
        acc += ws_o[(rec + s) * d + dd] * f;
    }
    out[((size_t)seq * Hq + h) * d + dd] = __float2bfloat16_rn(acc / L);
    if (lse && dd == 0) lse[(size_t)seq * Hq + h] = (M + __log2f(L)) * 0.69314718055994531f;
}

}  // namespace

// Keys per split: the largest of 2048, 1024, ..., 64 that still gives the grid at least
// 128 CTAs for a batch whose every sequence held max_len keys.  Long splits amortise each
// CTA's fixed work (query load and rotation, the first table stages, the partial it
// writes); 128 CTAs keep most of the 152 SMs streaming.  Measured on GB300 over split
// sizes 64 .. 2048: 2048 is fastest for the 8k-64k-token batches (PLaMo-3 and Gemma-4
// global, plain and shared K/V); 512 for 32 rings of 1024 at d = 256 (2 CTAs per
// sequence: 128 CTAs, 0.069 ms vs 0.072 at 256 and 0.118 at 1024) and for the 64-layer
// step's rings of 2048 (4.68 ms vs 4.98 at 256 and 7.37 at 1024).
DecodeSplit decode_split(int nseq, int Hkv, int d, int max_len) {
    const int heads_per_cta = kWarps / (d / kD);
    const long rows = static_cast<long>(nseq) * ((Hkv + heads_per_cta - 1) / heads_per_cta);
    DecodeSplit sp;
    sp.chunk = 2048;
    while (sp.chunk > 64 && rows * ((max_len + sp.chunk - 1) / sp.chunk) < 128) sp.chunk >>= 1;
    sp.nsplit = (max_len + sp.chunk - 1) / sp.chunk;
    return sp;
}

size_t decode_workspace_bytes(int nseq, int Hq, int Hkv, int d, int max_len) {
    const int ns = decode_split(nseq, Hkv, d, max_len).nsplit;
    return (decode_ml_floats(nseq, Hq, ns) + static_cast<size_t>(nseq) * Hq * ns * d) *
           sizeof(float);
}

cudaError_t launch_decode(const void *q, const gqa_kv_desc *descs, int nseq, int Hq, int Hkv,
                          int d, float scale, int max_len, void *o, float *lse, float *ws,
                          int *status, cudaStream_t s, const float *k_gamma) {
    const DecodeSplit sp = decode_split(nseq, Hkv, d, max_len);
    const int nsplit = sp.nsplit;
    float *ws_ml = ws;
    float *ws_o = ws + decode_ml_floats(nseq, Hq, nsplit);   // 16-byte aligned
    const int parts = d / kD;                       // warps per KV head
    const int heads_per_cta = kWarps / parts;
    const int heads = Hkv < heads_per_cta ? Hkv : heads_per_cta;
    dim3 grid(nsplit, nseq, (Hkv + heads_per_cta - 1) / heads_per_cta);
    const float scale_log2 = scale * 1.4426950408889634f;
    const bool shared = k_gamma != nullptr;
    auto kern = shared ? (parts == 1   ? decode_partial_kernel<1, true>
                          : parts == 2 ? decode_partial_kernel<2, true>
                                       : decode_partial_kernel<4, true>)
                       : (parts == 1   ? decode_partial_kernel<1, false>
                          : parts == 2 ? decode_partial_kernel<2, false>
                                       : decode_partial_kernel<4, false>);
    const int smem = shared ? kDecodeSmemShared : kDecodeSmem;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, grid, dim3(heads * parts * 32), smem, s,
                               static_cast<const __nv_bfloat16 *>(q), descs, Hq, Hkv,
                               scale_log2, max_len, sp.chunk, nsplit, ws_ml, ws_o, status,
                               k_gamma);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_combine_kernel, dim3(Hq, nseq), dim3(d), 0, s, descs, Hq, d,
                      max_len, sp.chunk, nsplit, static_cast<const float *>(ws_ml),
                      static_cast<const float *>(ws_o), static_cast<__nv_bfloat16 *>(o), lse,
                      status);
}

}  // namespace gqa
