// qknorm.cu -- the step in front of attention: per-head RMSNorm of Q and K, RoPE on the
// normalised K, and the cache append, fused so each projected row is read once.
//
// "PLaMo 3アーキテクチャ徹底解析": §3.2 RMSNorm with an effective gain gamma = c + w
// (N(x) = gamma * x / sqrt(mean(x^2) + eps)); §4.3 q_norm / k_norm normalise every
// (token, head) vector of d values with offset c = 1, eps = 1e-6 and one gain shared by
// all heads, V is not normalised; §4.4 the order is norm -> cache update (K normalised
// but not rotated, V as projected) -> RoPE -> attention; Gemma 4 also applies a gain-free
// RMSNorm to V (§8 of the same page).  The sums of squares and the scaling run in fp32;
// each output is rounded once to bf16.
//
// Shared K/V projection (Gemma 4 global layers, attention_k_eq_v, §5.2 and §8): one
// projection output Z gives K = RoPE(N_{gamma_k}(Z)) and V = N_1(Z).  The cache stores
// only Zn = bf16(N_1(Z)); since N_gamma(Z) = gamma * N_1(Z), the keys are recomputed from
// it as RoPE(gamma_k * Zn): the fp32 gain times the stored bf16 row, rotated in fp32 and
// rounded once to bf16, as the decode kernel forms them (the rotation's products may round
// in a different order there: at most one bf16 step apart).
//
// One warp per row.  Lane l holds the 32-bit words (bf16 pairs) l, l + 32, ... of the
// row's first half and the words d/4 later of the second half, so each RoPE pair
// (j, j + d/2) sits in one lane; loads and stores are 4-byte and coalesced per warp.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kMaxWordsPerLane = kMaxHeadDim / 2 / 32;   // d = 512: 8 words per lane

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Loads a row's words owned by this lane, returns 1 / sqrt(mean(x^2) + eps).  nw = words
// per lane in each half (0 for lanes past the end when d / 4 < 32).
struct Row {
    uint32_t a[kMaxWordsPerLane / 2], b[kMaxWordsPerLane / 2];   // first / second half
};

__device__ __forceinline__ float load_row(const uint32_t *src, int d, int lane, Row &row) {
    const int hw = d / 4;   // words per half
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < kMaxWordsPerLane / 2; ++m) {
        const int w = lane + 32 * m;
        if (w < hw) {
            row.a[m] = src[w];
            row.b[m] = src[w + hw];
            const float a0 = bf16lo(row.a[m]), a1 = bf16hi(row.a[m]);
            const float b0 = bf16lo(row.b[m]), b1 = bf16hi(row.b[m]);
            ss += a0 * a0 + a1 * a1 + b0 * b0 + b1 * b1;
        }
    }
    return ss;
}

// gamma[j] for the two elements of word w (elements 2w, 2w + 1)
__device__ __forceinline__ float2 gain2(const float *gamma, int w) {
    return gamma ? reinterpret_cast<const float2 *>(gamma)[w] : make_float2(1.f, 1.f);
}

// Normalises one row (scale inv), writes it to `norm_out` (nullable) and, rotated by the
// table row `tab` (nullable), to `rot_out`.
__device__ __forceinline__ void finish_row(const Row &row, int d, int lane, float inv,
                                           const float *gamma, uint32_t *norm_out,
                                           uint32_t *rot_out, const float2 *tab) {
    const int hw = d / 4;
#pragma unroll
    for (int m = 0; m < kMaxWordsPerLane / 2; ++m) {
        const int w = lane + 32 * m;
        if (w < hw) {
            const float2 ga = gain2(gamma, w), gb = gain2(gamma, w + hw);
            const float a0 = bf16lo(row.a[m]) * inv * ga.x, a1 = bf16hi(row.a[m]) * inv * ga.y;
            const float b0 = bf16lo(row.b[m]) * inv * gb.x, b1 = bf16hi(row.b[m]) * inv * gb.y;
            if (norm_out) {
                norm_out[w] = pack_bf16x2(a0, a1);
                norm_out[w + hw] = pack_bf16x2(b0, b1);
            }
            if (rot_out) {
                // pairs (2w, 2w + d/2) and (2w + 1, 2w + 1 + d/2): table entries 2w, 2w + 1
                const float4 t = reinterpret_cast<const float4 *>(tab)[w];
                rot_out[w] = pack_bf16x2(a0 * t.x - b0 * t.y, a1 * t.z - b1 * t.w);
                rot_out[w + hw] = pack_bf16x2(a0 * t.y + b0 * t.x, a1 * t.w + b1 * t.z);
            }
        }
    }
}

// Shared K/V row: Zn = bf16(x * inv) to `v_out` (nullable); the key row
// RoPE(gamma * Zn), formed in fp32 from the rounded Zn and rounded once, by the table row
// `tab` to `k_rot` (nullable).
__device__ __forceinline__ void finish_row_shared(const Row &row, int d, int lane, float inv,
                                                  const float *gamma, uint32_t *v_out,
                                                  uint32_t *k_rot, const float2 *tab) {
    const int hw = d / 4;
#pragma unroll
    for (int m = 0; m < kMaxWordsPerLane / 2; ++m) {
        const int w = lane + 32 * m;
        if (w < hw) {
            const uint32_t za = pack_bf16x2(bf16lo(row.a[m]) * inv, bf16hi(row.a[m]) * inv);
            const uint32_t zb = pack_bf16x2(bf16lo(row.b[m]) * inv, bf16hi(row.b[m]) * inv);
            if (v_out) {
                v_out[w] = za;
                v_out[w + hw] = zb;
            }
            if (k_rot) {
                const float2 ga = gain2(gamma, w), gb = gain2(gamma, w + hw);
                const float a0 = bf16lo(za) * ga.x, a1 = bf16hi(za) * ga.y;
                const float b0 = bf16lo(zb) * gb.x, b1 = bf16hi(zb) * gb.y;
                const float4 t = reinterpret_cast<const float4 *>(tab)[w];
                k_rot[w] = pack_bf16x2(a0 * t.x - b0 * t.y, a1 * t.z - b1 * t.w);
                k_rot[w + hw] = pack_bf16x2(a0 * t.y + b0 * t.x, a1 * t.w + b1 * t.z);
            }
        }
    }
}

// Prefill: Q rows [rows_q, d] -> q_out = N_q(q); K rows [rows_k, d] (row = (b, g, t)) ->
// k_out = N_k(k), k_rot = RoPE(N_k(k)) at position pos0 + t; with kv_shared the K rows are
// shared projection outputs Z: k_out = Zn (the values and the cache row), k_rot as above.
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(
    const uint32_t *__restrict__ q, const uint32_t *__restrict__ k, uint32_t *q_out,
    uint32_t *k_out, uint32_t *k_rot, long rows_q, long rows_k, int T, int d, int pos0,
    const float *__restrict__ q_gamma, const float *__restrict__ k_gamma, float eps,
    const float2 *__restrict__ table, int kv_shared) {
    const int lane = threadIdx.x & 31;
    const long warps = (long)gridDim.x * (blockDim.x >> 5);
    const int wpr = d / 2;   // words per row
    for (long r = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows_q + rows_k;
         r += warps) {
        Row row;
        if (r < rows_q) {
            const float ss = warp_sum(load_row(q + r * wpr, d, lane, row));
            finish_row(row, d, lane, rsqrtf(ss / d + eps), q_gamma, q_out + r * wpr, nullptr,
                       nullptr);
        } else {
            const long rk = r - rows_q;
            const int t = static_cast<int>(rk % T);
            const float ss = warp_sum(load_row(k + rk * wpr, d, lane, row));
            const float2 *tab = table ? table + (size_t)(pos0 + t) * (d / 2) : nullptr;
            if (kv_shared)
                finish_row_shared(row, d, lane, rsqrtf(ss / d + eps), k_gamma,
                                  k_out ? k_out + rk * wpr : nullptr,
                                  k_rot ? k_rot + rk * wpr : nullptr, tab);
            else
                finish_row(row, d, lane, rsqrtf(ss / d + eps), k_gamma,
                           k_out ? k_out + rk * wpr : nullptr,
                           k_rot ? k_rot + rk * wpr : nullptr, tab);
        }
    }
}

// Decode: one block per sequence.  The new token's slot is taken as kv_append takes it;
// Q rows are normalised into q_out, K rows normalised into the cache slot, V rows copied
// (or, with v_norm, normalised without a gain) into the cache slot, then count += 1.
// Shared K/V (v_new == nullptr, k_gamma == nullptr): the K rows are projection outputs Z and
// the K cache slot receives Zn = N_1(Z); no V cache is written.
__global__ void __launch_bounds__(256) qk_norm_append_kernel(
    gqa_kv_desc *descs, const uint32_t *__restrict__ q, const uint32_t *__restrict__ k_new,
    const uint32_t *__restrict__ v_new, int Hq, int Hkv, int d, const float *__restrict__ q_gamma,
    const float *__restrict__ k_gamma, float eps, int v_norm, uint32_t *q_out,
    int32_t *slots, int *status) {
    __shared__ int s_slot;
    const int seq = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    gqa_kv_desc *desc = descs + seq;
    if (threadIdx.x == 0) {
        const int cap = desc->cap, count = desc->count;
        int slot = -1;
        if (cap > 0 && count >= 0) {
            if (desc->is_ring) slot = count % cap;
            else if (count < cap) slot = count;
        }
        if (slot < 0) set_status(status, GQA_ERR_CAPACITY);
        s_slot = slot;
    }
    __syncthreads();
    const int slot = s_slot;
    const int wpr = d / 2;
    const long cap = desc->cap;
    uint32_t *kc = static_cast<uint32_t *>(desc->k), *vc = static_cast<uint32_t *>(desc->v);
    const int nw = blockDim.x >> 5;
    const int n_rows = Hq + (v_new ? 2 : 1) * Hkv;
    for (int r = warp; r < n_rows; r += nw) {
        Row row;
        if (r < Hq) {
            const long src = ((long)seq * Hq + r) * wpr;
            const float ss = warp_sum(load_row(q + src, d, lane, row));
            finish_row(row, d, lane, rsqrtf(ss / d + eps), q_gamma, q_out + src, nullptr,
                       nullptr);
        } else if (slot >= 0 && GQA_IN_BOUNDS(slot, cap, status, (kDiagCache << 24) | 2)) {
            const bool is_k = r < Hq + Hkv;
            const int g = is_k ? r - Hq : r - Hq - Hkv;
            const long src = ((long)seq * Hkv + g) * wpr;
            const long dst = ((long)g * cap + slot) * wpr;
            const float ss = warp_sum(load_row((is_k ? k_new : v_new) + src, d, lane, row));
            if (is_k || v_norm) {
                finish_row(row, d, lane, rsqrtf(ss / d + eps), is_k ? k_gamma : nullptr,
                           (is_k ? kc : vc) + dst, nullptr, nullptr);
            } else {
                finish_row(row, d, lane, 1.0f, nullptr, vc + dst, nullptr, nullptr);
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (slot >= 0) desc->count = desc->count + 1;
        if (slots) slots[seq] = slot;
    }
}

}  // namespace

cudaError_t launch_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out,
                                void *k_rot, int B, int Hq, int Hkv, int T, int d, int pos0,
                                const float *q_gamma, const float *k_gamma, float eps,
                                const float *table, int kv_shared, cudaStream_t s) {
    const long rows_q = q ? (long)B * Hq * T : 0, rows_k = (long)B * Hkv * T;
    long blocks = (rows_q + rows_k + 7) / 8;
    if (blocks > 152L * 16) blocks = 152L * 16;
    qk_norm_rope_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const uint32_t *>(q), static_cast<const uint32_t *>(k),
        static_cast<uint32_t *>(q_out), static_cast<uint32_t *>(k_out),
        static_cast<uint32_t *>(k_rot), rows_q, rows_k, T, d, pos0, q_gamma, k_gamma, eps,
        reinterpret_cast<const float2 *>(table), kv_shared);
    return cudaGetLastError();
}

cudaError_t launch_qk_norm_append(gqa_kv_desc *descs, int nseq, const void *q, const void *k_new,
                                  const void *v_new, int Hq, int Hkv, int d,
                                  const float *q_gamma, const float *k_gamma, float eps,
                                  int v_norm, void *q_out, int32_t *slots, int *status,
                                  cudaStream_t s) {
    qk_norm_append_kernel<<<nseq, 256, 0, s>>>(
        descs, static_cast<const uint32_t *>(q), static_cast<const uint32_t *>(k_new),
        static_cast<const uint32_t *>(v_new), Hq, Hkv, d, q_gamma, k_gamma, eps, v_norm,
        static_cast<uint32_t *>(q_out), slots, status);
    return cudaGetLastError();
}

}  // namespace gqa
