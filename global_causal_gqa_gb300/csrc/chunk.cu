// chunk.cu -- chunked prefill over an existing KV cache: the keys a chunk attends to,
// and the multi-token append that follows it.
//
// "PLaMo 3アーキテクチャ徹底解析" §4.4: the cache holds K before RoPE; a chunk of T new
// tokens attends to the tokens already cached followed by itself, with key positions
// 0..S-1 (S = cached + T) and query positions S-T..S-1 generated inside attention; a
// local layer's cache keeps only the newest tokens and re-numbers them from 0 (its
// window W is the ring's capacity, so every key a chunk query can see is in the ring or
// in the chunk).  The pages check that processing a sequence in chunks gives the same
// outputs as one pass.
//
// gather: for one sequence, rows 0..R-1 of the cache in logical order (R = count for a
// linear cache, min(count, cap) for a ring, oldest first) followed by the T chunk rows,
// K rotated at its row index and V copied, into contiguous [Hkv, S, d] buffers that
// gqa_attn_prefill consumes (k_is_rotated = 1).  append: the chunk's T tokens into the
// cache, T slots from count on (a ring keeps the last cap of them), then count += T.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

__device__ __forceinline__ void rotate_pairs(uint4 &av, uint4 &bv, const float4 *tr) {
    float cs[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 t = __ldg(tr + q);
        cs[4 * q + 0] = t.x;
        cs[4 * q + 1] = t.y;
        cs[4 * q + 2] = t.z;
        cs[4 * q + 3] = t.w;
    }
    const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
    uint32_t ao[4], bo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float a0 = bf16lo(aw[q]), a1 = bf16hi(aw[q]);
        const float b0 = bf16lo(bw[q]), b1 = bf16hi(bw[q]);
        const float c0 = cs[4 * q + 0], s0 = cs[4 * q + 1];
        const float c1 = cs[4 * q + 2], s1 = cs[4 * q + 3];
        ao[q] = pack_bf16x2(fmaf(a0, c0, -b0 * s0), fmaf(a1, c1, -b1 * s1));
        bo[q] = pack_bf16x2(fmaf(a0, s0, b0 * c0), fmaf(a1, s1, b1 * c1));
    }
    av = make_uint4(ao[0], ao[1], ao[2], ao[3]);
    bv = make_uint4(bo[0], bo[1], bo[2], bo[3]);
}

// One thread per (head, row, chunk pair c / c + d/16).
__global__ void prefill_gather_kernel(const gqa_kv_desc *__restrict__ desc_p,
                                      const uint4 *__restrict__ k_new,
                                      const uint4 *__restrict__ v_new, int T, int Hkv, int d,
                                      uint4 *k_out, uint4 *v_out, int S,
                                      const float4 *__restrict__ table, int table_len,
                                      int *status) {
    const gqa_kv_desc desc = *desc_p;
    const int cap = desc.cap;
    const int R = desc.is_ring ? min(desc.count, cap) : desc.count;
    if (R < 0 || R + T != S || S > table_len) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            set_status(status, S > table_len ? GQA_ERR_RANGE : GQA_ERR_CAPACITY);
        return;
    }
    const int first = desc.is_ring ? (desc.count - R) % max(cap, 1) : 0;
    const int cpr = d / 16;    // chunk pairs per row
    const int rc = d / 8;      // 16-byte chunks per row
    const long total = (long)Hkv * S * cpr;
    const uint4 *kc = static_cast<const uint4 *>(desc.k);
    const uint4 *vc = static_cast<const uint4 *>(desc.v);
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
         i += (long)gridDim.x * blockDim.x) {
        const int c = static_cast<int>(i % cpr);
        const long hr = i / cpr;
        const int r = static_cast<int>(hr % S), h = static_cast<int>(hr / S);
        const uint4 *ks, *vs;
        if (r < R) {
            int slot = first + r;
            if (slot >= cap) slot -= cap;
            if (!GQA_IN_BOUNDS(slot, cap, status, (kDiagCache << 24) | 3)) continue;
            ks = kc + ((long)h * cap + slot) * rc;
            vs = vc + ((long)h * cap + slot) * rc;
        } else {
            ks = k_new + ((long)h * T + (r - R)) * rc;
            vs = v_new + ((long)h * T + (r - R)) * rc;
        }
        if (!GQA_IN_BOUNDS(r, table_len, status, (kDiagCache << 24) | 4)) continue;
        uint4 a = ks[c], b = ks[c + cpr];
        rotate_pairs(a, b, table + ((long)r * (d / 2) + 8 * c) / 2);
        uint4 *ko = k_out + ((long)h * S + r) * rc;
        uint4 *vo = v_out + ((long)h * S + r) * rc;
        ko[c] = a;
        ko[c + cpr] = b;
        vo[c] = vs[c];
        vo[c + cpr] = vs[c + cpr];
    }
}

// One block per sequence: T tokens [Hkv, T, d] per sequence into slots count + t (linear,
// all or nothing) or (count + t) mod cap (ring; only the last cap tokens are written, the
// earlier ones would be overwritten within the same chunk), then count += T.
__global__ void kv_append_chunk_kernel(gqa_kv_desc *descs, const uint4 *__restrict__ k_new,
                                       const uint4 *__restrict__ v_new, int T, int Hkv, int d,
                                       int *status) {
    __shared__ int s_ok;
    const int seq = blockIdx.x;
    gqa_kv_desc *desc = descs + seq;
    const int cap = desc->cap, count = desc->count, ring = desc->is_ring;
    if (threadIdx.x == 0) {
        s_ok = cap > 0 && count >= 0 && (ring || (long)count + T <= cap);
        if (!s_ok) set_status(status, GQA_ERR_CAPACITY);
    }
    __syncthreads();
    if (s_ok) {
        const int rc = d / 8;
        const int t0 = ring && T > cap ? T - cap : 0;
        const long n = (long)Hkv * (T - t0) * rc;
        uint4 *kc = static_cast<uint4 *>(desc->k);
        uint4 *vc = static_cast<uint4 *>(desc->v);
        for (long i = threadIdx.x; i < n; i += blockDim.x) {
            const int c = static_cast<int>(i % rc);
            const long ht = i / rc;
            const int t = t0 + static_cast<int>(ht % (T - t0)), h = static_cast<int>(ht / (T - t0));
            const long slot = ring ? ((long)count + t) % cap : (long)count + t;
            if (!GQA_IN_BOUNDS(slot, cap, status, (kDiagCache << 24) | 5)) continue;
            const long src = (((long)seq * Hkv + h) * T + t) * rc + c;
            const long dst = ((long)h * cap + slot) * rc + c;
            kc[dst] = k_new[src];
            vc[dst] = v_new[src];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_ok) desc->count = count + T;
}

}  // namespace

cudaError_t launch_prefill_gather(const gqa_kv_desc *desc, const void *k_new, const void *v_new,
                                  int T, int Hkv, int d, void *k_out, void *v_out, int S,
                                  const float *table, int table_len, int *status,
                                  cudaStream_t s) {
    const long total = (long)Hkv * S * (d / 16);
    long blocks = (total + 255) / 256;
    if (blocks > 152L * 16) blocks = 152L * 16;
    if (blocks < 1) blocks = 1;
    prefill_gather_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        desc, static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), T, Hkv, d,
        static_cast<uint4 *>(k_out), static_cast<uint4 *>(v_out), S,
        reinterpret_cast<const float4 *>(table), table_len, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_append_chunk(gqa_kv_desc *descs, int nseq, const void *k_new,
                                   const void *v_new, int T, int Hkv, int d, int *status,
                                   cudaStream_t s) {
    kv_append_chunk_kernel<<<nseq, 256, 0, s>>>(descs, static_cast<const uint4 *>(k_new),
                                                static_cast<const uint4 *>(v_new), T, Hkv, d,
                                                status);
    return cudaGetLastError();
}

}  // namespace gqa
