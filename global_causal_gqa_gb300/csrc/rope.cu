// rope.cu -- RoPE cos/sin table and the standalone rotation kernel.
//
// Split-half pairs (j, j + d/2) rotated by p * omega_j ("PLaMo 3アーキテクチャ徹底解析"
// §6.1), with the amplitude factor on both cos and sin (§6.3).  The table stores
// (amp cos(p omega_j), amp sin(p omega_j)) as float pairs [p][j]; both are evaluated in
// double precision and rounded once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {

__global__ void rope_table_kernel(float2 *table, const InvFreq w, int half, double amp,
                                  long total) {
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
         i += (long)gridDim.x * blockDim.x) {
        const long p = i / half;
        const int j = static_cast<int>(i - p * half);
        double s, c;
        sincos(static_cast<double>(p) * w.w[j], &s, &c);
        table[i] = make_float2(static_cast<float>(amp * c), static_cast<float>(amp * s));
    }
}

cudaError_t launch_rope_table(float *table, const InvFreq &w, int d, double amp, int max_pos,
                              cudaStream_t s) {
    const int half = d / 2;
    const long total = static_cast<long>(max_pos) * half;
    const int threads = 256;
    long blocks = (total + threads - 1) / threads;
    if (blocks > 152L * 64) blocks = 152L * 64;
    rope_table_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        reinterpret_cast<float2 *>(table), w, half, amp, total);
    return cudaGetLastError();
}

// One thread rotates 8 pairs: chunk c (elements 8c..8c+7, the first half) with chunk
// c + d/16 (their partners j + d/2).  16-byte loads and stores; the table row is read
// as four 16-byte loads.
__global__ void rope_apply_kernel(const uint4 *__restrict__ x, uint4 *y, long rows, int T,
                                  int d, int pos0, const float4 *__restrict__ table,
                                  int table_len, int *status) {
    const int cpr = d / 16;  // chunk pairs per row
    const long total = rows * cpr;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
         i += (long)gridDim.x * blockDim.x) {
        const long row = i / cpr;
        const int c = static_cast<int>(i - row * cpr);
        const long pos = pos0 + (row % T);
        if (pos < 0 || pos >= table_len) {
            set_status(status, GQA_ERR_RANGE);
            continue;
        }
        const uint4 *xr = x + row * (d / 8);
        const uint4 av = xr[c];
        const uint4 bv = xr[c + cpr];
        // table row pos, pairs 8c..8c+7: 16 floats = 4 float4
        const float4 *tr = table + (pos * (d / 2) + 8 * c) / 2;
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
        uint4 *yr = y + row * (d / 8);
        yr[c] = make_uint4(ao[0], ao[1], ao[2], ao[3]);
        yr[c + cpr] = make_uint4(bo[0], bo[1], bo[2], bo[3]);
    }
}

cudaError_t launch_rope_apply(const void *x, void *y, long rows, int T, int d, int pos0,
                              const float *table, int table_len, int *status,
                              cudaStream_t s) {
    const long total = rows * (d / 16);
    const int threads = 256;
    long blocks = (total + threads - 1) / threads;
    if (blocks > 152L * 16) blocks = 152L * 16;
    if (blocks < 1) blocks = 1;
    rope_apply_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        static_cast<const uint4 *>(x), static_cast<uint4 *>(y), rows, T, d, pos0,
        reinterpret_cast<const float4 *>(table), table_len, status);
    return cudaGetLastError();
}

}  // namespace gqa
