// internal.h -- launchers shared between the kernel translation units and the C ABI.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "gqa_attn.h"

namespace gqa {

constexpr int kMaxHeadDim = 512;

struct InvFreq {
    double w[kMaxHeadDim / 2];
};

// Launches `kern` with programmatic stream serialization: its blocks may be scheduled
// while the previous kernel on the stream drains, so the launch latency overlaps that
// kernel's tail.  The kernel must call griddep_wait() before it reads anything an earlier
// kernel on the stream wrote (the decode step's append -> partial -> combine chain).
// Not while the stream is being captured into a CUDA graph: a graph already launches
// back to back, and with programmatic edges the 64-layer decode step ran 1% slower
// (eagerly it runs 7% faster with them).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        (void)cudaGetLastError();   // treat as capturing: plain stream order
        cap = cudaStreamCaptureStatusActive;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cap == cudaStreamCaptureStatusNone ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// RoPE table and application (rope.cu)
cudaError_t launch_rope_table(float *table, const InvFreq &w, int d, double amp, int max_pos,
                              cudaStream_t s);
cudaError_t launch_rope_apply(const void *x, void *y, long rows, int T, int d, int pos0,
                              const float *table, int table_len, int *status, cudaStream_t s);

// KV cache append (kv.cu)
cudaError_t launch_kv_append(gqa_kv_desc *descs, int nseq, const void *k_new,
                             const void *v_new, int Hkv, int d, int32_t *slots,
                             int *status, cudaStream_t s);

// Decode (decode.cu)
// The split-KV grid: `chunk` keys per split (a multiple of 16), `nsplit` splits per
// sequence, chosen on the host from the batch shape (decode.cu documents the rule).  The
// workspace holds nseq Hq nsplit partials, so its size and the launch use the same rule.
struct DecodeSplit {
    int chunk;
    int nsplit;
};
DecodeSplit decode_split(int nseq, int Hkv, int d, int max_len);
// Decode workspace layout: nseq Hq nsplit (m, l) float pairs, padded to a multiple of 4
// floats so that the O partials after them start on a 16-byte boundary (the partial
// kernel writes them with 16-byte stores), then nseq Hq nsplit rows of d floats.
__host__ __device__ inline size_t decode_ml_floats(int nseq, int Hq, int nsplit) {
    const size_t n = (size_t)2 * nseq * Hq * nsplit;
    return (n + 3) & ~(size_t)3;
}
// Raises `func`'s dynamic shared-memory limit to `bytes` on the current device, once per
// (kernel, device): the attribute belongs to a device's context, so each GPU a process
// drives needs its own call.  Thread-safe.
cudaError_t ensure_smem_attr(const void *func, int bytes);
// k_gamma == nullptr: separate K and V caches; otherwise each desc.k holds Zn of a shared
// K/V projection (keys RoPE(gamma_k * Zn) formed in fp32, values Zn) and desc.v is not read
cudaError_t launch_decode(const void *q, const gqa_kv_desc *descs, int nseq, int Hq, int Hkv,
                          int d, float scale, int max_len, void *o, float *lse,
                          float *ws, int *status, cudaStream_t s,
                          const float *k_gamma = nullptr);
// Bytes of decode workspace for this batch shape (the same rule as launch_decode).
size_t decode_workspace_bytes(int nseq, int Hq, int Hkv, int d, int max_len);

// d = 128 prefill: picks the persistent kernel (prefill.cu) or the one-CTA-per-item
// kernel (prefill_stream.cu) by the mean item length; returns a gqa_status.  fuse_k: K is
// before RoPE and the persistent kernel rotates each K tile in shared memory.
int launch_prefill(const void *q, const void *k_rot, const void *v, void *o, float *lse,
                   int B, int T, int S, int Hq, int Hkv, int d, int window, float scale,
                   const float *table, int table_len, int *status, cudaStream_t s,
                   bool fuse_k = false);

// d = 128 prefill, one CTA per work item (prefill_stream.cu); returns a gqa_status
int launch_prefill_stream(const void *q, const void *k_rot, const void *v, void *o, float *lse,
                          int B, int T, int S, int Hq, int Hkv, int d, int window, float scale,
                          const float *table, int *status, cudaStream_t s);

// Prefill for d = 256 / 512 (prefill_wide.cu); returns a gqa_status
int launch_prefill_wide(const void *q, const void *k_rot, const void *v, void *o, float *lse,
                        int B, int T, int S, int Hq, int Hkv, int d, int window, float scale,
                        const float *table, int *status, cudaStream_t s);

// Prefill for d = 512 on a cluster of two CTAs (prefill_pair.cu); returns a gqa_status
int launch_prefill_pair(const void *q, const void *k_rot, const void *v, void *o, float *lse,
                        int B, int T, int S, int Hq, int Hkv, int window, float scale,
                        const float *table, int *status, cudaStream_t s);

// Chunked prefill over a cache (chunk.cu)
cudaError_t launch_prefill_gather(const gqa_kv_desc *desc, const void *k_new, const void *v_new,
                                  int T, int Hkv, int d, void *k_out, void *v_out, int S,
                                  const float *table, int table_len, int *status,
                                  cudaStream_t s);
cudaError_t launch_kv_append_chunk(gqa_kv_desc *descs, int nseq, const void *k_new,
                                   const void *v_new, int T, int Hkv, int d, int *status,
                                   cudaStream_t s);

// Q/K RMSNorm, K RoPE and cache append (qknorm.cu)
cudaError_t launch_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out,
                                void *k_rot, int B, int Hq, int Hkv, int T, int d, int pos0,
                                const float *q_gamma, const float *k_gamma, float eps,
                                const float *table, int kv_shared, cudaStream_t s);
cudaError_t launch_qk_norm_append(gqa_kv_desc *descs, int nseq, const void *q, const void *k_new,
                                  const void *v_new, int Hq, int Hkv, int d,
                                  const float *q_gamma, const float *k_gamma, float eps,
                                  int v_norm, void *q_out, int32_t *slots, int *status,
                                  cudaStream_t s);

// Bounded-wait self-test (watchdog.cu)
cudaError_t launch_watchdog_selftest(int64_t limit_ns, int *status, cudaStream_t s);

}  // namespace gqa
