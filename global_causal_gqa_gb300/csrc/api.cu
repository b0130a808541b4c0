// api.cu -- the extern "C" entry points declared in gqa_attn.h.
//
// Host-side argument checks, the per-device status word, and launches on the caller's
// stream.  No entry point allocates memory or synchronises, except
// gqa_get_device_status (which synchronises the given stream to read the status word).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <set>
#include <utility>

#include "gqa_attn.h"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

// One status word per device.  Kernels record the first device-side error here with
// atomicCAS; gqa_get_device_status reads and clears it.
// Word 0: status; word 1: diagnostic code of the first device-side wait that expired;
// words 2-5: the first expired wait of each kernel role (0-3).
__device__ int g_status_word[6];

int *status_ptr() {
    static std::mutex mu;
    static int *ptrs[kMaxDevices] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int *>(p);
    }
    return ptrs[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool rope_dim_ok(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }

// The CUDA error behind the most recent GQA_ERR_CUDA returned on this host thread.
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

gqa_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return GQA_OK;
    t_last_cuda_error = e;
    return GQA_ERR_CUDA;
}

}  // namespace

namespace gqa {

cudaError_t ensure_smem_attr(const void *func, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;   // (kernel, device)
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({func, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({func, dev});
    return e;
}

}  // namespace gqa

extern "C" {

gqa_status gqa_rope_inv_freq(double *out, int d, double base, double yarn_factor,
                             double yarn_L0, double beta_fast, double beta_slow,
                             double rotate_fraction) {
    if (!out || d <= 0 || (d % 2) != 0 || !(base > 1.0) || !(yarn_factor >= 1.0) ||
        !(rotate_fraction > 0.0 && rotate_fraction <= 1.0))
        return GQA_ERR_INVALID_ARG;
    const int half = d / 2;
    const bool yarn = yarn_factor != 1.0;
    double lo = 0.0, hi = 1.0;
    if (yarn) {
        if (!(yarn_L0 > 0.0) || !(beta_fast > 0.0) || !(beta_slow > 0.0) || beta_fast == beta_slow)
            return GQA_ERR_INVALID_ARG;
        const double two_pi = 6.283185307179586476925286766559;
        lo = half * std::log(yarn_L0 / (two_pi * beta_fast)) / std::log(base);
        hi = half * std::log(yarn_L0 / (two_pi * beta_slow)) / std::log(base);
    }
    const int rotated = rotate_fraction < 1.0
                            ? static_cast<int>(std::floor(rotate_fraction * half + 0.5))
                            : half;
    for (int j = 0; j < half; ++j) {
        double w = std::pow(base, -2.0 * j / d);
        if (yarn) {
            double a = (j - lo) / (hi - lo);
            a = a < 0.0 ? 0.0 : (a > 1.0 ? 1.0 : a);
            w *= (1.0 - a) + a / yarn_factor;
        }
        out[j] = j < rotated ? w : 0.0;
    }
    return GQA_OK;
}

double gqa_yarn_amplitude(double s) { return 1.0 + 0.1 * std::log(s); }

size_t gqa_rope_table_bytes(int d, int max_pos) {
    if (d <= 0 || max_pos <= 0) return 0;
    return static_cast<size_t>(max_pos) * (d / 2) * 2 * sizeof(float);
}

gqa_status gqa_rope_table_build(float *table, const double *inv_freq, int d, double amp,
                                int max_pos, gqa_stream_t stream) {
    if (!table || !inv_freq || !rope_dim_ok(d) || max_pos <= 0 || !std::isfinite(amp) ||
        !(amp > 0.0))
        return GQA_ERR_INVALID_ARG;
    if (!aligned16(table)) return GQA_ERR_ALIGNMENT;
    gqa::InvFreq w{};
    for (int j = 0; j < d / 2; ++j) w.w[j] = inv_freq[j];
    return from_cuda(gqa::launch_rope_table(table, w, d, amp, max_pos,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_rope_apply(const void *x, void *y, int B, int H, int T, int d, int pos0,
                          const float *table, int table_len, gqa_stream_t stream) {
    if (!x || !y || !table || B <= 0 || H <= 0 || T <= 0 || table_len <= 0 || pos0 < 0)
        return GQA_ERR_INVALID_ARG;
    if (!rope_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(y) || !aligned16(table)) return GQA_ERR_ALIGNMENT;
    if (static_cast<long>(pos0) + T > table_len) return GQA_ERR_RANGE;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_rope_apply(x, y, static_cast<long>(B) * H * T, T, d, pos0,
                                            table, table_len, st,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

size_t gqa_prefill_workspace_bytes(int B, int Hkv, int S, int d) {
    if (B <= 0 || Hkv <= 0 || S <= 0 || d <= 0) return 0;
    return static_cast<size_t>(B) * Hkv * S * d * 2;
}

gqa_status gqa_attn_prefill(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int T, int S, int Hq, int Hkv, int d, int window,
                            float scale, const float *table, int table_len, int k_is_rotated,
                            void *workspace, size_t workspace_bytes, gqa_stream_t stream) {
    if (!q || !k || !v || !o || !table || B <= 0 || T <= 0 || S <= 0 || T > S || Hq <= 0 ||
        Hkv <= 0 || (Hq % Hkv) != 0 || !(scale > 0.f) || !std::isfinite(scale) ||
        k_is_rotated < 0 || k_is_rotated > 2)
        return GQA_ERR_INVALID_ARG;
    if (d != 128 && d != 256 && d != 512) return GQA_ERR_UNSUPPORTED;
    if (k_is_rotated == 2 && d != 128) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(table) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return GQA_ERR_ALIGNMENT;
    if (table_len < S) return GQA_ERR_RANGE;
    if (k_is_rotated == 0) {
        const size_t need = gqa_prefill_workspace_bytes(B, Hkv, S, d);
        if (!workspace || workspace_bytes < need) return GQA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return GQA_ERR_ALIGNMENT;
    }
    // the grid: one CTA per (b, KV head, head pair, 128-row block) for d = 128, per
    // (b, head, 128-row block) for d = 256, four per (b, KV head, head pair, 128-row block)
    // for d = 512
    const long mblocks = (T + 127) / 128;
    const long hpairs = static_cast<long>(B) * Hkv * ((Hq / Hkv + 1) / 2) * mblocks;
    const long blocks = d == 128 ? hpairs : d == 512 ? 4 * hpairs : static_cast<long>(B) * Hq * mblocks;
    if (blocks > 0x7fffffffL) return GQA_ERR_UNSUPPORTED;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // K rotated once at positions 0..S-1 into the workspace; Q is rotated inside the
    // attention kernel as each tile lands.
    const void *k_rot = k;
    if (k_is_rotated == 0) {
        cudaError_t e = gqa::launch_rope_apply(k, workspace, static_cast<long>(B) * Hkv * S, S,
                                               d, 0, table, table_len, st, s);
        if (e != cudaSuccess) return GQA_ERR_CUDA;
        k_rot = workspace;
    }
    const int rc = d == 128 ? gqa::launch_prefill(q, k_rot, v, o, lse, B, T, S, Hq, Hkv, d,
                                                  window, scale, table, table_len, st, s,
                                                  k_is_rotated == 2)
                            : gqa::launch_prefill_wide(q, k_rot, v, o, lse, B, T, S, Hq, Hkv,
                                                       d, window, scale, table, st, s);
    if (rc == GQA_ERR_CUDA) t_last_cuda_error = cudaGetLastError();
    return static_cast<gqa_status>(rc);
}

gqa_status gqa_kv_append(gqa_kv_desc *descs, int nseq, const void *k_new, const void *v_new,
                         int Hkv, int d, int32_t *slots_out, gqa_stream_t stream) {
    if (!descs || !k_new || !v_new || nseq <= 0 || Hkv <= 0) return GQA_ERR_INVALID_ARG;
    if (!rope_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(descs) & 7u))
        return GQA_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_kv_append(descs, nseq, k_new, v_new, Hkv, d, slots_out, st,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_prefill_gather(const gqa_kv_desc *desc, const void *k_new, const void *v_new,
                              int T, int Hkv, int d, void *k_out, void *v_out, int S,
                              const float *table, int table_len, gqa_stream_t stream) {
    if (!desc || !k_new || !v_new || !k_out || !v_out || !table || T <= 0 || Hkv <= 0 ||
        S < T || table_len <= 0)
        return GQA_ERR_INVALID_ARG;
    if (!rope_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_out) || !aligned16(v_out) ||
        !aligned16(table) || (reinterpret_cast<uintptr_t>(desc) & 7u))
        return GQA_ERR_ALIGNMENT;
    if (S > table_len) return GQA_ERR_RANGE;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_prefill_gather(desc, k_new, v_new, T, Hkv, d, k_out, v_out, S,
                                                table, table_len, st,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_kv_append_chunk(gqa_kv_desc *descs, int nseq, const void *k_new,
                               const void *v_new, int T, int Hkv, int d, gqa_stream_t stream) {
    if (!descs || !k_new || !v_new || nseq <= 0 || T <= 0 || Hkv <= 0)
        return GQA_ERR_INVALID_ARG;
    if (!rope_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(descs) & 7u))
        return GQA_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_kv_append_chunk(descs, nseq, k_new, v_new, T, Hkv, d, st,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out, void *k_rot,
                            int B, int Hq, int Hkv, int T, int d, int pos0,
                            const float *q_gamma, const float *k_gamma, float eps,
                            const float *table, int table_len, gqa_stream_t stream) {
    if (!q || !k || !q_out || !q_gamma || !k_gamma || B <= 0 || Hq <= 0 || Hkv <= 0 ||
        T <= 0 || pos0 < 0 || !(eps >= 0.f) || !std::isfinite(eps) || (k_rot && !table))
        return GQA_ERR_INVALID_ARG;
    if (!rope_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(q_out) || (k_out && !aligned16(k_out)) ||
        (k_rot && !aligned16(k_rot)) || !aligned16(q_gamma) || !aligned16(k_gamma) ||
        (table && !aligned16(table)))
        return GQA_ERR_ALIGNMENT;
    if (k_rot && (long)pos0 + T > (long)table_len) return GQA_ERR_RANGE;
    return from_cuda(gqa::launch_qk_norm_rope(q, k, q_out, k_out, k_rot, B, Hq, Hkv, T, d, pos0,
                                              q_gamma, k_gamma, eps, table, 0,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_qk_norm_rope_kv_shared(const void *q, const void *z, void *q_out, void *v_out,
                                      void *k_rot, int B, int Hq, int Hkv, int T, int d,
                                      int pos0, const float *q_gamma, const float *k_gamma,
                                      float eps, const float *table, int table_len,
                                      gqa_stream_t stream) {
    const bool with_q = q != nullptr;
    if (!z || (with_q && (!q_out || !q_gamma || Hq <= 0)) || (!with_q && q_out) ||
        (!v_out && !k_rot) || (k_rot && (!k_gamma || !table)) || B <= 0 || Hkv <= 0 ||
        T <= 0 || pos0 < 0 || !(eps >= 0.f) || !std::isfinite(eps))
        return GQA_ERR_INVALID_ARG;
    if (!rope_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
    if ((with_q && (!aligned16(q) || !aligned16(q_out) || !aligned16(q_gamma))) ||
        !aligned16(z) || (v_out && !aligned16(v_out)) || (k_rot && !aligned16(k_rot)) ||
        (k_gamma && !aligned16(k_gamma)) || (table && !aligned16(table)))
        return GQA_ERR_ALIGNMENT;
    if (k_rot && (long)pos0 + T > (long)table_len) return GQA_ERR_RANGE;
    return from_cuda(gqa::launch_qk_norm_rope(q, z, q_out, v_out, k_rot, B, with_q ? Hq : 0, Hkv,
                                              T, d, pos0, q_gamma, k_gamma, eps, table, 1,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_qk_norm_append(gqa_kv_desc *descs, int nseq, const void *q, const void *k_new,
                              const void *v_new, int Hq, int Hkv, int d, const float *q_gamma,
                              const float *k_gamma, float eps, int v_norm, void *q_out,
                              int32_t *slots_out, gqa_stream_t stream) {
    if (!descs || !q || !k_new || !v_new || !q_out || !q_gamma || !k_gamma || nseq <= 0 ||
        Hq <= 0 || Hkv <= 0 || !(eps >= 0.f) || !std::isfinite(eps) ||
        (v_norm != 0 && v_norm != 1))
        return GQA_ERR_INVALID_ARG;
    if (!rope_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(q_out) ||
        !aligned16(q_gamma) || !aligned16(k_gamma) || (reinterpret_cast<uintptr_t>(descs) & 7u))
        return GQA_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_qk_norm_append(descs, nseq, q, k_new, v_new, Hq, Hkv, d, q_gamma,
                                                k_gamma, eps, v_norm, q_out, slots_out, st,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_kv_shared_append(gqa_kv_desc *descs, int nseq, const void *q, const void *z_new,
                                int Hq, int Hkv, int d, const float *q_gamma, float eps,
                                void *q_out, int32_t *slots_out, gqa_stream_t stream) {
    if (!descs || !q || !z_new || !q_out || !q_gamma || nseq <= 0 || Hq <= 0 || Hkv <= 0 ||
        !(eps >= 0.f) || !std::isfinite(eps))
        return GQA_ERR_INVALID_ARG;
    if (!rope_dim_ok(d)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(z_new) || !aligned16(q_out) || !aligned16(q_gamma) ||
        (reinterpret_cast<uintptr_t>(descs) & 7u))
        return GQA_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_qk_norm_append(descs, nseq, q, z_new, nullptr, Hq, Hkv, d,
                                                q_gamma, nullptr, eps, 0, q_out, slots_out, st,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

size_t gqa_decode_workspace_bytes(int nseq, int Hq, int Hkv, int d, int max_len) {
    if (nseq <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || max_len <= 0) return 0;
    return gqa::decode_workspace_bytes(nseq, Hq, Hkv, d, max_len);
}

gqa_status gqa_attn_decode(const void *q, const gqa_kv_desc *descs, int nseq, int Hq, int Hkv,
                           int d, float scale, int max_len, void *o, float *lse,
                           void *workspace, size_t workspace_bytes, gqa_stream_t stream) {
    if (!q || !descs || !o || nseq <= 0 || Hq <= 0 || Hkv <= 0 || (Hq % Hkv) != 0 ||
        max_len <= 0 || !(scale > 0.f) || !std::isfinite(scale))
        return GQA_ERR_INVALID_ARG;
    if ((d != 128 && d != 256 && d != 512) || Hq / Hkv > 8) return GQA_ERR_UNSUPPORTED;
    if (nseq > 65535) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(o) || (reinterpret_cast<uintptr_t>(descs) & 7u) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return GQA_ERR_ALIGNMENT;
    const size_t need = gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len);
    if (!workspace || workspace_bytes < need) return GQA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GQA_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_decode(q, descs, nseq, Hq, Hkv, d, scale, max_len, o, lse,
                                        static_cast<float *>(workspace), st,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_attn_decode_kv_shared(const void *q, const gqa_kv_desc *descs, int nseq, int Hq,
                                     int Hkv, int d, float scale, const float *k_gamma,
                                     int max_len, void *o, float *lse, void *workspace,
                                     size_t workspace_bytes, gqa_stream_t stream) {
    if (!q || !descs || !o || !k_gamma || nseq <= 0 || Hq <= 0 || Hkv <= 0 ||
        (Hq % Hkv) != 0 || max_len <= 0 || !(scale > 0.f) || !std::isfinite(scale))
        return GQA_ERR_INVALID_ARG;
    if ((d != 128 && d != 256 && d != 512) || Hq / Hkv > 8) return GQA_ERR_UNSUPPORTED;
    if (nseq > 65535) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(o) || !aligned16(k_gamma) ||
        (reinterpret_cast<uintptr_t>(descs) & 7u) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return GQA_ERR_ALIGNMENT;
    const size_t need = gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len);
    if (!workspace || workspace_bytes < need) return GQA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GQA_ERR_ALIGNMENT;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(gqa::launch_decode(q, descs, nseq, Hq, Hkv, d, scale, max_len, o, lse,
                                        static_cast<float *>(workspace), st,
                                        reinterpret_cast<cudaStream_t>(stream), k_gamma));
}

// ---- decode with library-owned scratch (no allocation) ---------------------------------
// Some callers cannot hand the library a workspace: their device memory belongs to another
// component (a framework allocator that has reserved the GPU's memory up front, a serving
// runtime that forbids allocating inside its step loop), or they cannot afford the device
// synchronisation that cudaMalloc/cudaFree imply on every decode step.  For them the
// split-KV partials of one decode call live in this fixed array, compiled into the library
// and present on every GPU that loads it until the process exits.
constexpr size_t kDecodeStaticScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_decode_static_scratch[kDecodeStaticScratchBytes];

// Device address of the array on the current device.  In host code the array's name only
// stands in for the symbol; a kernel must be given this address instead.  Looked up once
// per device, with that device current, on the first call made on it.
static float *decode_static_scratch(void) {
    static std::mutex mu;
    static float *ptrs[kMaxDevices] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_static_scratch) != cudaSuccess || !p) return nullptr;
        ptrs[dev] = static_cast<float *>(p);
    }
    return ptrs[dev];
}

gqa_status gqa_attn_decode_static(const void *q, const gqa_kv_desc *descs, int nseq, int Hq,
                                  int Hkv, int d, float scale, int max_len, void *o,
                                  float *lse, gqa_stream_t stream) {
    if (!q || !descs || !o || nseq <= 0 || Hq <= 0 || Hkv <= 0 || (Hq % Hkv) != 0 ||
        max_len <= 0 || !(scale > 0.f) || !std::isfinite(scale))
        return GQA_ERR_INVALID_ARG;
    if ((d != 128 && d != 256 && d != 512) || Hq / Hkv > 8) return GQA_ERR_UNSUPPORTED;
    if (nseq > 65535) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(o) || (reinterpret_cast<uintptr_t>(descs) & 7u) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return GQA_ERR_ALIGNMENT;
    // the partials of this call must fit the fixed array
    if (gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len) > kDecodeStaticScratchBytes)
        return GQA_ERR_WORKSPACE;
    float *scratch = decode_static_scratch();
    if (!scratch) return GQA_ERR_CUDA;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    // Every partial record the combine pass reads is written earlier in the same call, so
    // nothing left in the array by a previous call is ever read: no clearing is needed.
    return from_cuda(gqa::launch_decode(q, descs, nseq, Hq, Hkv, d, scale, max_len, o, lse,
                                        scratch, st, reinterpret_cast<cudaStream_t>(stream)));
}

gqa_status gqa_get_device_status(gqa_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GQA_ERR_CUDA;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, st, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GQA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return GQA_ERR_CUDA;
    }
    return static_cast<gqa_status>(v);
}

gqa_status gqa_get_device_diag(gqa_stream_t stream, int32_t *diag, int n) {
    if (!diag || n <= 0) return GQA_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GQA_ERR_CUDA;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    int v[5] = {0, 0, 0, 0, 0};
    if (cudaMemcpy(v, st + 1, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GQA_ERR_CUDA;
    for (int i = 0; i < n; ++i) diag[i] = i < 5 ? v[i] : 0;
    const int zero[5] = {0, 0, 0, 0, 0};
    if (cudaMemcpy(st + 1, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return GQA_ERR_CUDA;
    return GQA_OK;
}

gqa_status gqa_watchdog_selftest(int64_t limit_ns, gqa_stream_t stream) {
    if (limit_ns < 1000 || limit_ns > 2000000000LL) return GQA_ERR_INVALID_ARG;
    int *st = status_ptr();
    if (!st) return GQA_ERR_CUDA;
    return from_cuda(
        gqa::launch_watchdog_selftest(limit_ns, st, reinterpret_cast<cudaStream_t>(stream)));
}

const char *gqa_status_string(int status) {
    switch (status) {
        case GQA_OK: return "ok";
        case GQA_ERR_INVALID_ARG: return "invalid argument";
        case GQA_ERR_UNSUPPORTED: return "unsupported shape or device";
        case GQA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case GQA_ERR_CAPACITY: return "cache full or length beyond bound";
        case GQA_ERR_CUDA: return "CUDA runtime error";
        case GQA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case GQA_ERR_WORKSPACE: return "workspace missing or too small";
        case GQA_ERR_RANGE: return "position beyond the RoPE table";
        case GQA_ERR_DEVICE_BOUNDS: return "device-side index check failed (debug build)";
        default: return "unknown status";
    }
}

const char *gqa_last_error_string(void) {
    return t_last_cuda_error == cudaSuccess ? "no CUDA error recorded"
                                            : cudaGetErrorString(t_last_cuda_error);
}

gqa_status gqa_device_check(void) {
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return GQA_ERR_CUDA;
    return (prop.major == 10 && prop.minor == 3) ? GQA_OK : GQA_ERR_UNSUPPORTED;
}

}  // extern "C"
