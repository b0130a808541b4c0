// kv.cu -- append one token's K and V per sequence to its cache.
//
// "PLaMo 3アーキテクチャ徹底解析" §4.4: the cache stores K before RoPE and V as projected.
// Global layers keep every token (linear cache: slot = tokens held); local layers keep
// the newest W-1 tokens plus the new one, which a ring of capacity W holds exactly:
// token i goes to slot i mod W and overwrites the token that just left the window.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {

// One block per sequence.  Thread 0 reads the count, every thread copies 16-byte chunks
// of the Hkv new K and V rows, then thread 0 publishes count + 1 and the slot.
__global__ void kv_append_kernel(gqa_kv_desc *descs, const uint4 *__restrict__ k_new,
                                 const uint4 *__restrict__ v_new, int Hkv, int d,
                                 int32_t *slots, int *status) {
    __shared__ int s_slot;
    griddep_wait();               // the descriptors and caches of earlier kernels
    griddep_launch_dependents();  // the decode kernels may start launching
    const int seq = blockIdx.x;
    gqa_kv_desc *desc = descs + seq;
    if (threadIdx.x == 0) {
        const int cap = desc->cap;
        const int count = desc->count;
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
    if (slot >= 0 && GQA_IN_BOUNDS(slot, desc->cap, status, (kDiagCache << 24) | 1)) {
        const int cpr = d / 8;  // 16-byte chunks per row
        const long cap = desc->cap;
        uint4 *kc = static_cast<uint4 *>(desc->k);
        uint4 *vc = static_cast<uint4 *>(desc->v);
        for (int i = threadIdx.x; i < Hkv * cpr; i += blockDim.x) {
            const int g = i / cpr, c = i - g * cpr;
            const long dst = ((long)g * cap + slot) * cpr + c;
            const long src = ((long)seq * Hkv + g) * cpr + c;
            kc[dst] = k_new[src];
            vc[dst] = v_new[src];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (slot >= 0) desc->count = desc->count + 1;
        if (slots) slots[seq] = slot;
    }
}

cudaError_t launch_kv_append(gqa_kv_desc *descs, int nseq, const void *k_new,
                             const void *v_new, int Hkv, int d, int32_t *slots, int *status,
                             cudaStream_t s) {
    return launch_pdl(kv_append_kernel, dim3(nseq), dim3(128), 0, s, descs,
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), Hkv,
                      d, slots, status);
}

}  // namespace gqa
