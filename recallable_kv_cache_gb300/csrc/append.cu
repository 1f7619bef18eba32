// Appending a decode step's K/V to the caches (ClusterKV page, section
// "Clustering in semantic space", clustering strategy during inference: every
// generated token's key and value join the KV cache and stay pending, attended
// in full, until the next block of m tokens is clustered).
//
// One warp per unit copies the unit's new K row and V row (d elements each,
// 16 bytes per lane) into row `pos` of K and V.  The sources may be device
// memory or pinned host memory that the device maps (then the rows cross the
// host link inside this kernel, with no separate copy).
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace ckv {
namespace {

// 16-byte chunks per row: D * elem / 16 (16 for bf16, 32 for fp32)
__global__ void __launch_bounds__(256) append_kv_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new, int units, int chunks,
                                                        size_t row_stride, size_t pos_off, uint4* __restrict__ K,
                                                        uint4* __restrict__ V) {
    const int u = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (u >= units) return;
    for (int c = lane; c < chunks; c += 32) {
        K[(size_t)u * row_stride + pos_off + c] = k_new[(size_t)u * chunks + c];
        V[(size_t)u * row_stride + pos_off + c] = v_new[(size_t)u * chunks + c];
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ckv

using namespace ckv;

extern "C" ckv_status ckv_append_kv(const void* k_new, const void* v_new, int32_t kv_dtype, int32_t units,
                                    int32_t max_len, int32_t pos, void* K, void* V, void* stream) {
    if (!k_new || !v_new || !K || !V) return CKV_ERR_ARG;
    if (kv_dtype != CKV_F32 && kv_dtype != CKV_BF16) return CKV_ERR_DTYPE;
    if (units < 1 || max_len < 1 || pos < 0 || pos >= max_len) return CKV_ERR_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(K) || !aligned16(V)) return CKV_ERR_ALIGN;
    const int elem = kv_dtype == CKV_BF16 ? 2 : 4;
    const int chunks = D * elem / 16;
    const size_t row_stride = (size_t)max_len * chunks;  // per unit, in 16-byte chunks
    append_kv_kernel<<<ceil_div(units, 8), 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), units, chunks, row_stride,
        (size_t)pos * chunks, static_cast<uint4*>(K), static_cast<uint4*>(V));
    return cudaGetLastError() == cudaSuccess ? CKV_OK : CKV_ERR_CUDA;
}
