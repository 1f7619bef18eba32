// Appending keys and values to the caches (ClusterKV page, section "Clustering
// in semantic space", clustering strategy during inference: every generated
// token's key and value join the KV cache and stay pending, attended in full,
// until the next block of m tokens is clustered; the prompt's K/V are the
// cache the prefill clustering reads).
//
// For every unit, rows [0, n) of the sources go to rows [pos, pos + n) of K
// and V.  The copy runs on the SMs in 16-byte vectors, several in flight per
// lane, so the sources may be device memory or pinned host memory that the
// device maps: then the rows cross the host link inside this kernel, with no
// separate copy (one row per unit for a decode step; a whole prompt at once).
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace ckv {
namespace {

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_UNROLL = 4;  // 16-byte vectors in flight per lane and tensor

// grid (row blocks, units): block b of unit u copies the chunks
// [b * span, (b + 1) * span) of the unit's n rows (chunks = 16-byte pieces,
// `cpr` per row).
__global__ void __launch_bounds__(APPEND_THREADS) append_kv_kernel(const uint4* __restrict__ k_src,
                                                                   const uint4* __restrict__ v_src, size_t src_stride,
                                                                   size_t n_chunks, size_t span, size_t dst_stride,
                                                                   size_t dst_off, uint4* __restrict__ K,
                                                                   uint4* __restrict__ V) {
    // the caller's previous kernels may still read or write the caches
    ptx::grid_dependency_wait();
    ptx::allow_dependent_launch();
    const int u = blockIdx.y;
    const size_t c0 = (size_t)blockIdx.x * span;
    const size_t c1 = c0 + span < n_chunks ? c0 + span : n_chunks;
    const uint4* ks = k_src + (size_t)u * src_stride;
    const uint4* vs = v_src + (size_t)u * src_stride;
    uint4* kd = K + (size_t)u * dst_stride + dst_off;
    uint4* vd = V + (size_t)u * dst_stride + dst_off;
    for (size_t c = c0 + threadIdx.x; c < c1; c += (size_t)APPEND_THREADS * APPEND_UNROLL) {
        uint4 kr[APPEND_UNROLL], vr[APPEND_UNROLL];
#pragma unroll
        for (int j = 0; j < APPEND_UNROLL; ++j) {
            const size_t cj = c + (size_t)j * APPEND_THREADS;
            if (cj < c1) {
                kr[j] = ks[cj];
                vr[j] = vs[cj];
            }
        }
#pragma unroll
        for (int j = 0; j < APPEND_UNROLL; ++j) {
            const size_t cj = c + (size_t)j * APPEND_THREADS;
            if (cj < c1) {
                kd[cj] = kr[j];
                vd[cj] = vr[j];
            }
        }
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ckv

using namespace ckv;

extern "C" ckv_status ckv_append_kv(const void* k_src, const void* v_src, int32_t src_len, int32_t kv_dtype,
                                    int32_t units, int32_t max_len, int32_t pos, int32_t n, void* K, void* V,
                                    void* stream) {
    if (!k_src || !v_src || !K || !V) return CKV_ERR_ARG;
    if (kv_dtype != CKV_F32 && kv_dtype != CKV_BF16) return CKV_ERR_DTYPE;
    if (units < 1 || max_len < 1 || n < 1 || src_len < n || pos < 0 || pos > max_len - n) return CKV_ERR_ARG;
    if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(K) || !aligned16(V)) return CKV_ERR_ALIGN;
    const int elem = kv_dtype == CKV_BF16 ? 2 : 4;
    const size_t cpr = (size_t)D * elem / 16;  // 16-byte chunks per row
    const size_t n_chunks = (size_t)n * cpr;
    // up to 256 KB of each tensor per CTA
    const size_t span = (size_t)APPEND_THREADS * APPEND_UNROLL * 16;
    const size_t blocks = (n_chunks + span - 1) / span;
    if (blocks > 0x7fffffffu || units > 65535) return CKV_ERR_ARG;
    CKV_TRACE("ckv_append_kv");
    const cudaError_t e = launch_dependent(
        append_kv_kernel, dim3((unsigned)blocks, units), dim3(APPEND_THREADS), 0, (cudaStream_t)stream,
        static_cast<const uint4*>(k_src), static_cast<const uint4*>(v_src), (size_t)src_len * cpr, n_chunks, span,
        (size_t)max_len * cpr, (size_t)pos * cpr, static_cast<uint4*>(K), static_cast<uint4*>(V));
    return e == cudaSuccess ? CKV_OK : CKV_ERR_CUDA;
}
