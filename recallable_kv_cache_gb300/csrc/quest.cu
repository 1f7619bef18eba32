// Page-granular selection, the comparator the ClusterKV page measures itself
// against (Quest; ClusterKV page, section "Background and design principles",
// drawbacks of existing recallable compression; pages of 16 tokens, Fig. 3b):
// pages of consecutive clustered tokens, each weighted by the upper bound of
// q . k over its tokens, sum_i max(q_i * max_i, q_i * min_i), with the
// per-channel maximum and minimum keys of the page (summed over the g query
// heads).  The selection itself (whole pages by descending weight up to the
// budget, the last trimmed) is the cluster selection with one cluster per
// page, so these two kernels only produce the page metadata and the weights.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace ckv {
namespace {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ void load4f(const __nv_bfloat16* p, float (&f)[4]) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
}
__device__ __forceinline__ void load4f(const float* p, float (&f)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x;
    f[1] = v.y;
    f[2] = v.z;
    f[3] = v.w;
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float (&f)[4]) {
    // the values are keys of this dtype: the conversion is exact
    uint2 w;
    w.x = (__float_as_uint(f[0]) >> 16) | (__float_as_uint(f[1]) & 0xffff0000u);
    w.y = (__float_as_uint(f[2]) >> 16) | (__float_as_uint(f[3]) & 0xffff0000u);
    *reinterpret_cast<uint2*>(p) = w;
}
__device__ __forceinline__ void store4(float* p, const float (&f)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
}

// One warp per page, lane l owns channels 4l .. 4l + 3.
template <typename T>
__global__ void __launch_bounds__(256) quest_pages_kernel(const T* __restrict__ K, int max_len, int sinks, int L,
                                                          int n_pages, T* __restrict__ pmax, T* __restrict__ pmin) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.y, p = blockIdx.x * 8 + warp;
    if (p >= n_pages) return;
    const int t0 = sinks + p * QUEST_PAGE, t1 = min(L, t0 + QUEST_PAGE);
    float mx[4], mn[4];
    load4f(K + ((size_t)u * max_len + t0) * D + 4 * lane, mx);
#pragma unroll
    for (int e = 0; e < 4; ++e) mn[e] = mx[e];
    for (int t = t0 + 1; t < t1; ++t) {
        float f[4];
        load4f(K + ((size_t)u * max_len + t) * D + 4 * lane, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            mx[e] = fmaxf(mx[e], f[e]);
            mn[e] = fminf(mn[e], f[e]);
        }
    }
    const size_t o = ((size_t)u * n_pages + p) * D + 4 * lane;
    store4(pmax + o, mx);
    store4(pmin + o, mn);
}

// One warp per page: weight = sum_h sum_i max(q_hi * max_i, q_hi * min_i),
// fp32 (each product of two values of the K/V dtype is exact in fp32).
template <typename T, int G>
__global__ void __launch_bounds__(256) quest_score_kernel(const T* __restrict__ q, const T* __restrict__ pmax,
                                                          const T* __restrict__ pmin, int n_pages,
                                                          float* __restrict__ scores) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.y, p = blockIdx.x * 8 + warp;
    if (p >= n_pages) return;
    float mx[4], mn[4];
    const size_t o = ((size_t)u * n_pages + p) * D + 4 * lane;
    load4f(pmax + o, mx);
    load4f(pmin + o, mn);
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float qh[4];
        load4f(q + ((size_t)u * G + h) * D + 4 * lane, qh);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc += fmaxf(qh[e] * mx[e], qh[e] * mn[e]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(FULL, acc, off);
    if (lane == 0) scores[(size_t)u * n_pages + p] = acc;
}

template <typename T>
cudaError_t score_g(const void* q, const void* pmax, const void* pmin, int units, int g, int n_pages, float* scores,
                    cudaStream_t s) {
    const dim3 grid(ceil_div(n_pages, 8), units);
    const T* qq = static_cast<const T*>(q);
    const T* mx = static_cast<const T*>(pmax);
    const T* mn = static_cast<const T*>(pmin);
    switch (g) {
        case 1: quest_score_kernel<T, 1><<<grid, 256, 0, s>>>(qq, mx, mn, n_pages, scores); break;
        case 2: quest_score_kernel<T, 2><<<grid, 256, 0, s>>>(qq, mx, mn, n_pages, scores); break;
        case 4: quest_score_kernel<T, 4><<<grid, 256, 0, s>>>(qq, mx, mn, n_pages, scores); break;
        case 8: quest_score_kernel<T, 8><<<grid, 256, 0, s>>>(qq, mx, mn, n_pages, scores); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ckv

using namespace ckv;

extern "C" ckv_status ckv_quest_pages(const void* K, int32_t kv_dtype, int32_t units, int32_t max_len, int32_t sinks,
                                      int32_t L, void* page_max, void* page_min, void* stream) {
    CKV_TRACE("ckv_quest_pages");
    if (!K || !page_max || !page_min) return CKV_ERR_ARG;
    if (kv_dtype != CKV_F32 && kv_dtype != CKV_BF16) return CKV_ERR_DTYPE;
    if (units < 1 || sinks < 0 || L <= sinks || L > max_len) return CKV_ERR_ARG;
    if (!aligned16(K) || !aligned16(page_max) || !aligned16(page_min)) return CKV_ERR_ALIGN;
    const int n_pages = ceil_div(L - sinks, QUEST_PAGE);
    const dim3 grid(ceil_div(n_pages, 8), units);
    cudaStream_t s = (cudaStream_t)stream;
    if (kv_dtype == CKV_BF16)
        quest_pages_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(K), max_len, sinks,
                                                              L, n_pages, static_cast<__nv_bfloat16*>(page_max),
                                                              static_cast<__nv_bfloat16*>(page_min));
    else
        quest_pages_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(K), max_len, sinks, L, n_pages,
                                                      static_cast<float*>(page_max), static_cast<float*>(page_min));
    return cudaGetLastError() == cudaSuccess ? CKV_OK : CKV_ERR_CUDA;
}

extern "C" ckv_status ckv_quest_score(const void* q, int32_t q_dtype, const void* page_max, const void* page_min,
                                      int32_t units, int32_t g, int32_t n_pages, float* scores, void* stream) {
    CKV_TRACE("ckv_quest_score");
    if (!q || !page_max || !page_min || !scores) return CKV_ERR_ARG;
    if (q_dtype != CKV_F32 && q_dtype != CKV_BF16) return CKV_ERR_DTYPE;
    if (units < 1 || n_pages < 1) return CKV_ERR_ARG;
    if (!aligned16(q) || !aligned16(page_max) || !aligned16(page_min)) return CKV_ERR_ALIGN;
    cudaStream_t s = (cudaStream_t)stream;
    const cudaError_t e = q_dtype == CKV_BF16
                              ? score_g<__nv_bfloat16>(q, page_max, page_min, units, g, n_pages, scores, s)
                              : score_g<float>(q, page_max, page_min, units, g, n_pages, scores, s);
    if (e == cudaErrorInvalidValue) return CKV_ERR_ARG;
    return e == cudaSuccess ? CKV_OK : CKV_ERR_CUDA;
}
