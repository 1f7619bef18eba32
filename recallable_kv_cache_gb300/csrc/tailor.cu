// Channel pre-score: a cheap alternative scorer over the centroid table, after
// TailorKV's channel contribution (TailorKV page, section on the dynamic
// retrieval of sparsity-friendly layers: channel i contributes
// s_i = |q_i| * max |K_i|, and attention scores are approximated from the
// critical channels only).  Applied to ClusterKV's centroid scoring: the
// query is the sum of the g heads (as in the exact score), K is the centroid
// table, and the score of cluster c is the partial dot product over the r
// channels of largest s_i.
//
//   centroid_channels_kernel  channel-major copy muT[u][i][c] of the scoring
//                             centroids and the per-channel maxima
//                             chmax[u][i] = max_c |mu_c,i| (rebuilt by the
//                             caller whenever the clusters change);
//   prescore_kernel           per unit: channel ranking, then r coalesced row
//                             reads of muT for the scores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace ckv {
namespace {

constexpr int CH_TILE = 64;        // centroids per transpose tile
constexpr int MAX_PRESCORE_R = 32;

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }

// One CTA per (tile of 64 centroids, unit): the tile goes through shared
// memory, every warp then writes whole channel rows (64 consecutive clusters)
// and folds |mu| of its channels into chmax (atomicMax on the bits of
// non-negative floats: the order of the tiles does not matter).
template <typename T>
__global__ void __launch_bounds__(256) centroid_channels_kernel(const T* __restrict__ mu, int cmax, int C,
                                                                T* __restrict__ muT, float* __restrict__ chmax) {
    __shared__ T tile[CH_TILE][D + 1];
    const int u = blockIdx.y, c0 = blockIdx.x * CH_TILE, tid = threadIdx.x;
    const T* src = mu + ((size_t)u * cmax + c0) * D;
    for (int e = tid; e < CH_TILE * D; e += 256) {
        const int c = e / D, i = e % D;
        tile[c][i] = c0 + c < C ? src[(size_t)c * D + i] : T(0.f);
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    for (int i = warp; i < D; i += 8) {
        T* dst = muT + ((size_t)u * D + i) * cmax + c0;
        float m = 0.f;
        for (int c = lane; c < CH_TILE; c += 32) {
            if (c0 + c < C) {
                dst[c] = tile[c][i];
                m = fmaxf(m, fabsf(to_f(tile[c][i])));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) atomicMax(reinterpret_cast<int*>(chmax) + (size_t)u * D + i, __float_as_int(m));
    }
}

// One CTA of 256 threads per unit.  Threads 0..127 own one channel each: the
// head sum qs_i (fp32, heads in order), s_i = |qs_i| * chmax_i, and its rank
// among the 128 channels by (s desc, channel asc), counted against all keys
// in shared memory.  Then every thread scores clusters c = tid, tid + 256, ...
// over the r ranked channels in rank order.
template <typename T, int G>
__global__ void __launch_bounds__(256) prescore_kernel(const T* __restrict__ q, const T* __restrict__ muT,
                                                       const float* __restrict__ chmax, int cmax, int C, int r,
                                                       float* __restrict__ scores, int32_t* __restrict__ channels) {
    __shared__ uint64_t key[D];
    __shared__ float qs_s[D];
    __shared__ int ch[MAX_PRESCORE_R];
    const int u = blockIdx.x, tid = threadIdx.x;
    if (tid < D) {
        float qs = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h) qs += to_f(q[((size_t)u * G + h) * D + tid]);
        const float s = fabsf(qs) * chmax[(size_t)u * D + tid];
        qs_s[tid] = qs;
        // larger key = larger s, then lower channel; s >= 0 so its bits order like its value
        key[tid] = ((uint64_t)__float_as_uint(s) << 8) | (uint64_t)(D - 1 - tid);
    }
    __syncthreads();
    if (tid < D) {
        const uint64_t k = key[tid];
        int rank = 0;
        for (int j = 0; j < D; ++j) rank += key[j] > k;
        if (rank < r) ch[rank] = tid;
    }
    __syncthreads();
    if (channels && tid < r) channels[(size_t)u * r + tid] = ch[tid];
    const T* mu_u = muT + (size_t)u * D * cmax;
    for (int c = tid; c < C; c += 256) {
        float acc = 0.f;
        for (int j = 0; j < r; ++j) {
            const int i = ch[j];
            acc = fmaf(qs_s[i], to_f(mu_u[(size_t)i * cmax + c]), acc);
        }
        scores[(size_t)u * C + c] = acc;
    }
}

template <typename T>
cudaError_t prescore_g(const void* q, const void* muT, const float* chmax, int units, int g, int cmax, int C, int r,
                       float* scores, int32_t* channels, cudaStream_t s) {
    const T* qq = static_cast<const T*>(q);
    const T* mt = static_cast<const T*>(muT);
    switch (g) {
        case 1: prescore_kernel<T, 1><<<units, 256, 0, s>>>(qq, mt, chmax, cmax, C, r, scores, channels); break;
        case 2: prescore_kernel<T, 2><<<units, 256, 0, s>>>(qq, mt, chmax, cmax, C, r, scores, channels); break;
        case 4: prescore_kernel<T, 4><<<units, 256, 0, s>>>(qq, mt, chmax, cmax, C, r, scores, channels); break;
        case 8: prescore_kernel<T, 8><<<units, 256, 0, s>>>(qq, mt, chmax, cmax, C, r, scores, channels); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ckv

using namespace ckv;

extern "C" ckv_status ckv_centroid_channels(ckv_ctx* ctx, void* muT, float* chmax, void* stream) {
    CKV_TRACE("ckv_centroid_channels");
    if (!ctx || !muT || !chmax) return CKV_ERR_ARG;
    if (!aligned16(muT) || !aligned16(chmax)) return CKV_ERR_ALIGN;
    if (ctx->n_clusters <= 0) return CKV_ERR_STATE;
    cudaStream_t s = (cudaStream_t)stream;
    const int U = ctx->cfg.units, C = ctx->n_clusters;
    if (cudaMemsetAsync(chmax, 0, (size_t)U * D * sizeof(float), s) != cudaSuccess) return CKV_ERR_CUDA;
    const dim3 grid(ceil_div(C, CH_TILE), U);
    if (ctx->cfg.kv_dtype == CKV_BF16)
        centroid_channels_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(ctx->mu_s), ctx->cmax, C, static_cast<__nv_bfloat16*>(muT), chmax);
    else
        centroid_channels_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(ctx->mu_s), ctx->cmax, C,
                                                             static_cast<float*>(muT), chmax);
    return cudaGetLastError() == cudaSuccess ? CKV_OK : CKV_ERR_CUDA;
}

extern "C" ckv_status ckv_channel_prescore(ckv_ctx* ctx, const void* q, int32_t q_dtype, const void* muT,
                                           const float* chmax, int32_t r, float* scores, int32_t* channels,
                                           void* stream) {
    CKV_TRACE("ckv_channel_prescore");
    if (!ctx || !q || !muT || !chmax || !scores) return CKV_ERR_ARG;
    if (q_dtype != ctx->cfg.kv_dtype) return CKV_ERR_DTYPE;
    if (r < 1 || r > MAX_PRESCORE_R) return CKV_ERR_ARG;
    if (ctx->n_clusters <= 0) return CKV_ERR_STATE;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    const int U = ctx->cfg.units, g = ctx->cfg.g, C = ctx->n_clusters;
    const cudaError_t e =
        ctx->cfg.kv_dtype == CKV_BF16
            ? prescore_g<__nv_bfloat16>(q, muT, chmax, U, g, ctx->cmax, C, r, scores, channels, s)
            : prescore_g<float>(q, muT, chmax, U, g, ctx->cmax, C, r, scores, channels, s);
    if (e == cudaErrorInvalidValue) return CKV_ERR_ARG;
    return e == cudaSuccess ? CKV_OK : CKV_ERR_CUDA;
}
