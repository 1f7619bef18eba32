// Reuse of earlier selections (ClusterKV page, section "Caching the KV of
// selected tokens": the GPU keeps the KV of the tokens selected in the last R
// decode steps, and only clusters missing from that cache are loaded; the
// cache-effectiveness analysis reports its hit rate for R = 1 and R = 2).
//
// With every K/V row resident in HBM nothing is loaded from the host, so here
// the hit count is a measurement: for every unit, the number of tokens of the
// current selection that also belong to at least one of the R previous
// selections (whole clusters are selected, so this is the token-weighted
// cluster hit rate).  One CTA per unit builds a bitmap of the previous
// selections' token ids in shared memory (atomicOr: the result does not depend
// on the order) and counts the current selection's tokens found in it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace ckv {
namespace {

constexpr int REUSE_THREADS = 256;
constexpr int REUSE_MAX_R = 8;

struct PrevSets {
    const int32_t* idx[REUSE_MAX_R];
    const int32_t* cnt[REUSE_MAX_R];
};

__device__ __forceinline__ int clamp_count(int c, int B) { return c < 0 ? 0 : (c > B ? B : c); }

__global__ void __launch_bounds__(REUSE_THREADS) overlap_kernel(PrevSets prev, int R, int B_prev,
                                                                const int32_t* __restrict__ idx_cur,
                                                                const int32_t* __restrict__ cnt_cur, int B_cur,
                                                                int max_len, int nwords, int32_t* __restrict__ hits) {
    extern __shared__ uint32_t bits[];  // [nwords]
    __shared__ int wsum[REUSE_THREADS / 32];
    const int u = blockIdx.x, tid = threadIdx.x;
    for (int i = tid; i < nwords; i += REUSE_THREADS) bits[i] = 0u;
    __syncthreads();
    for (int r = 0; r < R; ++r) {
        const int c = clamp_count(prev.cnt[r][u], B_prev);
        const int32_t* ip = prev.idx[r] + (size_t)u * B_prev;
        for (int p = tid; p < c; p += REUSE_THREADS) {
            const int t = ip[p];
            if ((unsigned)t < (unsigned)max_len) atomicOr(&bits[t >> 5], 1u << (t & 31));
        }
    }
    __syncthreads();
    const int c = clamp_count(cnt_cur[u], B_cur);
    const int32_t* ic = idx_cur + (size_t)u * B_cur;
    int h = 0;
    for (int p = tid; p < c; p += REUSE_THREADS) {
        const int t = ic[p];
        if ((unsigned)t < (unsigned)max_len) h += (bits[t >> 5] >> (t & 31)) & 1u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    if ((tid & 31) == 0) wsum[tid >> 5] = h;
    __syncthreads();
    if (tid == 0) {
        int s = 0;
        for (int w = 0; w < REUSE_THREADS / 32; ++w) s += wsum[w];
        hits[u] = s;
    }
}

}  // namespace
}  // namespace ckv

using namespace ckv;

extern "C" ckv_status ckv_selection_overlap(int32_t units, int32_t max_len, int32_t R, const int32_t* const* idx_prev,
                                            const int32_t* const* cnt_prev, int32_t B_prev, const int32_t* idx_cur,
                                            const int32_t* cnt_cur, int32_t B_cur, int32_t* hits, void* stream) {
    CKV_TRACE("ckv_selection_overlap");
    if (units < 1 || max_len < 1 || R < 0 || R > REUSE_MAX_R || B_prev < 0 || B_cur < 0) return CKV_ERR_ARG;
    if (!idx_cur || !cnt_cur || !hits || (R > 0 && (!idx_prev || !cnt_prev))) return CKV_ERR_ARG;
    PrevSets ps = {};
    for (int r = 0; r < R; ++r) {
        if (!idx_prev[r] || !cnt_prev[r]) return CKV_ERR_ARG;
        ps.idx[r] = idx_prev[r];
        ps.cnt[r] = cnt_prev[r];
    }
    const int nwords = ceil_div(max_len, 32);
    const size_t smem = (size_t)nwords * sizeof(uint32_t);
    if (smem > 200 * 1024) return CKV_ERR_CAPACITY;
    if (cudaFuncSetAttribute(overlap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return CKV_ERR_CUDA;
    overlap_kernel<<<units, REUSE_THREADS, smem, (cudaStream_t)stream>>>(ps, R, B_prev, idx_cur, cnt_cur, B_cur,
                                                                        max_len, nwords, hits);
    return cudaGetLastError() == cudaSuccess ? CKV_OK : CKV_ERR_CUDA;
}
