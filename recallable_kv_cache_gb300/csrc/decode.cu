// Decode-step kernels of the ClusterKV path:
//   score_kernel   cluster scores q . mu (section "Selection at semantic-cluster
//                  granularity"), a many-CTA stream over the centroid table
//                  (above 1024 clusters, and for ckv_score);
//   sel_kernel     (scores of the unit's clusters, up to 1024 of them,) rank
//                  clusters, prefix-sum their sizes, trim the last one and
//                  compact the token ids (section "Selection and indexing
//                  mechanism", Fig. 8), one CTA per unit;
//   attn_kernel    fp32 K/V: gather of the selected rows with bulk-async
//                  copies into shared memory and split-K flash-decode attention
//                  (section "Background": softmax(q K_S^T / sqrt(d)) V_S);
//                  attn_combine_kernel merges the split partials.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace ckv {
namespace {

constexpr unsigned FULL = 0xffffffffu;

template <typename T>
struct Vec;  // 16-byte chunk of a row -> floats
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4& w, float (&f)[8]) {
        f[0] = __uint_as_float(w.x << 16);
        f[1] = __uint_as_float(w.x & 0xffff0000u);
        f[2] = __uint_as_float(w.y << 16);
        f[3] = __uint_as_float(w.y & 0xffff0000u);
        f[4] = __uint_as_float(w.z << 16);
        f[5] = __uint_as_float(w.z & 0xffff0000u);
        f[6] = __uint_as_float(w.w << 16);
        f[7] = __uint_as_float(w.w & 0xffff0000u);
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4& w, float (&f)[4]) {
        f[0] = __uint_as_float(w.x);
        f[1] = __uint_as_float(w.y);
        f[2] = __uint_as_float(w.z);
        f[3] = __uint_as_float(w.w);
    }
};

__device__ __forceinline__ void set_err(int32_t* err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// ============================================================================
// scoring: scores[u][c] = sum_h q_h . mu_c = (sum_h q_h) . mu_c
// ============================================================================
constexpr int SCORE_UNROLL = 4;  // centroid rows in flight per lane group

template <typename T, int G>
__global__ void __launch_bounds__(256) score_kernel(const T* __restrict__ q,
                                                   const T* __restrict__ mu, int cmax, int C,
                                                   float* __restrict__ scores, int stride,
                                                   const int32_t* __restrict__ pf_sizes,
                                                   const int32_t* __restrict__ pf_offsets) {
    constexpr int CPL = Vec<T>::N;   // channels per lane
    constexpr int LPR = D / CPL;     // lanes per centroid row
    constexpr int RPI = 32 / LPR;    // rows per warp-wide load
    constexpr int UNROLL = SCORE_UNROLL;
    const int u = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPR, li = lane % LPR;
    ptx::grid_dependency_wait();  // q may come from the previous kernel
    ptx::allow_dependent_launch();
    // the selection that follows reads this unit's sizes and offsets first:
    // one warp of the unit's first block pulls those rows into L2 meanwhile
    if (pf_sizes && blockIdx.x == 0 && warp == 7) {
        for (int b = lane * 32; b < C + 1; b += 32 * 32) {
            if (b < C) ptx::prefetch_l2(pf_sizes + (size_t)u * cmax + b);
            ptx::prefetch_l2(pf_offsets + (size_t)u * (cmax + 1) + b);
        }
    }

    float qs[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) qs[c] = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint4 w = *reinterpret_cast<const uint4*>(q + ((size_t)u * G + h) * D + li * CPL);
        float f[CPL];
        Vec<T>::unpack(w, f);
#pragma unroll
        for (int c = 0; c < CPL; ++c) qs[c] += f[c];
    }

    const int row0 = (blockIdx.x * 8 + warp) * (RPI * UNROLL);
    uint4 v[UNROLL];
#pragma unroll
    for (int i = 0; i < UNROLL; ++i) {
        const int r = row0 + i * RPI + sub;
        v[i] = r < C ? *reinterpret_cast<const uint4*>(mu + ((size_t)u * cmax + r) * D + li * CPL)
                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < UNROLL; ++i) {
        float f[CPL];
        Vec<T>::unpack(v[i], f);
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) dot = fmaf(qs[c], f[c], dot);
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(FULL, dot, o);
        const int r = row0 + i * RPI + sub;
        if (li == 0 && r < C) scores[(size_t)u * stride + r] = dot;
    }
}

// ============================================================================
// selection: one CTA per unit
// ============================================================================
// ascending bitonic sort of one 64-bit key per lane
__device__ __forceinline__ uint64_t warp_sort32(uint64_t x, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t p = __shfl_xor_sync(FULL, x, j);
            const bool keep_min = ((lane & j) == 0) == ((lane & k) == 0);
            x = keep_min ? (x < p ? x : p) : (x < p ? p : x);
        }
    return x;
}
// a, b ascending across the lanes: the 32 smallest of a and b, ascending
__device__ __forceinline__ uint64_t warp_merge32(uint64_t a, uint64_t b, int lane) {
    const uint64_t br = __shfl_sync(FULL, b, 31 - lane);
    uint64_t x = a < br ? a : br;  // bitonic, holds the 32 smallest
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const uint64_t p = __shfl_xor_sync(FULL, x, j);
        x = (lane & j) ? (x < p ? p : x) : (x < p ? x : p);
    }
    return x;
}

__device__ __forceinline__ uint64_t rank_key(float s, int c) {
    if (s == 0.f) s = 0.f;  // -0 ranks like +0
    const uint32_t b = __float_as_uint(s);
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);  // ascending with s
    return ((uint64_t)(~ord) << 32) | (uint32_t)c;                      // descending score, asc c
}

// Scores of every cluster of unit u computed inside the selection's CTA
// (the same arithmetic as score_kernel, so the same bits): q summed over the
// g heads, then per centroid row LPR lanes take CPL channels each (fma chain
// in channel order) and a shuffle reduction over the row's lanes.  Rows are
// read in rounds of SEL_SCORE_UNROLL rows per lane group, the next round's
// loads in flight while the current one is reduced.  A warp scores at most 32
// rows (C <= N, rounds of nwarps * 2 * UN rows): lane j of the warp keeps
// the rank key of the warp's j-th row (~0 past the last), which the caller
// sorts in registers.  The first round's loads are issued before the barrier
// that publishes the staged q (they do not depend on it), so the two round
// trips overlap; every thread of the CTA calls this.
constexpr int SEL_SCORE_UNROLL = 2;
template <typename T, int G>
__device__ __forceinline__ uint64_t score_unit(const uint4* qsm, const T* __restrict__ mu, int u, int cmax,
                                               int C, int lane, int warp, int nwarps) {
    constexpr int CPL = Vec<T>::N;   // channels per lane
    constexpr int LPR = D / CPL;     // lanes per centroid row
    constexpr int RPI = 32 / LPR;    // rows per warp-wide load
    constexpr int UN = SEL_SCORE_UNROLL;
    const int sub = lane / LPR, li = lane % LPR;
    const T* mu_u = mu + (size_t)u * cmax * D + li * CPL;
    const int per_round = nwarps * RPI * UN;
    auto row_of = [&](int r0, int i) { return r0 + (i * nwarps + warp) * RPI + sub; };
    auto load = [&](int r0, uint4 (&v)[UN]) {
#pragma unroll
        for (int i = 0; i < UN; ++i) {
            const int r = row_of(r0, i);
            v[i] = r < C ? *reinterpret_cast<const uint4*>(mu_u + (size_t)r * D) : make_uint4(0, 0, 0, 0);
        }
    };
    uint4 cur[UN], nxt[UN];
    load(0, cur);
    __syncthreads();  // q staged in qsm
    float qs[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) qs[c] = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint4 w = qsm[(h * D + li * CPL) * (int)sizeof(T) / 16];
        float f[CPL];
        Vec<T>::unpack(w, f);
#pragma unroll
        for (int c = 0; c < CPL; ++c) qs[c] += f[c];
    }
    // this warp's j-th row: round j / (RPI * UN), i = (j / RPI) % UN, sub = j % RPI
    uint64_t key = ~0ull;
    int it = 0;  // (round, i) in order
    for (int r0 = 0; r0 < C; r0 += per_round) {
        if (r0 + per_round < C) load(r0 + per_round, nxt);
#pragma unroll
        for (int i = 0; i < UN; ++i, ++it) {
            float f[CPL];
            Vec<T>::unpack(cur[i], f);
            float dot = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) dot = fmaf(qs[c], f[c], dot);
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(FULL, dot, o);
            // every lane of a row's lane group holds its sum: lane j takes the
            // sum of the row with sub = j % RPI from that group's first lane
            const float mine = __shfl_sync(FULL, dot, (lane % RPI) * LPR);
            const int r = r0 + (i * nwarps + warp) * RPI + lane % RPI;
            if (lane / RPI == it && r < C) key = rank_key(mine, r);
        }
#pragma unroll
        for (int i = 0; i < UN; ++i) cur[i] = nxt[i];
    }
    return key;
}

// One CTA per unit.  Scores (computed by the CTA itself from q and the
// centroid copy up to 1024 clusters, else from score_kernel or the caller)
// become 64-bit keys (descending score, ascending cluster index) that are sorted by a
// bitonic network held in registers: exchange distances below 32 use warp
// shuffles, larger ones shared memory, and distances of at least the block
// size stay inside a thread (E keys per thread).  The sizes taken in rank
// order are prefix-summed, the budget cut found, and every output slot
// p < min(B, total) looks up its rank by binary search and copies its token id
// from the label-sorted permutation.  The sizes and offsets (and given
// scores) are loaded before any of them is used, so they share one round
// trip, which the scoring overlaps.
//
// G == 0: scores_in [units][sstride] are given.  G > 0: the scores are
// computed here from q [units][G][D] and the scoring copy mu [units][cmax][D]
// of type T.
template <int E, typename T, int G>
__global__ void __launch_bounds__(1024, 1) sel_kernel(
    const float* __restrict__ scores_in, int sstride, const T* __restrict__ q, const T* __restrict__ mu, int cmax,
    int C, int N, const int32_t* __restrict__ sizes, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ perm, int ntok, int B, int32_t* __restrict__ idx, int32_t* __restrict__ count,
    int32_t* __restrict__ dev_err) {
    extern __shared__ __align__(16) unsigned char sel_smem[];
    uint64_t* sk = reinterpret_cast<uint64_t*>(sel_smem);  // [N]
    int32_t* start = reinterpret_cast<int32_t*>(sk + N);   // [N]
    int32_t* cl = start + N;                               // [N]
    int32_t* szc = cl + N;                                 // [N] sizes by cluster
    int32_t* offc = szc + N;                               // [N] offsets by cluster
    float* scs = reinterpret_cast<float*>(offc + N);       // [N] scores computed here (the histogram's space)
    __shared__ int32_t wsum[32];
    __shared__ int32_t s_tot;
    const int u = blockIdx.x, tid = threadIdx.x, NT = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = NT >> 5;
    ptx::grid_dependency_wait();    // the scores, the cluster state and idx may come from the previous kernel
    ptx::allow_dependent_launch();

    // ---- 1. sizes / offsets / scores (registers first, shared memory after)
    int szr[E], ofr[E];
    float scr[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int c = e * NT + tid;
        szr[e] = c < C ? sizes[(size_t)u * cmax + c] : 0;
        ofr[e] = c < C ? offsets[(size_t)u * (cmax + 1) + c] : 0;
        if constexpr (G == 0) scr[e] = c < C ? scores_in[(size_t)u * sstride + c] : 0.f;
    }
    uint64_t wkey = ~0ull;  // scored here: this lane's key among its warp's rows
    if constexpr (G > 0) {
        static_assert(E == 1, "scoring in the selection uses one key slot per thread");
        // the unit's q (G rows) into shared memory once: every lane needs it,
        // and q may sit in mapped host memory
        constexpr int QV = G * D * (int)sizeof(T) / 16;
        uint4* qsm = reinterpret_cast<uint4*>(scs + N);
        for (int i = tid; i < QV; i += NT) qsm[i] = reinterpret_cast<const uint4*>(q + (size_t)u * G * D)[i];
        wkey = score_unit<T, G>(qsm, mu, u, cmax, C, lane, warp, nwarps);  // its first barrier publishes qsm
    }
    // ---- 2. unsorted keys (N is a multiple of NT: every slot is written).
    // Given scores: slot c holds cluster c's key.  Scored here: slot 32 w + j
    // holds the key of warp w's j-th row.  Either order serves: every later
    // step takes the cluster from the key; unused slots hold ~0.
    if constexpr (G > 0) {
        sk[tid] = wkey;
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int c = e * NT + tid;
            sk[c] = c < C ? rank_key(scr[e], c) : ~0ull;
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        szc[e * NT + tid] = szr[e];
        offc[e * NT + tid] = ofr[e];
    }

    // ---- 3. fast path: the 32 highest-ranked clusters.  Warp w sorts the E
    // lists of 32 keys it owns (in registers; sk keeps its order) and merges
    // them into its 32 smallest keys (scored here: straight from the scoring's
    // registers, before the barrier); then a merge tree across the warps: at
    // each level the lower half of the remaining lists takes in the upper
    // half (one merge per warp, all warps of a level at once), while the last
    // warp sums the sizes.  If those 32 clusters hold min(B, total) tokens,
    // the selection is a prefix of them and the rest of the ranking is not
    // needed.
    __shared__ int s_fast, s_nsel, s_total;
    uint64_t* part = reinterpret_cast<uint64_t*>(start);  // [nwarps][32] (start/cl reused)
    if constexpr (G > 0) {
        part[32 * warp + lane] = warp_sort32(wkey, lane);
        __syncthreads();  // sk, szc, offc and part
    } else {
        __syncthreads();  // sk, szc, offc
        uint64_t top = warp_sort32(sk[32 * warp + lane], lane);
#pragma unroll
        for (int e = 1; e < E; ++e)
            top = warp_merge32(top, warp_sort32(sk[32 * (warp + e * nwarps) + lane], lane), lane);
        part[32 * warp + lane] = top;
        __syncthreads();
    }
    if (warp == nwarps - 1) {  // never merges: nwarps >= 4, the tree's warps are below nwarps / 2
        int tot = 0;  // clustered tokens: the sum of all sizes
        for (int c = lane; c < C; c += 32) tot += szc[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
        if (lane == 0) s_total = tot;
    }
    for (int n = nwarps; n > 1; n >>= 1) {
        if (warp < n / 2) {
            const uint64_t a = part[32 * warp + lane], b = part[32 * (warp + n / 2) + lane];
            part[32 * warp + lane] = warp_merge32(a, b, lane);
        }
        __syncthreads();
    }
    if (warp == 0) {
        const int tot = s_total;
        const uint64_t top = part[lane];
        const int target = tot < B ? tot : B;
        const int c = (int)(uint32_t)top;
        const int sz = (top != ~0ull && c < C) ? szc[c] : 0;
        int incl = sz;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += t;
        }
        // ranks needed: the first rank whose inclusive prefix reaches the target
        const unsigned reach = __ballot_sync(FULL, incl >= target);
        const bool fast = target == 0 || reach != 0u;
        const int nsel = target == 0 ? 0 : (reach ? __ffs(reach) : 0);
        __syncwarp();  // every lane has read part before start / cl (same storage) are written
        if (fast && lane < nsel) {
            start[lane] = incl - sz;
            cl[lane] = c;
        }
        if (lane == 0) {
            s_fast = fast;
            s_nsel = nsel;
        }
    }
    __syncthreads();
    int nsorted;
    const int total = s_total;
    if (s_fast) {
        nsorted = s_nsel;
    } else {
    // ---- 3'. exact candidate pre-filter: a size-weighted histogram over the
    // top 12 bits of the keys (ascending key = descending score) gives the
    // first bin at which the cumulative size reaches min(B, total).  Clusters
    // in earlier bins rank before every cluster of that bin, clusters in later
    // bins after all of them, and the candidates (bins up to and including
    // that one) already hold at least the budget: only they need ranking.
    constexpr int HBITS = 12, NBIN = 1 << HBITS;
    int32_t* hist = offc + N;                                 // [NBIN]
    uint64_t* cand = reinterpret_cast<uint64_t*>(start);      // [<= NT] (start/cl reused)
    __shared__ int32_t s_bstar, s_M;
    for (int i = tid; i < NBIN; i += NT) hist[i] = 0;
    if (tid == 0) s_M = 0;
    __syncthreads();
    for (int i = tid; i < N; i += NT) {
        const uint64_t k = sk[i];
        if (k != ~0ull) atomicAdd(&hist[(int)(k >> (64 - HBITS))], szc[(int)(uint32_t)k]);
    }
    __syncthreads();
    {
        // block-wide: thread t owns bins [t*PER, t*PER + PER) (NT * PER == NBIN)
        const int PER = NBIN / NT;
        int ls = 0;
        for (int i = 0; i < PER; ++i) ls += hist[tid * PER + i];
        int incl = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int wt = lane < nwarps ? wsum[lane] : 0;
            int wi = wt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULL, wi, o);
                if (lane >= o) wi += t;
            }
            if (lane < nwarps) wsum[lane] = wi - wt;
            if (lane == 31) s_total = wi;
            if (lane == 0) s_bstar = -1;
        }
        __syncthreads();
        const int tot = s_total;
        const int target = tot < B ? tot : B;
        const int excl = wsum[warp] + incl - ls;  // bins before this thread's
        if (target > 0 && excl < target && excl + ls >= target) {
            int run = excl;
            for (int i = 0; i < PER; ++i) {
                run += hist[tid * PER + i];
                if (run >= target) {
                    s_bstar = tid * PER + i;  // exactly one thread crosses the target
                    break;
                }
            }
        }
    }
    __syncthreads();
    const int bstar = s_bstar;
    // every cluster needs ranking when the budget covers all tokens
    const bool take_all = total <= B;
    if (!take_all) {
        for (int i0 = 0; i0 < N; i0 += NT) {  // i0 is warp-uniform: the ballot sees all lanes
            const uint64_t k = sk[i0 + tid];
            const bool is_c = k != ~0ull && (int)(k >> (64 - HBITS)) <= bstar;
            const unsigned bal = __ballot_sync(FULL, is_c);
            int wbase = 0;
            if (lane == 0 && bal) wbase = atomicAdd(&s_M, __popc(bal));
            wbase = __shfl_sync(FULL, wbase, 0);
            if (is_c) {
                const int pos = wbase + __popc(bal & ((1u << lane) - 1u));
                if (pos < NT) cand[pos] = k;
            }
        }
    }
    __syncthreads();
    const int M = s_M;
    const bool small = !take_all && M <= NT;
    if (small && M <= 32) {
        // ---- 3a. up to 32 candidates: one warp, shuffles only
        if (warp == 0) {
            uint64_t ck = (lane < M) ? cand[lane] : ~0ull;
            for (int k = 2; k <= 32; k <<= 1)
                for (int j = k >> 1; j > 0; j >>= 1) {
                    const uint64_t p = __shfl_xor_sync(FULL, ck, j);
                    const bool keep_min = ((lane & j) == 0) == ((lane & k) == 0);
                    ck = keep_min ? (ck < p ? ck : p) : (ck < p ? p : ck);
                }
            if (lane < M) sk[lane] = ck;
        }
        nsorted = M;
    } else if (small) {
        // ---- 3b. sort the M candidates: one key per thread below N2
        int N2 = 32;
        while (N2 < M) N2 <<= 1;
        uint64_t ck = (tid < M) ? cand[tid] : ~0ull;
        for (int k = 2; k <= N2; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                if (j >= 32) {
                    __syncthreads();
                    if (tid < N2) cand[tid] = ck;
                    __syncthreads();
                    if (tid < N2) {
                        const uint64_t p = cand[tid ^ j];
                        const bool keep_min = ((tid & j) == 0) == ((tid & k) == 0);
                        ck = keep_min ? (ck < p ? ck : p) : (ck < p ? p : ck);
                    }
                } else {
                    const uint64_t p = __shfl_xor_sync(FULL, ck, j);
                    const bool keep_min = ((tid & j) == 0) == ((tid & k) == 0);
                    ck = keep_min ? (ck < p ? ck : p) : (ck < p ? p : ck);
                }
            }
        }
        __syncthreads();
        if (tid < M) sk[tid] = ck;
        nsorted = M;
    } else {
        // ---- 3c. full bitonic sort, ascending keys; position i = e * NT + tid
        uint64_t kv[E];
#pragma unroll
        for (int e = 0; e < E; ++e) kv[e] = sk[e * NT + tid];
        for (int k = 2; k <= N; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                if (j >= NT) {
                    const int ej = j / NT;
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        if (e & ej) continue;
                        const int pe = e | ej;
                        const int i = e * NT + tid;
                        const bool up = (i & k) == 0;
                        const uint64_t x = kv[e], y = kv[pe];
                        if ((x > y) == up) {
                            kv[e] = y;
                            kv[pe] = x;
                        }
                    }
                } else if (j >= 32) {
                    __syncthreads();
#pragma unroll
                    for (int e = 0; e < E; ++e) sk[e * NT + tid] = kv[e];
                    __syncthreads();
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int i = e * NT + tid;
                        const uint64_t p = sk[i ^ j];
                        const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
                        kv[e] = keep_min ? (kv[e] < p ? kv[e] : p) : (kv[e] < p ? p : kv[e]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int i = e * NT + tid;
                        const uint64_t p = __shfl_xor_sync(FULL, kv[e], j);
                        const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
                        kv[e] = keep_min ? (kv[e] < p ? kv[e] : p) : (kv[e] < p ? p : kv[e]);
                    }
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) sk[e * NT + tid] = kv[e];
        nsorted = C;
    }
    __syncthreads();

    // ---- 4. sizes in rank order, exclusive prefix sum over the ranked keys
    int base = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int i = e * NT + tid;
        const int c = i < nsorted ? (int)(uint32_t)sk[i] : 0;
        const int sz = i < nsorted ? szc[c] : 0;
        int incl = sz;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int wt = lane < nwarps ? wsum[lane] : 0;
            int wi = wt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULL, wi, o);
                if (lane >= o) wi += t;
            }
            if (lane < nwarps) wsum[lane] = wi - wt;
            if (lane == 31) s_tot = wi;  // the segment's total
        }
        __syncthreads();
        const int seg_total = s_tot;
        const int excl = base + wsum[warp] + incl - sz;
        __syncthreads();
        start[i] = excl;
        cl[i] = c;
        base += seg_total;
        __syncthreads();
    }

    }  // histogram path

    // ---- 5. cut at the budget and compact the token ids: FILL slots per
    // thread at a time, their positions first, then all their permutation
    // loads in flight together
    const int cnt = total < B ? total : B;
    if (tid == 0) count[u] = cnt;
    const int32_t* pu = perm + (size_t)u * ntok;
    int32_t* out = idx + (size_t)u * B;
    constexpr int FILL = 4;
    for (int p0 = 0; p0 < cnt; p0 += FILL * NT) {
        int pos[FILL];
#pragma unroll
        for (int f = 0; f < FILL; ++f) {
            const int p = p0 + f * NT + tid;
            pos[f] = -1;
            if (p < cnt) {
                // largest rank r with start[r] <= p (that cluster is non-empty and holds p)
                int lo = 0, hi = nsorted - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (start[mid] <= p) lo = mid;
                    else hi = mid - 1;
                }
                pos[f] = offc[cl[lo]] + (p - start[lo]);
            }
        }
        int32_t tok[FILL];
#pragma unroll
        for (int f = 0; f < FILL; ++f) tok[f] = (unsigned)pos[f] < (unsigned)ntok ? pu[pos[f]] : 0;
#pragma unroll
        for (int f = 0; f < FILL; ++f) {
            const int p = p0 + f * NT + tid;
            if (p < cnt) {
                if ((unsigned)pos[f] >= (unsigned)ntok) set_err(dev_err, CKV_DEV_BAD_CSR);
                out[p] = tok[f];
            }
        }
    }
}

// ============================================================================
// sparse decode attention
// ============================================================================
// Transposed reduction across the LPR lanes that share a row: N partial sums
// per lane become N / LPR complete sums per lane (lane li keeps values
// [li*VPL, li*VPL+VPL)); if N < LPR the sums end up replicated.
template <int N, int LPR>
__device__ __forceinline__ void xreduce(float (&a)[N], int li) {
    int n = N;
#pragma unroll
    for (int o = LPR / 2; o >= 1; o >>= 1) {
        if (n >= 2) {
            const bool up = (li & o) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                if (i < n / 2) {
                    const float send = up ? a[i] : a[i + n / 2];
                    const float keep = up ? a[i + n / 2] : a[i];
                    a[i] = keep + __shfl_xor_sync(FULL, send, o);
                }
            }
            n >>= 1;
        } else {
            a[0] += __shfl_xor_sync(FULL, a[0], o);
        }
    }
}

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

constexpr int ATT_CW = 8;                    // consumer warps per CTA
constexpr int ATT_STAGES = 3;                // shared-memory ring depth
constexpr int ATT_THREADS = 32 * (ATT_CW + 1);

template <typename T, int G>
struct AttnShape {
    static constexpr int CPL = Vec<T>::N;
    static constexpr int LPR = D / CPL;
    static constexpr int RPI = 32 / LPR;
    // rows per lane group per block (fewer for 8 heads to bound registers); when
    // G*NB < LPR the reduced logits end up replicated across lanes
    static constexpr int NB = G >= 8 ? 4 : 8;
    static constexpr int NV = G * NB;              // partial dots per lane
    static constexpr int VPL = NV >= LPR ? NV / LPR : 1;
    static constexpr int LOGL = ilog2(LPR);
    static constexpr int H = ilog2(NV) < LOGL ? ilog2(NV) : LOGL;  // halving steps
    static constexpr int REPL = LOGL - H;          // replication bits
    static constexpr int GL = NB / VPL;            // value holders per head
    static constexpr int RB = NB * RPI;            // rows per consumer warp per stage
    static constexpr int SR = ATT_CW * RB;         // rows per stage (one work item)
    static constexpr int PW = G * (D + 2);         // floats of one softmax partial
    static constexpr size_t SMEM = (size_t)ATT_STAGES * SR * D * sizeof(T) * 2   // K, V ring
                                   + (size_t)ATT_CW * PW * sizeof(float)          // warp states
                                   + (size_t)ATT_CW * RPI * NB * G * sizeof(float) // p exchange
                                   + (size_t)ATT_STAGES * SR * sizeof(int32_t)    // token ids
                                   + (size_t)ATT_STAGES * G * D * sizeof(T);      // q
};

struct AttnArgs {
    const void* q;
    const void* K;
    const void* V;
    const int32_t* idx;
    const int32_t* count;
    int max_len, sinks, clustered_end, cur_len, B;
    int ipu;    // work items (stages of SR rows) per unit
    int ipc;    // work items per CTA
    int total;  // units * ipu
    int max_slots;
    float qscale;
    float* out;
    float* part;
    int32_t* dev_err;
    long long wait_limit;  // SM cycles before a wait gives up
    int stall;             // failure detection test: consumer warp 0 first waits on a barrier nothing completes
};

// Persistent, warp-specialised sparse decode attention.  Work items are
// (unit, SR consecutive rows of the unit's attended set: sinks, then pending
// tokens, then the selected tokens); each CTA takes a contiguous range.
//   warp 0 (producer): resolves the token ids of an item, then streams its K
//     and V rows with 16-byte cp.async copies into one stage of a shared-memory
//     ring, signalling an mbarrier; q of the unit rides along.
//   warps 1..8 (consumers): RB rows each per item; logits of the g heads are
//     reduced across the lanes of a row with a transposed shuffle reduction,
//     an online softmax keeps (max, sum, acc) per head across all items of the
//     same unit; at a unit boundary the warp states are merged (in a fixed
//     order) into one partial per (unit, CTA).
// attn_combine_kernel then merges the partials of each unit, in CTA order.
template <typename T, int G>
__global__ void __launch_bounds__(ATT_THREADS, 1) attn_kernel(const AttnArgs a) {
    using S = AttnShape<T, G>;
    constexpr int CPL = S::CPL, LPR = S::LPR, RPI = S::RPI, NB = S::NB, NV = S::NV, VPL = S::VPL,
                  RB = S::RB, SR = S::SR, PW = S::PW;
    extern __shared__ __align__(128) unsigned char attn_smem[];
    T* sK = reinterpret_cast<T*>(attn_smem);                       // [STAGES][SR][D]
    T* sV = sK + (size_t)ATT_STAGES * SR * D;                      // [STAGES][SR][D]
    float* red = reinterpret_cast<float*>(sV + (size_t)ATT_STAGES * SR * D);  // [CW][PW]
    float* psm = red + ATT_CW * PW;                                // [CW][RPI][NB][G]
    int32_t* stok = reinterpret_cast<int32_t*>(psm + ATT_CW * RPI * NB * G);  // [STAGES][SR]
    T* sq = reinterpret_cast<T*>(stok + ATT_STAGES * SR);          // [STAGES][G][D]
    __shared__ int s_unit[ATT_STAGES], s_nrows[ATT_STAGES];
    __shared__ __align__(8) uint64_t full[ATT_STAGES], empty[ATT_STAGES], red_full, red_free, never;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int first = blockIdx.x * a.ipc;
    const int nitems = min(a.total, first + a.ipc) - first;
    const int pend = a.cur_len - a.clustered_end;

    if (tid == 0) {
        for (int st = 0; st < ATT_STAGES; ++st) {
            ptx::mbar_init(&full[st], 64);        // 32 header arrivals + 32 copy arrivals
            ptx::mbar_init(&empty[st], ATT_CW);
        }
        ptx::mbar_init(&red_full, ATT_CW);
        ptx::mbar_init(&red_free, ATT_CW);
        ptx::mbar_init(&never, 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();

    auto give_up = [&]() {
        if (atomicExch(&abort_flag, 1) == 0) set_err(a.dev_err, CKV_DEV_TIMEOUT);
    };

    if (warp == 0) {
        // ================================================================ producer
        constexpr int LPC = D * (int)sizeof(T) / 16;  // lanes per row copy
        constexpr int RPC = 32 / LPC;                 // rows per warp-wide copy
        constexpr int EPC = 16 / (int)sizeof(T);      // elements per 16-byte chunk
        const T* Kb = static_cast<const T*>(a.K);
        const T* Vb = static_cast<const T*>(a.V);
        const T* qb = static_cast<const T*>(a.q);
        const int csub = lane / LPC, ch = lane % LPC;
        int cur_u = -1, R = 0;
        for (int it = 0; it < nitems; ++it) {
            const int st = it % ATT_STAGES;
            if (it >= ATT_STAGES &&
                !__all_sync(FULL, ptx::mbar_wait(&empty[st], ((it / ATT_STAGES) - 1) & 1, a.wait_limit, &abort_flag))) {
                give_up();
                break;
            }
            const int item = first + it;
            const int u = item / a.ipu, k = item % a.ipu;
            if (u != cur_u) {
                int cnt = a.count[u];
                if (cnt < 0 || cnt > a.B) {
                    if (lane == 0) set_err(a.dev_err, CKV_DEV_BAD_COUNT);
                    cnt = cnt < 0 ? 0 : a.B;
                }
                R = a.sinks + pend + cnt;
                cur_u = u;
            }
            const int row0 = k * SR;
            const int nrows = max(0, min(SR, R - row0));
            int32_t* tk = stok + st * SR;
#pragma unroll
            for (int qq = 0; qq < SR / 32; ++qq) {
                const int rl = lane + 32 * qq;
                int tok = -1;
                if (rl < nrows) {
                    const int r = row0 + rl;
                    if (r < a.sinks) tok = r;
                    else if (r < a.sinks + pend) tok = a.clustered_end + (r - a.sinks);
                    else tok = a.idx[(size_t)u * a.B + (r - a.sinks - pend)];
                    if (tok < 0 || tok >= a.cur_len) {
                        set_err(a.dev_err, CKV_DEV_BAD_INDEX);
                        tok = -1;
                    }
                }
                tk[rl] = tok;
            }
            if (lane == 0) {
                s_unit[st] = u;
                s_nrows[st] = nrows;
            }
            __syncwarp();
            // q of the unit (G rows of D elements)
            for (int e = lane; e < G * D / EPC; e += 32)
                ptx::cp_async16(sq + (size_t)st * G * D + e * EPC, qb + (size_t)u * G * D + e * EPC);
            const size_t ubase = (size_t)u * a.max_len * D + ch * EPC;
            T* dK = sK + (size_t)st * SR * D + ch * EPC;
            T* dV = sV + (size_t)st * SR * D + ch * EPC;
            for (int r = csub; r < nrows; r += RPC) {
                const int tok = tk[r];
                if (tok >= 0) {
                    ptx::cp_async16(dK + (size_t)r * D, Kb + ubase + (size_t)tok * D);
                    ptx::cp_async16(dV + (size_t)r * D, Vb + ubase + (size_t)tok * D);
                }
            }
            ptx::mbar_arrive(&full[st]);           // header and ids written
            ptx::cp_async_mbar_arrive(&full[st]);  // arrives when this lane's copies land
        }
        ptx::cp_async_wait_all();
    } else {
        // ================================================================ consumers
        const int w = warp - 1;
        const int sub = lane / LPR, li = lane % LPR;
        const int b = li >> S::REPL;
        const int hl = (b * VPL) / NB;
        float* pw = psm + (size_t)w * (RPI * NB * G) + sub * (NB * G);
        float qv[G][CPL], acc[G][CPL], m[G];
        float lsum = 0.f;
        int cur_u = -1, flushes = 0;
        bool alive = true;

        auto reset = [&](int st) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint4 wq = *reinterpret_cast<const uint4*>(sq + (size_t)st * G * D + h * D + li * CPL);
                float f[CPL];
                Vec<T>::unpack(wq, f);
                m[h] = -INFINITY;
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    qv[h][c] = f[c] * a.qscale;
                    acc[h][c] = 0.f;
                }
            }
            lsum = 0.f;
        };

        // merge the warp states of unit u into this CTA's partial for u: every
        // consumer warp publishes its state, then combines 1/CW of the outputs
        // over all warps in a fixed order
        auto flush = [&](int u) -> bool {
            float ls = lsum;
#pragma unroll
            for (int o = 1; o < S::GL; o <<= 1) ls += __shfl_xor_sync(FULL, ls, o << S::REPL);
            float lh[G], mm[G], ac[G][CPL];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                lh[h] = __shfl_sync(FULL, ls, (sub * LPR) + ((h * S::GL) << S::REPL));
                mm[h] = m[h];
#pragma unroll
                for (int c = 0; c < CPL; ++c) ac[h][c] = acc[h][c];
            }
            if constexpr (RPI == 2) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float mo = __shfl_xor_sync(FULL, mm[h], 16);
                    const float lo = __shfl_xor_sync(FULL, lh[h], 16);
                    const float M = fmaxf(mm[h], mo);
                    const float fa = (M == -INFINITY) ? 0.f : exp2f(mm[h] - M);
                    const float fb = (M == -INFINITY) ? 0.f : exp2f(mo - M);
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        const float ao = __shfl_xor_sync(FULL, ac[h][c], 16);
                        ac[h][c] = ac[h][c] * fa + ao * fb;
                    }
                    lh[h] = lh[h] * fa + lo * fb;
                    mm[h] = M;
                }
            }
            // the previous merge has finished reading the exchange area
            if (flushes > 0 &&
                !__all_sync(FULL, ptx::mbar_wait(&red_free, (flushes - 1) & 1, a.wait_limit, &abort_flag)))
                return false;
            float* rw = red + (size_t)w * PW;
            if (sub == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
#pragma unroll
                    for (int c = 0; c < CPL; ++c) rw[h * (D + 2) + li * CPL + c] = ac[h][c];
                    if (li == 0) {
                        rw[h * (D + 2) + D] = mm[h];
                        rw[h * (D + 2) + D + 1] = lh[h];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&red_full);
            if (!__all_sync(FULL, ptx::mbar_wait(&red_full, flushes & 1, a.wait_limit, &abort_flag)))
                return false;
            const int c0 = (u * a.ipu) / a.ipc;
            float* pp = a.part + ((size_t)u * a.max_slots + (blockIdx.x - c0)) * PW;
            for (int e = w * 32 + lane; e < G * D; e += ATT_CW * 32) {
                const int h = e / D, c = e % D;
                float M = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < ATT_CW; ++ww) M = fmaxf(M, red[ww * PW + h * (D + 2) + D]);
                float o = 0.f, l = 0.f;
#pragma unroll
                for (int ww = 0; ww < ATT_CW; ++ww) {
                    const float mw = red[ww * PW + h * (D + 2) + D];
                    const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
                    o += red[ww * PW + h * (D + 2) + c] * f;
                    l += red[ww * PW + h * (D + 2) + D + 1] * f;
                }
                pp[h * (D + 2) + c] = o;
                if (c == 0) {
                    pp[h * (D + 2) + D] = M;
                    pp[h * (D + 2) + D + 1] = l;
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&red_free);
            ++flushes;
            return true;
        };

        if (a.stall && w == 0 &&
            !__all_sync(FULL, ptx::mbar_wait(&never, 0, a.wait_limit, &abort_flag))) {
            give_up();
            alive = false;
        }
        for (int it = 0; it < nitems && alive; ++it) {
            const int st = it % ATT_STAGES;
            if (!__all_sync(FULL, ptx::mbar_wait(&full[st], (it / ATT_STAGES) & 1, a.wait_limit, &abort_flag))) {
                give_up();
                alive = false;
                break;
            }
            const int u = s_unit[st], nrows = s_nrows[st];
            if (u != cur_u) {
                if (cur_u >= 0 && !flush(cur_u)) {
                    give_up();
                    alive = false;
                    break;
                }
                cur_u = u;
                reset(st);
            }
            const int wrow0 = w * RB;
            if (wrow0 < nrows) {
                const T* kb = sK + ((size_t)st * SR + wrow0) * D + li * CPL;
                const T* vb = sV + ((size_t)st * SR + wrow0) * D + li * CPL;
                const int32_t* tk = stok + st * SR + wrow0;
                unsigned vbits = 0;
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int r = j * RPI + sub;
                    if (wrow0 + r < nrows && tk[r] >= 0) vbits |= 1u << j;
                }
                float av[NV];
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const uint4 wk = *reinterpret_cast<const uint4*>(kb + (size_t)(j * RPI + sub) * D);
                    float f[CPL];
                    Vec<T>::unpack(wk, f);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float d0 = 0.f;
#pragma unroll
                        for (int c = 0; c < CPL; ++c) d0 = fmaf(qv[h][c], f[c], d0);
                        av[h * NB + j] = d0;
                    }
                }
                xreduce<NV, LPR>(av, li);
                float bm = -INFINITY;
#pragma unroll
                for (int t = 0; t < VPL; ++t) {
                    const int j = (b * VPL + t) % NB;
                    if (!((vbits >> j) & 1u)) av[t] = -INFINITY;
                    bm = fmaxf(bm, av[t]);
                }
#pragma unroll
                for (int o = 1; o < S::GL; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, o << S::REPL));
                float mnew[G], scl[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float hb = __shfl_sync(FULL, bm, (sub * LPR) + ((h * S::GL) << S::REPL));
                    mnew[h] = fmaxf(m[h], hb);
                    scl[h] = (mnew[h] == -INFINITY) ? 1.f : exp2f(m[h] - mnew[h]);
                }
                float mh = mnew[0], sh = scl[0];
#pragma unroll
                for (int h = 1; h < G; ++h)
                    if (h == hl) {
                        mh = mnew[h];
                        sh = scl[h];
                    }
                float psum = 0.f;
#pragma unroll
                for (int t = 0; t < VPL; ++t) {
                    const int v = b * VPL + t;
                    const float p = (av[t] == -INFINITY) ? 0.f : exp2f(av[t] - mh);
                    psum += p;
                    pw[(v % NB) * G + (v / NB)] = p;
                }
                lsum = lsum * sh + psum;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    m[h] = mnew[h];
#pragma unroll
                    for (int c = 0; c < CPL; ++c) acc[h][c] *= scl[h];
                }
                __syncwarp();
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    if (!((vbits >> j) & 1u)) continue;
                    const uint4 wv = *reinterpret_cast<const uint4*>(vb + (size_t)(j * RPI + sub) * D);
                    float f[CPL];
                    Vec<T>::unpack(wv, f);
                    float p[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) p[h] = pw[j * G + h];
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int c = 0; c < CPL; ++c) acc[h][c] = fmaf(p[h], f[c], acc[h][c]);
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty[st]);
        }
        if (alive && cur_u >= 0 && !flush(cur_u)) give_up();
    }
}

// One CTA per unit: merge the per-CTA softmax partials of the unit (slot
// order) into o_h = acc / l.  The slots a unit has are fixed by the static
// work split: CTAs (u*ipu)/ipc .. (u*ipu + ipu - 1)/ipc.
template <int G>
__global__ void __launch_bounds__(128) attn_combine_kernel(const float* __restrict__ part, int ipu, int ipc,
                                                           int max_slots, float* __restrict__ out) {
    constexpr int PW = G * (D + 2);
    __shared__ float fs[16][G];
    __shared__ float ls[G];
    const int u = blockIdx.x, tid = threadIdx.x;
    const int c0 = (u * ipu) / ipc, c1 = (u * ipu + ipu - 1) / ipc;
    const int ncov = min(c1 - c0 + 1, 16);
    const float* pu = part + (size_t)u * max_slots * PW;
    if (tid < G) {
        const int h = tid;
        float M = -INFINITY;
        for (int t = 0; t < ncov; ++t) M = fmaxf(M, pu[(size_t)t * PW + h * (D + 2) + D]);
        float l = 0.f;
        for (int t = 0; t < ncov; ++t) {
            const float mt = pu[(size_t)t * PW + h * (D + 2) + D];
            const float f = (mt == -INFINITY) ? 0.f : exp2f(mt - M);
            fs[t][h] = f;
            l += pu[(size_t)t * PW + h * (D + 2) + D + 1] * f;
        }
        ls[h] = l;
    }
    __syncthreads();
    for (int e = tid; e < G * D; e += 128) {
        const int h = e / D, c = e % D;
        float o = 0.f;
        for (int t = 0; t < ncov; ++t) o += pu[(size_t)t * PW + h * (D + 2) + c] * fs[t][h];
        out[((size_t)u * G + h) * D + c] = ls[h] > 0.f ? o / ls[h] : 0.f;
    }
}

template <typename T, int G>
cudaError_t launch_attn_t(const void* q, const void* K, const void* V, const int32_t* idx,
                          const int32_t* count, int units, int max_len, int sinks,
                          int clustered_end, int cur_len, int B, float* out, float* part,
                          int max_splits, int32_t* dev_err, int num_sms, long long wait_limit, int stall,
                          cudaStream_t st) {
    using S = AttnShape<T, G>;
    AttnArgs a;
    a.q = q;
    a.K = K;
    a.V = V;
    a.idx = idx;
    a.count = count;
    a.max_len = max_len;
    a.sinks = sinks;
    a.clustered_end = clustered_end;
    a.cur_len = cur_len;
    a.B = B;
    a.ipu = (sinks + (cur_len - clustered_end) + B + S::SR - 1) / S::SR;
    if (a.ipu < 1) a.ipu = 1;
    if (a.ipu > max_splits) return cudaErrorInvalidValue;
    a.total = a.ipu * units;
    int grid = num_sms > 0 ? num_sms : 152;
    if (grid > a.total) grid = a.total;
    a.ipc = (a.total + grid - 1) / grid;
    // a unit spans at most 16 CTAs (the combine kernel's limit)
    if (a.ipc * 15 < a.ipu) a.ipc = (a.ipu + 14) / 15;
    grid = (a.total + a.ipc - 1) / a.ipc;
    a.max_slots = max_splits;
    a.qscale = 1.4426950408889634f / sqrtf((float)D);
    a.out = out;
    a.part = part;
    a.dev_err = dev_err;
    a.wait_limit = wait_limit;
    a.stall = stall;
    auto kern = attn_kernel<T, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, ATT_THREADS, S::SMEM, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    attn_combine_kernel<G><<<units, 128, 0, st>>>(part, a.ipu, a.ipc, max_splits, out);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_score_t(const void* q, const void* mu, int g, int units, int cmax, int C,
                           float* scores, int stride, const int32_t* pf_sizes, const int32_t* pf_offsets,
                           const cudaAccessPolicyWindow* win, cudaStream_t s) {
    constexpr int RPW = (32 / (D / Vec<T>::N)) * SCORE_UNROLL;  // rows per warp
    dim3 grid((C + 8 * RPW - 1) / (8 * RPW), units);
#define CKV_SCORE(G)                                                                                          \
    return launch_dependent_win(score_kernel<T, G>, grid, dim3(256), 0, s, win, (const T*)q, (const T*)mu, cmax, \
                                C, scores, stride, pf_sizes, pf_offsets)
    switch (g) {
        case 1: CKV_SCORE(1);
        case 2: CKV_SCORE(2);
        case 4: CKV_SCORE(4);
        case 8: CKV_SCORE(8);
    }
#undef CKV_SCORE
    return cudaErrorInvalidValue;
}

template <int E, typename T, int G>
cudaError_t launch_sel_t(const ckv_ctx* ctx, const float* scores, int stride, const void* q, int C, int N, int B,
                         int32_t* idx, int32_t* count, cudaStream_t s) {
    // keys, starts, ranks, sizes, offsets; then the histogram (or the scores
    // computed here followed by q: at most 4 KB, N <= 1024 leaves >= 12 KB)
    const size_t smem = (size_t)N * 24 + (size_t)(N > 4096 ? N : 4096) * 4;
    auto kern = sel_kernel<E, T, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // the centroid copy is what this launch re-reads each step when it scores
    const cudaAccessPolicyWindow* win = !ctx->l2_on ? nullptr : (G > 0 ? &ctx->l2_mu : &ctx->l2_perm);
    return launch_dependent_win(kern, dim3(ctx->cfg.units), dim3(N / E), smem, s, win, scores, stride,
                                static_cast<const T*>(q), static_cast<const T*>(ctx->mu_s), ctx->cmax, C, N,
                                (const int32_t*)ctx->sizes, (const int32_t*)ctx->offsets,
                                (const int32_t*)ctx->perm, ctx->ntok, B, idx, count, ctx->dev_err);
}

template <int E>
cudaError_t launch_sel_e(const ckv_ctx* ctx, const float* scores, int stride, const void* q, int C, int N, int B,
                         int32_t* idx, int32_t* count, cudaStream_t s) {
    if (scores) return launch_sel_t<E, float, 0>(ctx, scores, stride, nullptr, C, N, B, idx, count, s);
    if constexpr (E == 1) {  // scoring inside the selection: one key per thread only
#define CKV_SEL(T, G) return launch_sel_t<E, T, G>(ctx, nullptr, 0, q, C, N, B, idx, count, s)
        if (ctx->cfg.kv_dtype == CKV_BF16) {
            switch (ctx->cfg.g) {
                case 1: CKV_SEL(__nv_bfloat16, 1);
                case 2: CKV_SEL(__nv_bfloat16, 2);
                case 4: CKV_SEL(__nv_bfloat16, 4);
                case 8: CKV_SEL(__nv_bfloat16, 8);
            }
        } else {
            switch (ctx->cfg.g) {
                case 1: CKV_SEL(float, 1);
                case 2: CKV_SEL(float, 2);
                case 4: CKV_SEL(float, 4);
                case 8: CKV_SEL(float, 8);
            }
        }
#undef CKV_SEL
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_score(const ckv_ctx* ctx, const void* q, int C, float* scores, int stride,
                         cudaStream_t s, bool prefetch_csr) {
    if (C <= 0) return cudaSuccess;
    const int32_t* ps = prefetch_csr ? ctx->sizes : nullptr;
    const int32_t* po = prefetch_csr ? ctx->offsets : nullptr;
    const cudaAccessPolicyWindow* win = ctx->l2_on ? &ctx->l2_mu : nullptr;
    if (ctx->cfg.kv_dtype == CKV_BF16)
        return launch_score_t<__nv_bfloat16>(q, ctx->mu_s, ctx->cfg.g, ctx->cfg.units, ctx->cmax, C,
                                             scores, stride, ps, po, win, s);
    return launch_score_t<float>(q, ctx->mu_s, ctx->cfg.g, ctx->cfg.units, ctx->cmax, C, scores,
                                 stride, ps, po, win, s);
}

cudaError_t launch_select(const ckv_ctx* ctx, const void* q, const float* scores, int stride, int C, int B,
                          int32_t* idx, int32_t* count, cudaStream_t s) {
    int N = 128;
    while (N < C) N <<= 1;
    if (!scores && N > 1024) {
        // many clusters: scores of every cluster into the context's scratch
        // (a many-CTA stream over the centroid table), then the selection
        // reads them; up to 1024 clusters each selection CTA scores its unit
        cudaError_t e = launch_score(ctx, q, C, ctx->scores, ctx->cmax, s, true);
        if (e != cudaSuccess) return e;
        scores = ctx->scores;
        stride = ctx->cmax;
    }
    if (N <= 1024) return launch_sel_e<1>(ctx, scores, stride, q, C, N, B, idx, count, s);
    if (N == 2048) return launch_sel_e<2>(ctx, scores, stride, q, C, N, B, idx, count, s);
    if (N == 4096) return launch_sel_e<4>(ctx, scores, stride, q, C, N, B, idx, count, s);
    if (N == 8192) return launch_sel_e<8>(ctx, scores, stride, q, C, N, B, idx, count, s);
    return cudaErrorInvalidValue;
}

int attention_rows_per_split(int kv_dtype, int g) {
    if (kv_dtype == CKV_BF16) {
        return attention_mma_rows_per_tile();
    } else {
        switch (g) {
            case 1: return AttnShape<float, 1>::SR;
            case 2: return AttnShape<float, 2>::SR;
            case 4: return AttnShape<float, 4>::SR;
            case 8: return AttnShape<float, 8>::SR;
        }
    }
    return 0;
}

cudaError_t launch_attention(const void* q, const void* K, const void* V, const int32_t* idx,
                             const int32_t* count, int units, int g, int kv_dtype, int max_len,
                             int sinks, int clustered_end, int cur_len, int B, float* out,
                             float* part, int max_splits, int32_t* dev_err,
                             int num_sms, long long wait_limit, int stall, cudaStream_t s) {
#define CKV_ATTN(T, G)                                                                          \
    return launch_attn_t<T, G>(q, K, V, idx, count, units, max_len, sinks, clustered_end,      \
                               cur_len, B, out, part, max_splits, dev_err, num_sms, wait_limit, stall, s)
    if (kv_dtype == CKV_BF16) {
        // bf16 K/V: tensor-core kernel (attn_mma.cu); fp32 K/V: CUDA-core kernel below
        return launch_attention_mma(q, K, V, idx, count, units, g, max_len, sinks, clustered_end, cur_len, B,
                                    out, part, max_splits, dev_err, num_sms, s);
    } else {
        switch (g) {
            case 1: CKV_ATTN(float, 1);
            case 2: CKV_ATTN(float, 2);
            case 4: CKV_ATTN(float, 4);
            case 8: CKV_ATTN(float, 8);
        }
    }
#undef CKV_ATTN
    return cudaErrorInvalidValue;
}

}  // namespace ckv
