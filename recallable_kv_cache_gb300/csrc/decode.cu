// Decode-step kernels of the ClusterKV path:
//   score_kernel   cluster scores q . mu (section "Selection at semantic-cluster
//                  granularity"), HBM-bound stream over the centroid table;
//   select_kernel  rank clusters, prefix-sum their sizes, trim the last one and
//                  compact the token ids (section "Selection and indexing
//                  mechanism", Fig. 8), one CTA per unit;
//   attn_kernel    gather of the selected K/V rows with bulk-async copies into
//                  shared memory and split-K flash-decode attention (section
//                  "Background": softmax(q K_S^T / sqrt(d)) V_S), with the
//                  cross-split combine done by the last CTA of each unit.
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
template <typename T, int G>
__global__ void __launch_bounds__(256) score_kernel(const T* __restrict__ q,
                                                   const T* __restrict__ mu, int cmax, int C,
                                                   float* __restrict__ scores, int stride) {
    constexpr int CPL = Vec<T>::N;   // channels per lane
    constexpr int LPR = D / CPL;     // lanes per centroid row
    constexpr int RPI = 32 / LPR;    // rows per warp-wide load
    constexpr int UNROLL = 4;
    const int u = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPR, li = lane % LPR;

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
__device__ __forceinline__ uint64_t rank_key(float s, int c) {
    if (s == 0.f) s = 0.f;  // -0 ranks like +0
    const uint32_t b = __float_as_uint(s);
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);  // ascending with s
    return ((uint64_t)(~ord) << 32) | (uint32_t)c;                      // descending score, asc c
}

constexpr int SEL_THREADS = 512;

__global__ void __launch_bounds__(SEL_THREADS) select_kernel(
    const float* __restrict__ scores, int stride, int C, int npow2, const int32_t* __restrict__ sizes,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm, int cmax, int ntok, int B,
    int32_t* __restrict__ idx, int32_t* __restrict__ count, int32_t* __restrict__ dev_err) {
    extern __shared__ __align__(16) unsigned char sel_smem[];
    uint64_t* keys = reinterpret_cast<uint64_t*>(sel_smem);
    int32_t* start = reinterpret_cast<int32_t*>(keys + npow2);
    int32_t* rc = start + npow2;
    __shared__ int32_t warp_tot[SEL_THREADS / 32];
    __shared__ int32_t s_total;

    const int u = blockIdx.x;
    const int tid = threadIdx.x;
    const float* sc = scores + (size_t)u * stride;
    for (int i = tid; i < npow2; i += SEL_THREADS) keys[i] = i < C ? rank_key(sc[i], i) : ~0ull;
    __syncthreads();

    // bitonic sort, ascending keys
    for (int k = 2; k <= npow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < (npow2 >> 1); i += SEL_THREADS) {
                const int lo = ((i & ~(j - 1)) << 1) | (i & (j - 1));
                const int hi = lo + j;
                const uint64_t a = keys[lo], b = keys[hi];
                const bool up = (lo & k) == 0;
                if ((a > b) == up) {
                    keys[lo] = b;
                    keys[hi] = a;
                }
            }
            __syncthreads();
        }
    }

    // sizes in rank order, exclusive prefix sum (each thread a contiguous run)
    const int per = (npow2 + SEL_THREADS - 1) / SEL_THREADS;
    const int r0 = tid * per;
    int run = 0;
    for (int r = r0; r < r0 + per && r < npow2; ++r) {
        const int c = (int)(uint32_t)keys[r];
        const int sz = r < C ? sizes[(size_t)u * cmax + c] : 0;
        rc[r] = c;
        start[r] = sz;  // temporarily the size
        run += sz;
    }
    // block exclusive scan of the per-thread runs
    const int lane = tid & 31, warp = tid >> 5;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wt = lane < SEL_THREADS / 32 ? warp_tot[lane] : 0;
        int wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, wi, o);
            if (lane >= o) wi += t;
        }
        if (lane < SEL_THREADS / 32) warp_tot[lane] = wi - wt;  // exclusive
        if (lane == 31) s_total = wi;
    }
    __syncthreads();
    int base = warp_tot[warp] + incl - run;
    for (int r = r0; r < r0 + per && r < npow2; ++r) {
        const int sz = start[r];
        start[r] = base;
        base += sz;
    }
    __syncthreads();

    const int total = s_total;
    const int cnt = total < B ? total : B;
    if (tid == 0) count[u] = cnt;
    const int32_t* off = offsets + (size_t)u * (cmax + 1);
    const int32_t* pu = perm + (size_t)u * ntok;
    int32_t* out = idx + (size_t)u * B;
    for (int p = tid; p < cnt; p += SEL_THREADS) {
        // largest rank r < C with start[r] <= p (that cluster is non-empty and holds p)
        int lo = 0, hi = C - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (start[mid] <= p) lo = mid;
            else hi = mid - 1;
        }
        const int pos = off[rc[lo]] + (p - start[lo]);
        if ((unsigned)pos < (unsigned)ntok) {
            out[p] = pu[pos];
        } else {
            set_err(dev_err, CKV_DEV_BAD_CSR);
            out[p] = 0;
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

template <typename T, int G>
struct AttnShape {
    static constexpr int CPL = Vec<T>::N;
    static constexpr int LPR = D / CPL;
    static constexpr int RPI = 32 / LPR;
    // rows per lane group per block: enough values to fill the lanes (G*NB >= LPR)
    static constexpr int NB = (LPR / G) > 8 ? (LPR / G) : 8;
    static constexpr int NV = G * NB;              // partial dots per lane
    static constexpr int VPL = NV >= LPR ? NV / LPR : 1;
    static constexpr int LOGL = ilog2(LPR);
    static constexpr int H = ilog2(NV) < LOGL ? ilog2(NV) : LOGL;  // halving steps
    static constexpr int REPL = LOGL - H;          // replication bits
    static constexpr int GL = NB / VPL;            // value holders per head
    static constexpr int RW = NB * RPI;            // rows per warp
    static constexpr int RS = 4 * RW;              // rows per CTA (4 warps)
};

template <typename T, int G>
__global__ void __launch_bounds__(128) attn_kernel(
    const T* __restrict__ q, const T* __restrict__ K, const T* __restrict__ V,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ count, int max_len, int sinks,
    int clustered_end, int cur_len, int B, float qscale, float* __restrict__ out,
    float* __restrict__ part, int32_t* __restrict__ counters, int32_t* __restrict__ dev_err) {
    using S = AttnShape<T, G>;
    constexpr int CPL = S::CPL, LPR = S::LPR, RPI = S::RPI, NB = S::NB, NV = S::NV,
                  VPL = S::VPL, RW = S::RW, RS = S::RS;
    constexpr int ROWB = D * (int)sizeof(T);
    constexpr int PW = G * (D + 2);  // floats per partial

    extern __shared__ __align__(128) unsigned char attn_smem[];
    T* Ks = reinterpret_cast<T*>(attn_smem);
    T* Vs = Ks + RS * D;
    float* red = reinterpret_cast<float*>(Vs + RS * D);  // [4 warps][PW]
    float* ps = red + 4 * PW;                            // [4 warps][RPI][NB][G]
    __shared__ __align__(8) uint64_t bars[4];
    __shared__ int32_t toks[RS];
    __shared__ int s_last;

    const int u = blockIdx.y, s = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pend = cur_len - clustered_end;
    int cnt = count[u];
    if (cnt < 0 || cnt > B) {
        if (s == 0 && tid == 0) set_err(dev_err, CKV_DEV_BAD_COUNT);
        cnt = cnt < 0 ? 0 : B;
    }
    const int R = sinks + pend + cnt;
    const int nsplit = (R + RS - 1) / RS;
    if (s >= nsplit) return;
    const int r0 = s * RS;
    const int nrows = min(RS, R - r0);

    // ---- gather: lane l of warp w copies row w*RW + l
    uint64_t* bar = &bars[warp];
    int tok = -1;
    const int myrow = warp * RW + lane;
    if (lane < RW && myrow < nrows) {
        const int r = r0 + myrow;
        if (r < sinks) tok = r;
        else if (r < sinks + pend) tok = clustered_end + (r - sinks);
        else tok = idx[(size_t)u * B + (r - sinks - pend)];
        if (tok < 0 || tok >= cur_len) {
            set_err(dev_err, CKV_DEV_BAD_INDEX);
            tok = -1;
        }
        toks[myrow] = tok;
    }
    const unsigned vmask = __ballot_sync(FULL, tok >= 0);
    const int nvalid = __popc(vmask);
    if (lane == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    if (nvalid) {
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar, (uint32_t)nvalid * 2u * ROWB);
        __syncwarp();
        if (tok >= 0) {
            const size_t off = ((size_t)u * max_len + tok) * D;
            ptx::bulk_g2s(Ks + (size_t)myrow * D, K + off, ROWB, bar);
            ptx::bulk_g2s(Vs + (size_t)myrow * D, V + off, ROWB, bar);
        }
    }

    // ---- query (pre-scaled by log2(e)/sqrt(d)) while the copies fly
    const int sub = lane / LPR, li = lane % LPR;
    float qv[G][CPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint4 w = *reinterpret_cast<const uint4*>(q + ((size_t)u * G + h) * D + li * CPL);
        float f[CPL];
        Vec<T>::unpack(w, f);
#pragma unroll
        for (int c = 0; c < CPL; ++c) qv[h][c] = f[c] * qscale;
    }
    float acc[G][CPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[h][c] = 0.f;
    // m and the lane's share of l (of its own head)
    float m[G];
#pragma unroll
    for (int h = 0; h < G; ++h) m[h] = -INFINITY;
    float lsum = 0.f;

    bool ok = true;
    if (nvalid) ok = ptx::mbar_wait(bar, 0, WAIT_LIMIT, nullptr);
    if (!ok) set_err(dev_err, CKV_DEV_TIMEOUT);
    __syncwarp();

    if (ok) {
        // ---- logits for the NB rows of this lane group (rows wrow = j*RPI + sub)
        float a[NV];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int wrow = j * RPI + sub;
            const uint4 w = *reinterpret_cast<const uint4*>(Ks + (size_t)(warp * RW + wrow) * D + li * CPL);
            float f[CPL];
            Vec<T>::unpack(w, f);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float d0 = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) d0 = fmaf(qv[h][c], f[c], d0);
                a[h * NB + j] = d0;
            }
        }
        xreduce<NV, LPR>(a, li);
        // lane holds values v = b*VPL + t, b = li >> REPL; head = v / NB, row j = v % NB
        const int b = li >> S::REPL;
        const int hl = (b * VPL) / NB;
        float bm = -INFINITY;
#pragma unroll
        for (int t = 0; t < VPL; ++t) {
            const int j = (b * VPL + t) % NB;
            const int wrow = warp * RW + j * RPI + sub;
            const bool valid = wrow < nrows && toks[wrow] >= 0;
            if (!valid) a[t] = -INFINITY;
            bm = fmaxf(bm, a[t]);
        }
        // max over the head's value holders (bits REPL .. REPL+log2(GL)-1 of li)
#pragma unroll
        for (int o = 1; o < S::GL; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL, bm, o << S::REPL));
        float mnew[G], scl[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const int src = (sub * LPR) + ((h * S::GL) << S::REPL);
            const float hb = __shfl_sync(FULL, bm, src);
            mnew[h] = fmaxf(m[h], hb);
            scl[h] = (mnew[h] == -INFINITY) ? 1.f : exp2f(m[h] - mnew[h]);
        }
        float* pw = ps + warp * (RPI * NB * G) + sub * (NB * G);
        float psum = 0.f;
#pragma unroll
        for (int t = 0; t < VPL; ++t) {
            const int v = b * VPL + t;
            const float p = (a[t] == -INFINITY) ? 0.f : exp2f(a[t] - mnew[hl]);
            psum += p;
            pw[(v % NB) * G + (v / NB)] = p;
        }
        lsum = lsum * scl[hl] + psum;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = mnew[h];
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[h][c] *= scl[h];
        }
        __syncwarp();
        // ---- P V
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int wrow = j * RPI + sub;
            const uint4 w = *reinterpret_cast<const uint4*>(Vs + (size_t)(warp * RW + wrow) * D + li * CPL);
            float f[CPL];
            Vec<T>::unpack(w, f);
            float p[G];
#pragma unroll
            for (int h = 0; h < G; ++h) p[h] = pw[j * G + h];
            const bool valid = (warp * RW + wrow) < nrows && toks[warp * RW + wrow] >= 0;
            if (valid) {
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int c = 0; c < CPL; ++c) acc[h][c] = fmaf(p[h], f[c], acc[h][c]);
            }
        }
        // l of the lane's head: sum over the distinct value holders
#pragma unroll
        for (int o = 1; o < S::GL; o <<= 1) lsum += __shfl_xor_sync(FULL, lsum, o << S::REPL);
    }

    // ---- combine the RPI row groups of the warp (bf16: two half-warps)
    float lh[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const int src = (sub * LPR) + ((h * S::GL) << S::REPL);
        lh[h] = __shfl_sync(FULL, lsum, src);
    }
    if (RPI == 2) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mo = __shfl_xor_sync(FULL, m[h], 16);
            const float lo = __shfl_xor_sync(FULL, lh[h], 16);
            const float M = fmaxf(m[h], mo);
            const float fa = (M == -INFINITY) ? 0.f : exp2f(m[h] - M);
            const float fb = (M == -INFINITY) ? 0.f : exp2f(mo - M);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const float ao = __shfl_xor_sync(FULL, acc[h][c], 16);
                acc[h][c] = acc[h][c] * fa + ao * fb;
            }
            lh[h] = lh[h] * fa + lo * fb;
            m[h] = M;
        }
    }
    float* rw = red + warp * PW;
    if (sub == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int c = 0; c < CPL; ++c) rw[h * (D + 2) + li * CPL + c] = acc[h][c];
        if (li == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                rw[h * (D + 2) + D] = m[h];
                rw[h * (D + 2) + D + 1] = lh[h];
            }
        }
    }
    __syncthreads();

    // ---- combine the 4 warps and write this split's partial
    float* pp = part + ((size_t)u * gridDim.x + s) * PW;
    for (int e = tid; e < G * D; e += 128) {
        const int h = e / D, c = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, red[w * PW + h * (D + 2) + D]);
        float o = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float mw = red[w * PW + h * (D + 2) + D];
            const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
            o += red[w * PW + h * (D + 2) + c] * f;
            l += red[w * PW + h * (D + 2) + D + 1] * f;
        }
        pp[h * (D + 2) + c] = o;
        if (c == 0) {
            pp[h * (D + 2) + D] = M;
            pp[h * (D + 2) + D + 1] = l;
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(&counters[u], 1);
        s_last = (prev == nsplit - 1);
    }
    __syncthreads();
    if (!s_last) return;

    // ---- last CTA of the unit: combine the splits in split order
    __threadfence();
    const float* pu = part + (size_t)u * gridDim.x * PW;
    for (int e = tid; e < G * D; e += 128) {
        const int h = e / D, c = e % D;
        float M = -INFINITY;
        for (int t = 0; t < nsplit; ++t) M = fmaxf(M, __ldcg(pu + (size_t)t * PW + h * (D + 2) + D));
        float o = 0.f, l = 0.f;
        for (int t = 0; t < nsplit; ++t) {
            const float mt = __ldcg(pu + (size_t)t * PW + h * (D + 2) + D);
            const float f = (mt == -INFINITY) ? 0.f : exp2f(mt - M);
            o += __ldcg(pu + (size_t)t * PW + h * (D + 2) + c) * f;
            l += __ldcg(pu + (size_t)t * PW + h * (D + 2) + D + 1) * f;
        }
        out[((size_t)u * G + h) * D + c] = l > 0.f ? o / l : 0.f;
    }
    if (tid == 0) counters[u] = 0;
}

template <typename T, int G>
cudaError_t launch_attn_t(const void* q, const void* K, const void* V, const int32_t* idx,
                          const int32_t* count, int units, int max_len, int sinks,
                          int clustered_end, int cur_len, int B, float* out, float* part,
                          int32_t* counters, int max_splits, int32_t* dev_err, cudaStream_t st) {
    using S = AttnShape<T, G>;
    const int rows = sinks + (cur_len - clustered_end) + B;
    const int splits = (rows + S::RS - 1) / S::RS;
    if (splits > max_splits) return cudaErrorInvalidValue;
    const size_t smem = (size_t)2 * S::RS * D * sizeof(T) + (size_t)4 * G * (D + 2) * sizeof(float) +
                        (size_t)4 * S::RPI * S::NB * G * sizeof(float);
    auto kern = attn_kernel<T, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const float qscale = 1.4426950408889634f / sqrtf((float)D);
    dim3 grid(splits, units);
    kern<<<grid, 128, smem, st>>>((const T*)q, (const T*)K, (const T*)V, idx, count, max_len, sinks,
                                  clustered_end, cur_len, B, qscale, out, part, counters, dev_err);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_score_t(const void* q, const void* mu, int g, int units, int cmax, int C,
                           float* scores, int stride, cudaStream_t s) {
    constexpr int RPW = (32 / (D / Vec<T>::N)) * 4;  // rows per warp
    dim3 grid((C + 8 * RPW - 1) / (8 * RPW), units);
    switch (g) {
        case 1: score_kernel<T, 1><<<grid, 256, 0, s>>>((const T*)q, (const T*)mu, cmax, C, scores, stride); break;
        case 2: score_kernel<T, 2><<<grid, 256, 0, s>>>((const T*)q, (const T*)mu, cmax, C, scores, stride); break;
        case 4: score_kernel<T, 4><<<grid, 256, 0, s>>>((const T*)q, (const T*)mu, cmax, C, scores, stride); break;
        case 8: score_kernel<T, 8><<<grid, 256, 0, s>>>((const T*)q, (const T*)mu, cmax, C, scores, stride); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score(const ckv_ctx* ctx, const void* q, int C, float* scores, int stride,
                         cudaStream_t s) {
    if (C <= 0) return cudaSuccess;
    if (ctx->cfg.kv_dtype == CKV_BF16)
        return launch_score_t<__nv_bfloat16>(q, ctx->mu_s, ctx->cfg.g, ctx->cfg.units, ctx->cmax, C,
                                             scores, stride, s);
    return launch_score_t<float>(q, ctx->mu_s, ctx->cfg.g, ctx->cfg.units, ctx->cmax, C, scores,
                                 stride, s);
}

cudaError_t launch_select(const ckv_ctx* ctx, const float* scores, int stride, int C, int B,
                          int32_t* idx, int32_t* count, cudaStream_t s) {
    int npow2 = 1;
    while (npow2 < C) npow2 <<= 1;
    if (npow2 < 2) npow2 = 2;
    const size_t smem = (size_t)npow2 * 16;
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    select_kernel<<<ctx->cfg.units, SEL_THREADS, smem, s>>>(scores, stride, C, npow2, ctx->sizes,
                                                            ctx->offsets, ctx->perm, ctx->cmax,
                                                            ctx->ntok, B, idx, count, ctx->dev_err);
    return cudaGetLastError();
}

int attention_rows_per_split(int kv_dtype, int g) {
    if (kv_dtype == CKV_BF16) {
        switch (g) {
            case 1: return AttnShape<__nv_bfloat16, 1>::RS;
            case 2: return AttnShape<__nv_bfloat16, 2>::RS;
            case 4: return AttnShape<__nv_bfloat16, 4>::RS;
            case 8: return AttnShape<__nv_bfloat16, 8>::RS;
        }
    } else {
        switch (g) {
            case 1: return AttnShape<float, 1>::RS;
            case 2: return AttnShape<float, 2>::RS;
            case 4: return AttnShape<float, 4>::RS;
            case 8: return AttnShape<float, 8>::RS;
        }
    }
    return 0;
}

cudaError_t launch_attention(const void* q, const void* K, const void* V, const int32_t* idx,
                             const int32_t* count, int units, int g, int kv_dtype, int max_len,
                             int sinks, int clustered_end, int cur_len, int B, float* out,
                             float* part, int32_t* counters, int max_splits, int32_t* dev_err,
                             int num_sms, cudaStream_t s) {
    (void)num_sms;
#define CKV_ATTN(T, G)                                                                          \
    return launch_attn_t<T, G>(q, K, V, idx, count, units, max_len, sinks, clustered_end,      \
                               cur_len, B, out, part, counters, max_splits, dev_err, s)
    if (kv_dtype == CKV_BF16) {
        switch (g) {
            case 1: CKV_ATTN(__nv_bfloat16, 1);
            case 2: CKV_ATTN(__nv_bfloat16, 2);
            case 4: CKV_ATTN(__nv_bfloat16, 4);
            case 8: CKV_ATTN(__nv_bfloat16, 8);
        }
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
