// Cosine K-means over each unit's keys (ClusterKV page, section "Clustering in
// semantic space": sampled keys as initial centroids, assignment to the
// centroid of largest cosine similarity, centroid = mean of the assigned keys;
// clustering strategy during inference: 16 sinks kept, prompt clustered at
// prefill, every m = 320 new tokens clustered among themselves into C+ = 4).
//
// The update is a deterministic segmented reduction instead of the page's
// shared-memory atomicAdd kernel (section "Semantic clustering optimisation",
// Fig. 7): per-chunk label histograms, a scan, a stable scatter of token ids
// into a label-sorted permutation (the cluster metadata of section "Selection
// and indexing mechanism", Fig. 8), then per-cluster sums over fixed 64-row
// segments of that permutation with compensated fp32 summation in a fixed
// order, and a per-cluster combine of the segments in order.  No float
// atomics: the result is bit-reproducible.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace ckv {

cudaError_t launch_assign_tc(const ckv_ctx* ctx, const void* K, int n, int C, int32_t* labels,
                             cudaStream_t s);

namespace {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ void set_err(int32_t* err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// lane `lane` of a warp loads channels [4*lane, 4*lane + 4) of a key row
__device__ __forceinline__ float4 load4(const float* row, int lane) {
    return *reinterpret_cast<const float4*>(row + 4 * lane);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* row, int lane) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + 4 * lane);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

// Centroid operand copies from one fp32 centroid row held as float4 per lane:
// the scoring copy (bf16 of mu) and the normalised direction mu / ||mu||
// (bf16 for bf16 keys, else fp32).  ||mu||^2 is summed per lane then by a
// fixed xor tree, so every lane gets identical bits; zero rows give 0.
__device__ __forceinline__ float4 normalise(float4 v) {
    float ss = v.x * v.x;
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
    const float nrm = sqrtf(ss);
    if (!(nrm > 0.f)) return make_float4(0.f, 0.f, 0.f, 0.f);
    return make_float4(v.x / nrm, v.y / nrm, v.z / nrm, v.w / nrm);
}

__device__ __forceinline__ void write_shadows(float4 v, int lane, bool bf16, __nv_bfloat16* mus_row,
                                              void* muhat_row) {
    const float4 x = normalise(v);
    if (bf16) {
        *reinterpret_cast<uint2*>(mus_row + 4 * lane) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(muhat_row) + 4 * lane) =
            make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
    } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(muhat_row) + 4 * lane) = x;
    }
}

struct StateRefs {
    float* mu32;
    __nv_bfloat16* mu_s;  // null for fp32 keys (the fp32 master is the scoring copy)
    void* mu_hat;
    int cmax, cmax_pad;
    bool bf16;
    __device__ __forceinline__ void store(int u, int c, float4 v, int lane) const {
        *reinterpret_cast<float4*>(mu32 + ((size_t)u * cmax + c) * D + 4 * lane) = v;
        __nv_bfloat16* mus = bf16 ? mu_s + ((size_t)u * cmax + c) * D : nullptr;
        void* mh = bf16 ? (void*)(reinterpret_cast<__nv_bfloat16*>(mu_hat) + ((size_t)u * cmax_pad + c) * D)
                        : (void*)(reinterpret_cast<float*>(mu_hat) + ((size_t)u * cmax_pad + c) * D);
        write_shadows(v, lane, bf16, mus, mh);
    }
};

StateRefs refs(const ckv_ctx* ctx) {
    StateRefs r;
    r.mu32 = ctx->mu32;
    r.bf16 = ctx->cfg.kv_dtype == CKV_BF16;
    r.mu_s = r.bf16 ? reinterpret_cast<__nv_bfloat16*>(ctx->mu_s) : nullptr;
    r.mu_hat = ctx->mu_hat;
    r.cmax = ctx->cmax;
    r.cmax_pad = ctx->cmax_pad;
    return r;
}

// ---------------------------------------------------------------- shadows / seed
__global__ void __launch_bounds__(256) shadows_kernel(StateRefs st, int c0, int c1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = c0 + blockIdx.x * 8 + warp, u = blockIdx.y;
    if (c >= c1) return;
    const float4 v = load4(st.mu32 + ((size_t)u * st.cmax + c) * D, lane);
    st.store(u, c, v, lane);
}

template <typename T>
__global__ void __launch_bounds__(256) seed_kernel(const T* __restrict__ K, int max_len, int first,
                                                   int stride, int C, StateRefs st) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x * 8 + warp, u = blockIdx.y;
    if (j >= C) return;
    const float4 v = load4(K + ((size_t)u * max_len + first + (size_t)j * stride) * D, lane);
    st.store(u, j, v, lane);
}

// ---------------------------------------------------------------- fp32-key assignment
// One thread per key, key in registers, centroid directions staged through
// shared memory 32 at a time; dot products in fp32 in channel order.
__global__ void __launch_bounds__(128) assign_f32_kernel(const float* __restrict__ K, int max_len,
                                                         int sinks, int n, const float* __restrict__ mu_hat,
                                                         int cmax_pad, int C, int32_t* __restrict__ labels) {
    __shared__ __align__(16) float cs[32][D];
    const int u = blockIdx.y, i = blockIdx.x * 128 + threadIdx.x;
    const bool valid = i < n;
    float k[D];
    if (valid) {
        const float4* row = reinterpret_cast<const float4*>(K + ((size_t)u * max_len + sinks + i) * D);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) {
            const float4 v = row[c];
            k[4 * c] = v.x;
            k[4 * c + 1] = v.y;
            k[4 * c + 2] = v.z;
            k[4 * c + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int c = 0; c < D; ++c) k[c] = 0.f;
    }
    float best = -INFINITY;
    int arg = 0;
    for (int c0 = 0; c0 < C; c0 += 32) {
        __syncthreads();
        const int nc = min(32, C - c0);
        for (int e = threadIdx.x; e < nc * (D / 4); e += 128) {
            const int r = e / (D / 4), q = e % (D / 4);
            reinterpret_cast<float4*>(cs[r])[q] =
                reinterpret_cast<const float4*>(mu_hat + ((size_t)u * cmax_pad + c0 + r) * D)[q];
        }
        __syncthreads();
        for (int r = 0; r < nc; ++r) {
            float dot = 0.f;
#pragma unroll
            for (int c = 0; c < D; ++c) dot = fmaf(k[c], cs[r][c], dot);
            if (dot > best) {
                best = dot;
                arg = c0 + r;
            }
        }
    }
    if (valid) labels[(size_t)u * n + i] = arg;
}

// ---------------------------------------------------------------- block scan
// Exclusive scan of a[0..count) in shared memory by a 1024-thread block;
// returns the total.  Each thread owns a contiguous run.
__device__ int block_exclusive_scan(int32_t* a, int count, int32_t* warp_buf /*[33]*/) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (count + 1023) / 1024;
    const int b0 = tid * per;
    int run = 0;
    for (int i = b0; i < b0 + per && i < count; ++i) run += a[i];
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_buf[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int wt = warp_buf[lane];
        int wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, wi, o);
            if (lane >= o) wi += t;
        }
        warp_buf[lane] = wi - wt;
        if (lane == 31) warp_buf[32] = wi;
    }
    __syncthreads();
    int base = warp_buf[warp] + incl - run;
    for (int i = b0; i < b0 + per && i < count; ++i) {
        const int v = a[i];
        a[i] = base;
        base += v;
    }
    const int total = warp_buf[32];
    __syncthreads();
    return total;
}

// ---------------------------------------------------------------- CSR build
__global__ void __launch_bounds__(1024) csr_count_kernel(const int32_t* __restrict__ labels, int n, int C,
                                                         int cmax, int nchunk, int32_t* __restrict__ chunk_cnt,
                                                         int32_t* dev_err) {
    extern __shared__ int32_t hist[];
    const int u = blockIdx.y, k = blockIdx.x, tid = threadIdx.x;
    for (int c = tid; c < C; c += 1024) hist[c] = 0;
    __syncthreads();
    const int i = k * CSR_CHUNK + tid;
    if (i < n) {
        int l = labels[(size_t)u * n + i];
        if (l < 0 || l >= C) {
            set_err(dev_err, CKV_DEV_BAD_LABEL);
            l = 0;
        }
        atomicAdd(&hist[l], 1);
    }
    __syncthreads();
    int32_t* out = chunk_cnt + ((size_t)u * nchunk + k) * cmax;
    for (int c = tid; c < C; c += 1024) out[c] = hist[c];
}

__global__ void __launch_bounds__(1024) csr_scan_kernel(int n, int C, int cmax, int nchunk,
                                                        int32_t* __restrict__ chunk_cnt, int32_t* __restrict__ sizes,
                                                        int32_t* __restrict__ offsets, int32_t* __restrict__ task_off,
                                                        int32_t* __restrict__ task_cl, int max_tasks) {
    extern __shared__ int32_t sm[];
    int32_t* off = sm;          // [C]
    int32_t* tk = sm + C;       // [C]
    __shared__ int32_t wb[33];
    const int u = blockIdx.x, tid = threadIdx.x;
    for (int c = tid; c < C; c += 1024) {
        // chunk counts of cluster c -> exclusive prefix over chunks, 16 loads in flight
        int run = 0;
        int32_t* col = chunk_cnt + (size_t)u * nchunk * cmax + c;
        for (int k0 = 0; k0 < nchunk; k0 += 16) {
            int v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = (k0 + j < nchunk) ? col[(size_t)(k0 + j) * cmax] : 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (k0 + j < nchunk) col[(size_t)(k0 + j) * cmax] = run;
                run += v[j];
            }
        }
        sizes[(size_t)u * cmax + c] = run;
        off[c] = run;
        tk[c] = (run + SEG_ROWS - 1) / SEG_ROWS;
    }
    __syncthreads();
    const int total = block_exclusive_scan(off, C, wb);
    const int tasks = block_exclusive_scan(tk, C, wb);
    int32_t* o = offsets + (size_t)u * (cmax + 1);
    int32_t* to = task_off + (size_t)u * (cmax + 1);
    for (int c = tid; c < C; c += 1024) {
        o[c] = off[c];
        to[c] = tk[c];
        const int t1 = (c + 1 < C) ? tk[c + 1] : tasks;
        for (int t = tk[c]; t < t1; ++t) task_cl[(size_t)u * max_tasks + t] = c;
    }
    if (tid == 0) {
        o[C] = total;
        to[C] = tasks;
    }
    (void)n;
}

// One warp per chunk of CSR_CHUNK tokens: a per-cluster cursor in shared
// memory starts at the chunk's first position in each cluster's segment
// (cluster offset + the earlier chunks' counts), then the chunk's tokens go by
// in 32-token rounds, in index order: lanes with the same label find each other
// (match_any), take consecutive positions by lane order from the cursor, and
// the lowest of them advances it.  Every token lands at its stable
// (label, index) position with no atomics.
constexpr int SCATTER_WARPS = 8;

__global__ void __launch_bounds__(32 * SCATTER_WARPS) csr_scatter_kernel(
    const int32_t* __restrict__ labels, int n, int C, int cmax, int nchunk, const int32_t* __restrict__ chunk_cnt,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int ntok, int sinks, int cstride) {
    extern __shared__ int32_t cursor_all[];  // [SCATTER_WARPS][cstride]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.y, k = blockIdx.x * SCATTER_WARPS + warp;
    if (k >= nchunk) return;
    int32_t* cursor = cursor_all + warp * cstride;
    const int32_t* cc = chunk_cnt + ((size_t)u * nchunk + k) * cmax;
    const int32_t* of = offsets + (size_t)u * (cmax + 1);
    for (int c = lane; c < C; c += 32) cursor[c] = of[c] + cc[c];
    __syncwarp();
    const int32_t* lab = labels + (size_t)u * n;
    int32_t* pu = perm + (size_t)u * ntok;
    const int i0 = k * CSR_CHUNK;
    constexpr int ROUNDS = CSR_CHUNK / 32;
    constexpr int PF = 8;  // label loads in flight per lane
    for (int r0 = 0; r0 < ROUNDS; r0 += PF) {
        int lv[PF];
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            const int i = i0 + 32 * (r0 + j) + lane;
            int l = i < n ? lab[i] : -1;
            if (i < n && (l < 0 || l >= C)) l = 0;  // reported by the count pass
            lv[j] = l;
        }
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            const int i = i0 + 32 * (r0 + j) + lane;
            const int l = lv[j];
            const unsigned peers = __match_any_sync(FULL, l);
            const int leader = __ffs(peers) - 1;
            int base = 0;
            if (lane == leader && l >= 0) {
                base = cursor[l];
                cursor[l] = base + __popc(peers);
            }
            base = __shfl_sync(FULL, base, leader);
            if (l >= 0) pu[base + __popc(peers & ((1u << lane) - 1u))] = sinks + i;
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------------- centroid sums
// Kahan-compensated accumulation
struct Kahan {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float y = x - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
    __device__ __forceinline__ float value() const { return s - c; }
};

template <typename T>
__global__ void __launch_bounds__(256) segsum_kernel(const T* __restrict__ K, int max_len, int C,
                                                     const int32_t* __restrict__ sizes,
                                                     const int32_t* __restrict__ offsets,
                                                     const int32_t* __restrict__ perm,
                                                     const int32_t* __restrict__ task_off,
                                                     const int32_t* __restrict__ task_cl, int cmax, int ntok,
                                                     int max_tasks, float* __restrict__ seg_part) {
    constexpr int CPL = 16 / (int)sizeof(T);  // channels per lane
    constexpr int LPR = D / CPL;              // lanes per row
    constexpr int RPI = 32 / LPR;             // rows in flight per warp-wide load
    __shared__ int32_t toks[8][SEG_ROWS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.y, t = blockIdx.x * 8 + warp;
    const int32_t* to = task_off + (size_t)u * (cmax + 1);
    if (t >= to[C]) return;
    const int c = task_cl[(size_t)u * max_tasks + t];
    const int seg = t - to[c];
    const int cbeg = offsets[(size_t)u * (cmax + 1) + c];
    const int beg = cbeg + seg * SEG_ROWS;
    const int rows = min(SEG_ROWS, cbeg + sizes[(size_t)u * cmax + c] - beg);
    for (int r = lane; r < rows; r += 32) toks[warp][r] = perm[(size_t)u * ntok + beg + r];
    __syncwarp();
    const int sub = lane / LPR, li = lane % LPR;
    Kahan acc[CPL];
    const T* Ku = K + (size_t)u * max_len * D + li * CPL;
    constexpr int SUNR = 8;  // row loads in flight per lane
    for (int r0 = sub; r0 < rows; r0 += SUNR * RPI) {
        uint4 w[SUNR];
#pragma unroll
        for (int q = 0; q < SUNR; ++q) {
            const int r = r0 + q * RPI;
            w[q] = r < rows ? *reinterpret_cast<const uint4*>(Ku + (size_t)toks[warp][r] * D)
                            : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < SUNR; ++q) {
            if (r0 + q * RPI >= rows) break;
            if constexpr (sizeof(T) == 2) {
                const uint32_t ww[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[2 * e].add(__uint_as_float(ww[e] << 16));
                    acc[2 * e + 1].add(__uint_as_float(ww[e] & 0xffff0000u));
                }
            } else {
                acc[0].add(__uint_as_float(w[q].x));
                acc[1].add(__uint_as_float(w[q].y));
                acc[2].add(__uint_as_float(w[q].z));
                acc[3].add(__uint_as_float(w[q].w));
            }
        }
    }
    float v[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        v[e] = acc[e].value();
        if constexpr (RPI == 2) v[e] += __shfl_xor_sync(FULL, v[e], 16);  // even rows + odd rows
    }
    if (sub == 0) {
        float* out = seg_part + ((size_t)u * max_tasks + t) * D + li * CPL;
#pragma unroll
        for (int e = 0; e < CPL; e += 4)
            *reinterpret_cast<float4*>(out + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    }
}

__global__ void __launch_bounds__(256) finalize_kernel(int C, const int32_t* __restrict__ sizes,
                                                       const int32_t* __restrict__ task_off,
                                                       const float* __restrict__ seg_part, int max_tasks,
                                                       StateRefs st) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x * 8 + warp, u = blockIdx.y;
    if (c >= C) return;
    const int sz = sizes[(size_t)u * st.cmax + c];
    if (sz == 0) return;  // empty cluster keeps its centroid
    const int32_t* to = task_off + (size_t)u * (st.cmax + 1);
    Kahan a[4];
    for (int t = to[c]; t < to[c + 1]; ++t) {
        const float4 p = *reinterpret_cast<const float4*>(seg_part + ((size_t)u * max_tasks + t) * D + 4 * lane);
        a[0].add(p.x);
        a[1].add(p.y);
        a[2].add(p.z);
        a[3].add(p.w);
    }
    const float fs = (float)sz;
    const float4 mean = make_float4(a[0].value() / fs, a[1].value() / fs, a[2].value() / fs, a[3].value() / fs);
    st.store(u, c, mean, lane);
}

// ---------------------------------------------------------------- incremental
// One CTA per unit clusters the m newest keys into cp clusters entirely in
// shared memory: keys in their own dtype (bf16 rows at a 272-byte pitch, fp32
// rows padded to D+1 floats), stride seeding, `iters` Lloyd iterations with the
// same operand precision as the prefill path, then the CSR segment is appended.
// Per iteration:
//   assignment  bf16 keys: mma.sync m16n8k16 (16 keys x 8 centroid directions
//               per instruction; exact bf16 products, fp32 sums), arg-max over
//               the columns of each row in a lane quad; fp32 keys: one thread
//               per key, fp32 dot products;
//   order       warp 0 builds the stable cluster order of the keys (counts by
//               ballot, ranks by match_any), i.e. this iteration's CSR;
//   update      thread (cluster, channel) sums its channel over the cluster's
//               keys in token order (compensated), mean of the raw keys; an
//               empty cluster keeps its centroid.
constexpr int INCR_THREADS = 512;
constexpr int INCR_MAX_CP = 16;

template <typename T>
struct IncrLayout {
    static constexpr bool BF16 = sizeof(T) == 2;
    static constexpr int KP = BF16 ? D + 8 : D + 1;  // row pitch in elements
};

__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(float x) { return x; }

__device__ __forceinline__ uint32_t pack_bf16_exact(float lo, float hi) {
    // both values are bf16-representable: keep their top halves
    return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xffff0000u);
}

template <typename T>
__global__ void __launch_bounds__(INCR_THREADS) incr_kernel(const T* __restrict__ K, int max_len, int start,
                                                            int m, int cp, int iters, int stride, int C_old,
                                                            int csr_base, StateRefs st, int32_t* __restrict__ sizes,
                                                            int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                            int ntok) {
    using LY = IncrLayout<T>;
    constexpr int KP = LY::KP;
    extern __shared__ __align__(16) unsigned char incr_smem[];
    const int m16 = (m + 15) & ~15;
    T* ks = reinterpret_cast<T*>(incr_smem);                                   // [m16][KP]
    int32_t* lab = reinterpret_cast<int32_t*>(ks + (size_t)m16 * KP);          // [m16]
    int32_t* order = lab + m16;                                                // [m16]
    __shared__ __align__(16) float mu[INCR_MAX_CP][D];
    __shared__ __align__(16) float muh[INCR_MAX_CP][D];
    __shared__ int32_t cnt[INCR_MAX_CP], off[INCR_MAX_CP], run[INCR_MAX_CP];
    const int u = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwarps = INCR_THREADS / 32;

    // keys (rows past m are zero: they only pad the last 16-row MMA tile)
    for (int r = warp; r < m16; r += nwarps) {
        T* dst = ks + (size_t)r * KP;
        if (r < m) {
            const T* src = K + ((size_t)u * max_len + start + r) * D;
            if constexpr (LY::BF16) {
                reinterpret_cast<uint2*>(dst)[lane] = reinterpret_cast<const uint2*>(src)[lane];
            } else {
                const float4 v = reinterpret_cast<const float4*>(src)[lane];
                dst[4 * lane] = v.x;
                dst[4 * lane + 1] = v.y;
                dst[4 * lane + 2] = v.z;
                dst[4 * lane + 3] = v.w;
            }
        } else {
            for (int c = lane; c < D; c += 32) dst[c] = T(0.f);
        }
    }
    __syncthreads();
    for (int e = tid; e < cp * D; e += INCR_THREADS)
        mu[e / D][e % D] = to_f32(ks[(size_t)(e / D) * stride * KP + e % D]);
    for (int j = tid; j < cp; j += INCR_THREADS) cnt[j] = 0;
    __syncthreads();

    for (int it = 0; it < iters; ++it) {
        // centroid directions in the operand precision
        for (int j = warp; j < cp; j += nwarps) {
            const float4 v = make_float4(mu[j][4 * lane], mu[j][4 * lane + 1], mu[j][4 * lane + 2], mu[j][4 * lane + 3]);
            float4 x = normalise(v);
            if (st.bf16) {
                x.x = __bfloat162float(__float2bfloat16_rn(x.x));
                x.y = __bfloat162float(__float2bfloat16_rn(x.y));
                x.z = __bfloat162float(__float2bfloat16_rn(x.z));
                x.w = __bfloat162float(__float2bfloat16_rn(x.w));
            }
            muh[j][4 * lane] = x.x;
            muh[j][4 * lane + 1] = x.y;
            muh[j][4 * lane + 2] = x.z;
            muh[j][4 * lane + 3] = x.w;
        }
        __syncthreads();
        // ---- assignment: lab[i] = arg-max_j k_i . muh_j, ties to the lower j
        if constexpr (LY::BF16) {
            const int g = lane >> 2, q4 = lane & 3;
            const int ntiles = (cp + 7) >> 3;  // 8 centroid columns per MMA
            const uint32_t kbase = static_cast<uint32_t>(__cvta_generic_to_shared(ks));
            for (int mt = warp; mt < m16 / 16; mt += nwarps) {
                float best0 = -INFINITY, best1 = -INFINITY;
                int arg0 = 0, arg1 = 0;
                for (int nt = 0; nt < ntiles; ++nt) {
                    const int col = nt * 8 + g;  // centroid of this lane's B column
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int mi = lane >> 3;
                        const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
                        const uint32_t addr =
                            kbase + (uint32_t)(row * KP + kk * 16 + (mi >> 1) * 8) * 2u;
                        uint32_t a0, a1, a2, a3;
                        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                                     : "r"(addr));
                        uint32_t b0 = 0u, b1 = 0u;
                        if (col < cp) {
                            const float* mh = muh[col] + kk * 16 + 2 * q4;
                            b0 = pack_bf16_exact(mh[0], mh[1]);
                            b1 = pack_bf16_exact(mh[8], mh[9]);
                        }
                        asm volatile(
                            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                            : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
                            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                    }
                    // this lane holds rows g (acc 0, 1) and g + 8 (acc 2, 3),
                    // columns nt*8 + 2*q4 and + 1, visited in increasing order
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int cc = nt * 8 + 2 * q4 + e;
                        if (cc < cp) {
                            if (acc[e] > best0) { best0 = acc[e]; arg0 = cc; }
                            if (acc[2 + e] > best1) { best1 = acc[2 + e]; arg1 = cc; }
                        }
                    }
                }
                // quad reduction: larger value, then lower column
#pragma unroll
                for (int o = 1; o <= 2; o <<= 1) {
                    const float ob0 = __shfl_xor_sync(FULL, best0, o), ob1 = __shfl_xor_sync(FULL, best1, o);
                    const int oa0 = __shfl_xor_sync(FULL, arg0, o), oa1 = __shfl_xor_sync(FULL, arg1, o);
                    if (ob0 > best0 || (ob0 == best0 && oa0 < arg0)) { best0 = ob0; arg0 = oa0; }
                    if (ob1 > best1 || (ob1 == best1 && oa1 < arg1)) { best1 = ob1; arg1 = oa1; }
                }
                if (q4 == 0) {
                    lab[mt * 16 + g] = arg0;
                    lab[mt * 16 + g + 8] = arg1;
                }
            }
        } else {
            for (int i = tid; i < m; i += INCR_THREADS) {
                const T* kr = ks + (size_t)i * KP;
                float best = -INFINITY;
                int arg = 0;
                for (int j = 0; j < cp; ++j) {
                    float dot = 0.f;
#pragma unroll 8
                    for (int c = 0; c < D; ++c) dot = fmaf(to_f32(kr[c]), muh[j][c], dot);
                    if (dot > best) {
                        best = dot;
                        arg = j;
                    }
                }
                lab[i] = arg;
            }
        }
        __syncthreads();
        // ---- stable cluster order of the keys (warp 0)
        if (warp == 0) {
            int my_cnt = 0;  // lane j < cp: size of cluster j
            for (int b = 0; b < m; b += 32) {
                const int l = (b + lane < m) ? lab[b + lane] : -1;
                for (int j = 0; j < cp; ++j) {
                    const int n = __popc(__ballot_sync(FULL, l == j));
                    if (lane == j) my_cnt += n;
                }
            }
            int incl = my_cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
            }
            if (lane < cp) {
                cnt[lane] = my_cnt;
                off[lane] = incl - my_cnt;
                run[lane] = 0;
            }
            __syncwarp();
            for (int b = 0; b < m; b += 32) {
                const int i = b + lane;
                const int l = i < m ? lab[i] : -1;
                const unsigned peers = __match_any_sync(FULL, l);
                const int rank = __popc(peers & ((1u << lane) - 1u));
                if (i < m) order[off[l] + run[l] + rank] = i;
                __syncwarp();
                if (i < m && rank == 0) run[l] += __popc(peers);
                __syncwarp();
            }
        }
        __syncthreads();
        // ---- update: thread (j, c) over cluster j's keys in token order
        for (int e = tid; e < cp * D; e += INCR_THREADS) {
            const int j = e / D, c = e % D;
            const int n = cnt[j], o0 = off[j];
            if (n > 0) {
                Kahan a;
                for (int p = 0; p < n; ++p) a.add(to_f32(ks[(size_t)order[o0 + p] * KP + c]));
                mu[j][c] = a.value() / (float)n;
            }
        }
        __syncthreads();
    }

    // CSR segment of the last assignment: sizes, offsets, stable permutation
    if (iters > 0)
        for (int p = tid; p < m; p += INCR_THREADS) perm[(size_t)u * ntok + csr_base + p] = start + order[p];
    else if (tid == 0)
        for (int j = 0; j < cp; ++j) off[j] = 0;
    __syncthreads();
    if (iters == 0)  // no assignment: every key in cluster 0 (the seeds are the centroids)
        for (int p = tid; p < m; p += INCR_THREADS) perm[(size_t)u * ntok + csr_base + p] = start + p;
    for (int j = warp; j < cp; j += nwarps) {
        const float4 v = make_float4(mu[j][4 * lane], mu[j][4 * lane + 1], mu[j][4 * lane + 2], mu[j][4 * lane + 3]);
        st.store(u, C_old + j, v, lane);
        if (lane == 0) {
            sizes[(size_t)u * st.cmax + C_old + j] = iters > 0 ? cnt[j] : (j == 0 ? m : 0);
            offsets[(size_t)u * (st.cmax + 1) + C_old + j] = csr_base + (iters > 0 ? off[j] : (j == 0 ? 0 : m));
        }
    }
    if (tid == 0) offsets[(size_t)u * (st.cmax + 1) + C_old + cp] = csr_base + m;
}

template <typename T>
cudaError_t update_t(const ckv_ctx* ctx, const T* K, int n, int C, const int32_t* labels, cudaStream_t s) {
    const int U = ctx->cfg.units;
    const int nchunk = ceil_div(n, CSR_CHUNK);
    const size_t hsm = (size_t)C * sizeof(int32_t);
    csr_count_kernel<<<dim3(nchunk, U), 1024, hsm, s>>>(labels, n, C, ctx->cmax, nchunk, ctx->chunk_cnt,
                                                        ctx->dev_err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t ssm = (size_t)2 * C * sizeof(int32_t);
    e = cudaFuncSetAttribute(csr_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
    if (e != cudaSuccess) return e;
    csr_scan_kernel<<<U, 1024, ssm, s>>>(n, C, ctx->cmax, nchunk, ctx->chunk_cnt, ctx->sizes, ctx->offsets,
                                         ctx->task_off, ctx->task_cl, ctx->max_tasks);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int cstride = round_up(C, 32);
    const size_t wsm = (size_t)SCATTER_WARPS * cstride * sizeof(int32_t);
    e = cudaFuncSetAttribute(csr_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsm);
    if (e != cudaSuccess) return e;
    csr_scatter_kernel<<<dim3(ceil_div(nchunk, SCATTER_WARPS), U), 32 * SCATTER_WARPS, wsm, s>>>(
        labels, n, C, ctx->cmax, nchunk, ctx->chunk_cnt, ctx->offsets, ctx->perm, ctx->ntok, ctx->cfg.sinks, cstride);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int max_t = ceil_div(n, SEG_ROWS) + C;
    segsum_kernel<T><<<dim3(ceil_div(max_t, 8), U), 256, 0, s>>>(
        K, ctx->cfg.max_len, C, ctx->sizes, ctx->offsets, ctx->perm, ctx->task_off, ctx->task_cl, ctx->cmax,
        ctx->ntok, ctx->max_tasks, ctx->seg_part);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    finalize_kernel<<<dim3(ceil_div(C, 8), U), 256, 0, s>>>(C, ctx->sizes, ctx->task_off, ctx->seg_part,
                                                            ctx->max_tasks, refs(ctx));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_shadows(const ckv_ctx* ctx, int c0, int c1, cudaStream_t s) {
    if (c1 <= c0) return cudaSuccess;
    shadows_kernel<<<dim3(ceil_div(c1 - c0, 8), ctx->cfg.units), 256, 0, s>>>(refs(ctx), c0, c1);
    return cudaGetLastError();
}

cudaError_t launch_seed(const ckv_ctx* ctx, const void* K, int C, int stride, cudaStream_t s) {
    dim3 grid(ceil_div(C, 8), ctx->cfg.units);
    if (ctx->cfg.kv_dtype == CKV_BF16)
        seed_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)K, ctx->cfg.max_len, ctx->cfg.sinks,
                                                        stride, C, refs(ctx));
    else
        seed_kernel<float><<<grid, 256, 0, s>>>((const float*)K, ctx->cfg.max_len, ctx->cfg.sinks, stride, C,
                                                refs(ctx));
    return cudaGetLastError();
}

cudaError_t launch_assign(const ckv_ctx* ctx, const void* K, int n, int C, int32_t* labels, cudaStream_t s) {
    if (ctx->cfg.kv_dtype == CKV_BF16) return launch_assign_tc(ctx, K, n, C, labels, s);
    assign_f32_kernel<<<dim3(ceil_div(n, 128), ctx->cfg.units), 128, 0, s>>>(
        (const float*)K, ctx->cfg.max_len, ctx->cfg.sinks, n, (const float*)ctx->mu_hat, ctx->cmax_pad, C, labels);
    return cudaGetLastError();
}

cudaError_t launch_update(const ckv_ctx* ctx, const void* K, int n, int C, const int32_t* labels,
                          cudaStream_t s) {
    if (ctx->cfg.kv_dtype == CKV_BF16) return update_t(ctx, (const __nv_bfloat16*)K, n, C, labels, s);
    return update_t(ctx, (const float*)K, n, C, labels, s);
}

size_t incremental_smem(int m, bool bf16) {
    const size_t m16 = (size_t)((m + 15) & ~15);
    const size_t row = bf16 ? (size_t)IncrLayout<__nv_bfloat16>::KP * 2 : (size_t)IncrLayout<float>::KP * 4;
    return m16 * row + 2 * m16 * sizeof(int32_t);
}

cudaError_t launch_incremental(const ckv_ctx* ctx, const void* K, int start, int m, int c_plus, int C_old,
                               int csr_base, cudaStream_t s) {
    if (c_plus > INCR_MAX_CP) return cudaErrorInvalidValue;
    const size_t smem = incremental_smem(m, ctx->cfg.kv_dtype == CKV_BF16);
    const int stride = (m / c_plus) < ctx->cfg.ratio ? (m / c_plus) : ctx->cfg.ratio;
    cudaError_t e;
    if (ctx->cfg.kv_dtype == CKV_BF16) {
        e = cudaFuncSetAttribute(incr_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        incr_kernel<__nv_bfloat16><<<ctx->cfg.units, INCR_THREADS, smem, s>>>(
            (const __nv_bfloat16*)K, ctx->cfg.max_len, start, m, c_plus, ctx->cfg.iters, stride < 1 ? 1 : stride,
            C_old, csr_base, refs(ctx), ctx->sizes, ctx->offsets, ctx->perm, ctx->ntok);
    } else {
        e = cudaFuncSetAttribute(incr_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        incr_kernel<float><<<ctx->cfg.units, INCR_THREADS, smem, s>>>(
            (const float*)K, ctx->cfg.max_len, start, m, c_plus, ctx->cfg.iters, stride < 1 ? 1 : stride, C_old,
            csr_base, refs(ctx), ctx->sizes, ctx->offsets, ctx->perm, ctx->ntok);
    }
    return cudaGetLastError();
}

}  // namespace ckv
