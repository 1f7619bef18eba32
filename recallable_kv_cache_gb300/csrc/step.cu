// One decode step of every unit with the cluster selection and the sparse
// attention in one persistent kernel (ClusterKV page: section "Selection and
// indexing mechanism", Fig. 8, for the selection; section "Background" for
// softmax(q K_S^T / sqrt(d)) V_S over the attended set S = sinks + pending
// tokens + the selected clusters' tokens).
//
// The selection of a unit is short but latency-bound, and the HBM sits idle
// while it runs if the attention waits for every selection to finish.  Here
// each CTA (one per SM) holds two kinds of warps:
//   selector warps (2):  for their units, in turn: the scores written by the
//     scoring kernel, the cluster sizes and prefix offsets are loaded once;
//     an exact radix select over the score bits, weighted by cluster size,
//     finds the score at which the ranked sizes reach min(B, clustered
//     tokens); the clusters up to that score are sorted by (score desc,
//     index asc), their sizes prefix-summed, the last one trimmed, and the
//     token ids copied from the label-sorted permutation into idx in rank
//     order; then the unit's ready flag is released;
//   attention warps (10):  each walks two contiguous tile ranges (16 rows per
//     tile): first its share of the tiles that need no selection (the sinks
//     and the pending tokens of every unit), then its share of the selected
//     tiles, whose token ids it reads once the unit's flag is set.  So the
//     K/V stream starts while the selections run.  The per-warp ring, the
//     mma.sync arithmetic and the online softmax are those of the bf16
//     attention kernel; one partial per (unit, phase, warp).
// step_combine_kernel merges each unit's partials in a fixed order (phase
// then warp) and clears the unit's flag for the next step.
//
// Every wait on a flag is bounded: a selection that is not published in time
// counts as empty and sets CKV_DEV_TIMEOUT.  The selector warps wait only
// for the scoring kernel (griddepcontrol), the attention warps only for
// selector warps of this grid; one CTA per SM and a grid of at most one CTA
// per SM, so every CTA the attention waits for can become resident.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "mma_sync.cuh"
#include "ptx.cuh"

namespace ckv {
namespace {

using namespace mmas;

constexpr unsigned FULL = 0xffffffffu;
constexpr int SW = 2;             // selector warps per CTA
constexpr int AW = 10;            // attention warps per CTA
constexpr int NW = SW + AW;
constexpr int TR = 16;            // rows per tile
constexpr int NST = 2;            // ring stages per attention warp
constexpr int PITCH = D * 2 + 16; // 272-byte row pitch: conflict-free ldmatrix
constexpr int TILE_BYTES = TR * PITCH;
constexpr int STAGE_BYTES = 2 * TILE_BYTES;
constexpr int RING_BYTES = AW * NST * STAGE_BYTES;
constexpr int SEL_CMAX = STEP_MAX_CLUSTERS;  // clusters a selector warp holds in shared memory

struct SelScratch {
    uint64_t key[SEL_CMAX];  // rank keys; after the cut, the candidates in rank order
    int32_t sz[SEL_CMAX];    // sizes by cluster
    int32_t of[SEL_CMAX];    // prefix offsets by cluster
    int2 rso[SEL_CMAX];      // per rank: (first output slot, perm offset)
    int32_t hist[256];
};
constexpr size_t STEP_SMEM = (size_t)RING_BYTES + (size_t)SW * sizeof(SelScratch);

struct StepArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    const float* scores;
    const int32_t* sizes;
    const int32_t* offsets;
    const int32_t* perm;
    int32_t* idx;
    int32_t* count;
    int32_t* flag;
    int units, C, cmax, ntok, B;
    int max_len, sinks, clustered_end, cur_len;
    int tA, tB;      // tiles per unit: sinks + pending, selected
    int apw, bpw;    // tiles per attention warp of each phase
    int max_slots;
    float qscale;
    long long wait_limit;
    int stall;       // failure detection test: the selector warps publish nothing
    float* part;
    int32_t* dev_err;
};

__device__ __forceinline__ void set_err(int32_t* err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int32_t* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 64-bit rank key: ascending key = descending score, ties by ascending index
__device__ __forceinline__ uint64_t rank_key(float s, int c) {
    if (s == 0.f) s = 0.f;  // -0 ranks like +0
    const uint32_t b = __float_as_uint(s);
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((uint64_t)(~ord) << 32) | (uint32_t)c;
}
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

// ---------------------------------------------------------------------------
// selection of unit u by one warp
// ---------------------------------------------------------------------------
__device__ void warp_select(const StepArgs& a, SelScratch& s, int u, int lane) {
    const int C = a.C;
    // 1. scores (from the scoring kernel: read past L1), sizes, offsets
    int tot = 0;
    for (int c0 = 0; c0 < C; c0 += 32 * 16) {
        float scv[16];
        int szv[16], ofv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = c0 + 32 * i + lane;
            scv[i] = c < C ? __ldcg(a.scores + (size_t)u * a.cmax + c) : 0.f;
            szv[i] = c < C ? __ldcg(a.sizes + (size_t)u * a.cmax + c) : 0;
            ofv[i] = c < C ? __ldcg(a.offsets + (size_t)u * (a.cmax + 1) + c) : 0;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = c0 + 32 * i + lane;
            if (c < C) {
                s.key[c] = rank_key(scv[i], c);
                s.sz[c] = szv[i];
                s.of[c] = ofv[i];
                tot += szv[i];
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
    const int target = tot < a.B ? tot : a.B;
    __syncwarp();
    int R = 0;  // ranks taken
    if (target > 0) {
        // 2. radix select over the top 32 key bits (the inverted score), each
        // cluster weighted by its size: T = the score bits at which the ranked
        // sizes first reach the target.  Clusters above T (key bits < T) are
        // all taken; those at T are taken in index order.
        uint32_t prefix = 0, pmask = 0;
        int above = 0;
        for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) s.hist[lane * 8 + i] = 0;
            __syncwarp();
            for (int c = lane; c < C; c += 32) {
                const uint32_t h = (uint32_t)(s.key[c] >> 32);
                if ((h & pmask) == prefix) atomicAdd(&s.hist[(h >> shift) & 255], s.sz[c]);
            }
            __syncwarp();
            int hv[8], ls = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                hv[i] = s.hist[lane * 8 + i];
                ls += hv[i];
            }
            int incl = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
            }
            int run = above + incl - ls, bin = -1, ab = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (bin < 0 && run + hv[i] >= target) {
                    bin = lane * 8 + i;
                    ab = run;
                }
                run += hv[i];
            }
            const unsigned fb = __ballot_sync(FULL, bin >= 0);
            const int src = __ffs(fb) - 1;  // the first bin that reaches the target
            bin = __shfl_sync(FULL, bin, src);
            above = __shfl_sync(FULL, ab, src);
            prefix |= (uint32_t)bin << shift;
            pmask |= 255u << shift;
            __syncwarp();
        }
        // 3. candidates (key bits <= T), compacted in place in cluster order
        int M = 0;
        for (int c0 = 0; c0 < C; c0 += 32) {
            const int c = c0 + lane;
            const uint64_t k = c < C ? s.key[c] : ~0ull;
            const bool take = c < C && (uint32_t)(k >> 32) <= prefix;
            const unsigned b = __ballot_sync(FULL, take);
            __syncwarp();  // chunk read by every lane before any write below c0 + 32
            if (take) s.key[M + __popc(b & ((1u << lane) - 1u))] = k;
            M += __popc(b);
        }
        __syncwarp();
        // 4. rank order, 5. prefix of the ranked sizes and the cut
        if (M <= 32) {
            uint64_t k = lane < M ? s.key[lane] : ~0ull;
            k = warp_sort32(k, lane);
            const int c = (int)(uint32_t)k;
            const int z = lane < M ? s.sz[c] : 0;
            int incl = z;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
            }
            const unsigned reach = __ballot_sync(FULL, lane < M && incl >= target);
            R = __ffs(reach);  // > 0: the candidates hold the target
            if (lane < R) s.rso[lane] = make_int2(incl - z, s.of[c]);
        } else {
            int N2 = 64;
            while (N2 < M) N2 <<= 1;
            for (int i = M + lane; i < N2; i += 32) s.key[i] = ~0ull;
            __syncwarp();
            for (int k = 2; k <= N2; k <<= 1)
                for (int j = k >> 1; j > 0; j >>= 1) {
                    for (int i = lane; i < N2; i += 32) {
                        const int p = i ^ j;
                        if (p > i) {
                            const uint64_t x = s.key[i], y = s.key[p];
                            if ((x > y) == ((i & k) == 0)) {
                                s.key[i] = y;
                                s.key[p] = x;
                            }
                        }
                    }
                    __syncwarp();
                }
            int base = 0;
            for (int r0 = 0; r0 < M && R == 0; r0 += 32) {
                const int r = r0 + lane;
                const int c = r < M ? (int)(uint32_t)s.key[r] : 0;
                const int z = r < M ? s.sz[c] : 0;
                int incl = z;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(FULL, incl, o);
                    if (lane >= o) incl += t;
                }
                incl += base;
                const unsigned reach = __ballot_sync(FULL, r < M && incl >= target);
                const int lim = reach ? __ffs(reach) : 32;
                if (lane < lim && r < M) s.rso[r] = make_int2(incl - z, s.of[c]);
                if (reach) R = r0 + __ffs(reach);
                base = __shfl_sync(FULL, incl, 31);
            }
        }
        __syncwarp();
        // 6. output slot p -> the last rank whose first slot is <= p (that rank
        // is non-empty and holds p) -> its token id from the permutation
        const int32_t* pu = a.perm + (size_t)u * a.ntok;
        int32_t* out = a.idx + (size_t)u * a.B;
        for (int p0 = 0; p0 < target; p0 += 32 * 8) {
            int pos[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int p = p0 + 32 * i + lane;
                int lo = 0, hi = R - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s.rso[mid].x <= p) lo = mid;
                    else hi = mid - 1;
                }
                pos[i] = p < target ? s.rso[lo].y + (p - s.rso[lo].x) : -1;
            }
            int tok[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) tok[i] = ((unsigned)pos[i] < (unsigned)a.ntok) ? __ldcg(pu + pos[i]) : 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int p = p0 + 32 * i + lane;
                if (p < target) {
                    if ((unsigned)pos[i] >= (unsigned)a.ntok) set_err(a.dev_err, CKV_DEV_BAD_CSR);
                    out[p] = tok[i];
                }
            }
        }
    }
    if (lane == 0) a.count[u] = target;
    // 7. publish: every lane's idx stores, then the flag (release)
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release(a.flag + u, 1);
    __syncwarp();  // the scratch is reused for the next unit
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(NW * 32, 1) step_kernel(const StepArgs a) {
    constexpr int PW = G * (D + 2);
    extern __shared__ __align__(128) unsigned char step_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp >= AW) {
        // ================================================================ selectors
        SelScratch& s = reinterpret_cast<SelScratch*>(step_smem + RING_BYTES)[warp - AW];
        ptx::grid_dependency_wait();  // the scores come from the scoring kernel
        if (a.stall) return;          // no flag is ever set: every attention wait runs out
        for (int u = blockIdx.x * SW + (warp - AW); u < a.units; u += gridDim.x * SW) warp_select(a, s, u, lane);
        return;
    }

    // ==================================================================== attention
    // The attention warps read q, K and V (written before the scoring kernel
    // started: complete once this grid runs) and, per unit, idx and count after
    // that unit's flag; they never wait for the scoring kernel itself.
    const int aw = blockIdx.x * AW + warp;
    const int totA = a.units * a.tA, totB = a.units * a.tB;
    const int a_lo = min(totA, aw * a.apw), a_hi = min(totA, a_lo + a.apw);
    const int b_lo = min(totB, aw * a.bpw), b_hi = min(totB, b_lo + a.bpw);
    const int nAw = a_hi - a_lo, nT = nAw + (b_hi - b_lo);
    if (nT <= 0) return;
    unsigned char* wbase = step_smem + (size_t)warp * NST * STAGE_BYTES;
    const uint32_t wbase_addr = ptx::smem_u32(wbase);
    const int pend = a.cur_len - a.clustered_end;
    const int nsp = a.sinks + pend;

    // tile i of this warp: (unit, phase, tile of the phase within the unit)
    auto unit_of = [&](int i) -> int { return i < nAw ? (a_lo + i) / a.tA : (b_lo + i - nAw) / a.tB; };

    // token of row (lane & 15) of tile i, -1 if none
    int fu = -1, cnt_u = 0;
    auto ids_for = [&](int i) -> int {
        if (i >= nT) return -1;
        if (i < nAw) {
            const int t = a_lo + i;
            const int r = (t % a.tA) * TR + (lane & 15);
            return r < a.sinks ? r : (r < nsp ? a.clustered_end + (r - a.sinks) : -1);
        }
        const int t = b_lo + i - nAw;
        const int u = t / a.tB;
        const int j = (t % a.tB) * TR + (lane & 15);
        int tok;
        if (u != fu) {
            // first tile of unit u in this warp: wait for its selection
            bool ok = true;
            if (lane == 0) {
                ok = ld_acquire(a.flag + u) != 0;
                if (!ok) {
                    const long long t0 = clock64();
                    while (!(ok = ld_acquire(a.flag + u) != 0) && clock64() - t0 < a.wait_limit) __nanosleep(32);
                }
            }
            ok = __shfl_sync(FULL, ok, 0) != 0;
            __syncwarp();
            int c = ok ? __ldcg(a.count + u) : 0;
            tok = j < a.B ? __ldcg(a.idx + (size_t)u * a.B + j) : -1;  // loaded with the count
            if (!ok && lane == 0) set_err(a.dev_err, CKV_DEV_TIMEOUT);
            if (c < 0 || c > a.B) {
                if (lane == 0) set_err(a.dev_err, CKV_DEV_BAD_COUNT);
                c = c < 0 ? 0 : a.B;
            }
            cnt_u = c;
            fu = u;
        } else {
            tok = j < cnt_u ? __ldcg(a.idx + (size_t)u * a.B + j) : -1;
        }
        if (j >= cnt_u) return -1;
        if (tok < 0 || tok >= a.cur_len) {
            set_err(a.dev_err, CKV_DEV_BAD_INDEX);
            tok = -1;
        }
        return tok;
    };
    auto valid_bits = [&](int ids) -> unsigned { return __ballot_sync(FULL, ids >= 0) & 0xffffu; };
    const int sub = lane >> 4, li = lane & 15;
    auto issue = [&](int st, int i, int ids) {
        if (i < nT) {
            const int u = unit_of(i);
            const __nv_bfloat16* Ku = a.K + (size_t)u * a.max_len * D + li * 8;
            const __nv_bfloat16* Vu = a.V + (size_t)u * a.max_len * D + li * 8;
            unsigned char* dst = wbase + st * STAGE_BYTES + li * 16;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = 2 * j + sub;
                int tok = __shfl_sync(FULL, ids, r);
                tok = tok >= 0 ? tok : 0;  // a missing row copies token 0 (masked)
                ptx::cp_async16(dst + r * PITCH, Ku + (size_t)tok * D);
                ptx::cp_async16(dst + TILE_BYTES + r * PITCH, Vu + (size_t)tok * D);
            }
        }
        ptx::cp_async_commit();
    };

    uint32_t qa[8][2];
    float o[8][4];
    float mrun = -INFINITY, lrun = 0.f;
    const int qh = lane >> 2;
    auto reset = [&](int u) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            if (qh < G) {
                const uint32_t* qp =
                    reinterpret_cast<const uint32_t*>(a.q + ((size_t)u * G + qh) * D + 16 * ks) + (lane & 3);
                qa[ks][0] = qp[0];
                qa[ks][1] = qp[4];
            } else {
                qa[ks][0] = 0u;
                qa[ks][1] = 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
        mrun = -INFINITY;
        lrun = 0.f;
    };
    // partial slot of (unit u, phase ph) for this warp: the phase-A warps of u
    // first, then its phase-B warps, each in warp order
    auto flush = [&](int u, int ph) {
        int slot;
        const int wa0 = a.tA > 0 ? (u * a.tA) / a.apw : 0;
        if (ph == 0) {
            slot = aw - wa0;
        } else {
            const int na = a.tA > 0 ? (u * a.tA + a.tA - 1) / a.apw - wa0 + 1 : 0;
            slot = na + aw - (u * a.tB) / a.bpw;
        }
        float lt = lrun;
        lt += __shfl_xor_sync(FULL, lt, 1);
        lt += __shfl_xor_sync(FULL, lt, 2);
        float* pp = a.part + ((size_t)u * a.max_slots + slot) * PW;
        if ((lane & 3) == 0 && qh < G) {
            pp[qh * (D + 2) + D] = mrun;
            pp[qh * (D + 2) + D + 1] = lt;
        }
        const int h0 = (lane & 3) * 2;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int c = 16 * mt + qh;
            if (h0 < G) {
                pp[h0 * (D + 2) + c] = o[mt][0];
                pp[h0 * (D + 2) + c + 8] = o[mt][2];
            }
            if (h0 + 1 < G) {
                pp[(h0 + 1) * (D + 2) + c] = o[mt][1];
                pp[(h0 + 1) * (D + 2) + c + 8] = o[mt][3];
            }
        }
    };

    // ---- prologue: the first NST tiles in flight, ids of the next one ready
    unsigned vb[NST];
#pragma unroll
    for (int j = 0; j < NST; ++j) {
        const int ids = ids_for(j);
        vb[j] = valid_bits(ids);
        issue(j, j, ids);
    }
    int ids_pend = ids_for(NST);
    int cur_u = unit_of(0), cur_ph = nAw > 0 ? 0 : 1;
    reset(cur_u);

    for (int i = 0; i < nT; ++i) {
        const int st = i % NST;
        const int ids_next = ids_for(i + NST + 1);  // in flight during this tile
        ptx::cp_async_wait_group<NST - 1>();
        __syncwarp();
        const unsigned valid = vb[0];
        const int u = unit_of(i), ph = i < nAw ? 0 : 1;
        if (u != cur_u || ph != cur_ph) {
            flush(cur_u, cur_ph);
            cur_u = u;
            cur_ph = ph;
            reset(u);
        }
        const uint32_t kb = wbase_addr + (uint32_t)(st * STAGE_BYTES);
        const uint32_t vbs = kb + (uint32_t)TILE_BYTES;
        if (valid) {
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int chunk = 4 * kk + (lane >> 3);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int row = nt * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + (uint32_t)(row * PITCH + chunk * 16), b0, b1, b2, b3);
                    mma(s[nt], qa[2 * kk][0], 0u, qa[2 * kk][1], 0u, b0, b1);
                    mma(s[nt], qa[2 * kk + 1][0], 0u, qa[2 * kk + 1][1], 0u, b2, b3);
                }
            }
            float v[4];
            const int r0 = (lane & 3) * 2;
            v[0] = ((valid >> r0) & 1u) ? s[0][0] * a.qscale : -INFINITY;
            v[1] = ((valid >> (r0 + 1)) & 1u) ? s[0][1] * a.qscale : -INFINITY;
            v[2] = ((valid >> (r0 + 8)) & 1u) ? s[1][0] * a.qscale : -INFINITY;
            v[3] = ((valid >> (r0 + 9)) & 1u) ? s[1][1] * a.qscale : -INFINITY;
            float tm = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
            tm = fmaxf(tm, __shfl_xor_sync(FULL, tm, 1));
            tm = fmaxf(tm, __shfl_xor_sync(FULL, tm, 2));
            const float mnew = fmaxf(mrun, tm);
            const float msub = (mnew == -INFINITY) ? 0.f : mnew;
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = ex2(v[e] - msub);
            const bool grew = mnew != mrun;
            const float sc = grew ? ex2(mrun - msub) : 1.f;
            lrun = lrun * sc + ((p[0] + p[1]) + (p[2] + p[3]));
            mrun = mnew;
            const uint32_t bh0 = pack2(p[0], p[1]), bh1 = pack2(p[2], p[3]);
            const uint32_t bl0 = pack2(p[0] - lo_of(bh0), p[1] - hi_of(bh0));
            const uint32_t bl1 = pack2(p[2] - lo_of(bh1), p[3] - hi_of(bh1));
            if (__any_sync(FULL, grew)) {
                const float sc0 = __shfl_sync(FULL, sc, ((lane & 3) * 2) * 4);
                const float sc1 = __shfl_sync(FULL, sc, ((lane & 3) * 2 + 1) * 4);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    o[mt][0] *= sc0;
                    o[mt][1] *= sc1;
                    o[mt][2] *= sc0;
                    o[mt][3] *= sc1;
                }
            }
            const int vrow = ((lane >> 3) >> 1) * 8 + (lane & 7);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int chunk = 2 * mt + ((lane >> 3) & 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vbs + (uint32_t)(vrow * PITCH + chunk * 16), a0, a1, a2, a3);
                mma(o[mt], a0, a1, a2, a3, bh0, bh1);
                mma(o[mt], a0, a1, a2, a3, bl0, bl1);
            }
        }
        __syncwarp();
        issue(st, i + NST, ids_pend);
#pragma unroll
        for (int j = 0; j + 1 < NST; ++j) vb[j] = vb[j + 1];
        vb[NST - 1] = valid_bits(ids_pend);
        ids_pend = ids_next;
    }
    ptx::cp_async_wait_all();
    flush(cur_u, cur_ph);
}

// One CTA per unit, one thread per output (head, channel): merge the unit's
// partials (phase-A warps, then phase-B warps, each in warp order) into
//   o_h = sum_w acc_w 2^(m_w - M) / sum_w l_w 2^(m_w - M),  M = max_w m_w,
// and clear the unit's ready flag for the next step.
constexpr int SC_MAX_SLOTS = 20;

template <int G>
__global__ void __launch_bounds__(G * D) step_combine_kernel(const float* __restrict__ part, int tA, int apw, int tB,
                                                             int bpw, int max_slots, float* __restrict__ out,
                                                             int32_t* __restrict__ flag) {
    constexpr int PW = G * (D + 2);
    const int u = blockIdx.x, tid = threadIdx.x;
    const int na = tA > 0 ? (u * tA + tA - 1) / apw - (u * tA) / apw + 1 : 0;
    const int nb = (u * tB + tB - 1) / bpw - (u * tB) / bpw + 1;
    const int ns = na + nb;
    const float* pu = part + (size_t)u * max_slots * PW;
    const int h = tid / D, c = tid % D;
    float mv[SC_MAX_SLOTS], lv[SC_MAX_SLOTS], av[SC_MAX_SLOTS];
#pragma unroll
    for (int t = 0; t < SC_MAX_SLOTS; ++t)
        if (t < ns) {
            const float* sp = pu + (size_t)t * PW + h * (D + 2);
            mv[t] = sp[D];
            lv[t] = sp[D + 1];
            av[t] = sp[c];
        }
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < SC_MAX_SLOTS; ++t)
        if (t < ns) M = fmaxf(M, mv[t]);
    float l = 0.f, acc = 0.f;
#pragma unroll
    for (int t = 0; t < SC_MAX_SLOTS; ++t)
        if (t < ns) {
            const float f = (mv[t] == -INFINITY) ? 0.f : exp2f(mv[t] - M);
            l += lv[t] * f;
            acc += av[t] * f;
        }
    out[((size_t)u * G + h) * D + c] = l > 0.f ? acc / l : 0.f;
    if (tid == 0) flag[u] = 0;
}

template <int G>
cudaError_t launch_step_t(const StepArgs& a, int grid, cudaStream_t s, float* out) {
    auto kern = step_kernel<G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)STEP_SMEM);
    if (e != cudaSuccess) return e;
    if ((e = launch_dependent(kern, dim3(grid), dim3(NW * 32), STEP_SMEM, s, a)) != cudaSuccess) return e;
    step_combine_kernel<G><<<a.units, G * D, 0, s>>>(a.part, a.tA, a.apw, a.tB, a.bpw, a.max_slots, out, a.flag);
    return cudaGetLastError();
}

// tiles per warp of a phase (tpu tiles per unit, tot in all) over `warps`
// warps: an even share, at least one, and at least tpu / 8 so that a unit's
// tiles of one phase are spread over at most 9 warps (the combine merges at
// most 18 partials per unit in registers)
int per_warp(int tpu, int tot, int warps) {
    int w = tot > 0 ? (tot + warps - 1) / warps : 1;
    const int floor8 = (tpu + 7) / 8;
    return w > floor8 ? w : (floor8 > 0 ? floor8 : 1);
}

}  // namespace

bool step_supported(int kv_dtype, int g, int C, int units, int num_sms) {
    (void)g;
    return kv_dtype == CKV_BF16 && C >= 1 && C <= SEL_CMAX && units <= SW * (num_sms > 0 ? num_sms : 152);
}

cudaError_t launch_step(const ckv_ctx* ctx, const void* q, const void* K, const void* V, int C, int B, int cur_len,
                        int32_t* idx, int32_t* count, float* out, long long wait_limit, cudaStream_t s) {
    StepArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.K = static_cast<const __nv_bfloat16*>(K);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.scores = ctx->scores;
    a.sizes = ctx->sizes;
    a.offsets = ctx->offsets;
    a.perm = ctx->perm;
    a.idx = idx;
    a.count = count;
    a.flag = ctx->sel_flag;
    a.units = ctx->cfg.units;
    a.C = C;
    a.cmax = ctx->cmax;
    a.ntok = ctx->ntok;
    a.B = B;
    a.max_len = ctx->cfg.max_len;
    a.sinks = ctx->cfg.sinks;
    a.clustered_end = ctx->clustered_end;
    a.cur_len = cur_len;
    const int grid = ctx->num_sms > 0 ? ctx->num_sms : 152;
    a.tA = (a.sinks + (cur_len - a.clustered_end) + TR - 1) / TR;
    a.tB = (B + TR - 1) / TR;
    if (a.tB < 1) a.tB = 1;  // B = 0: one empty tile per unit keeps the slot arithmetic uniform
    a.apw = per_warp(a.tA, a.units * a.tA, grid * AW);
    a.bpw = per_warp(a.tB, a.units * a.tB, grid * AW);
    a.max_slots = ctx->max_splits;
    a.qscale = 1.4426950408889634f / sqrtf((float)D);
    a.wait_limit = wait_limit;
    a.stall = ctx->stall;
    a.part = ctx->attn_part;
    a.dev_err = ctx->dev_err;
    // every unit's partials must fit its slots and the combine's register merge
    const int na = a.tA > 0 ? (a.tA + a.apw - 1) / a.apw + 1 : 0;
    const int nb = (a.tB + a.bpw - 1) / a.bpw + 1;
    if (na + nb > a.max_slots || na + nb > SC_MAX_SLOTS) return cudaErrorInvalidValue;
    switch (ctx->cfg.g) {
        case 1: return launch_step_t<1>(a, grid, s, out);
        case 2: return launch_step_t<2>(a, grid, s, out);
        case 4: return launch_step_t<4>(a, grid, s, out);
        case 8: return launch_step_t<8>(a, grid, s, out);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ckv
