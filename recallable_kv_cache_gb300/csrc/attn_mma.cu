// Sparse decode attention over bf16 K/V on the tensor cores (ClusterKV page,
// section "Background": softmax(q K_S^T / sqrt(d)) V_S over the selected
// tokens; here S = sinks + pending tokens + the selected clusters' tokens).
//
// The work is HBM-bound: every attended K and V row (256 bytes each) is read
// once for all g query heads.  The arithmetic per row (g dot products of 128
// channels and g axpys) is mapped on mma.sync m16n8k16 so that the issue slots
// stay free for the gather:
//   S^T[h][r] = q[h] . K[r]   M = 16 (the g heads, zero-padded), N = 8 rows,
//                             K = 16 channels; A = q from registers, B = K rows
//                             from shared memory (ldmatrix);
//   O^T[c][h] += V[r][c] P[h][r]  M = 16 channels, N = 8 heads, K = 16 rows;
//                             A = V rows (ldmatrix.trans), B = P taken straight
//                             from the S^T accumulators.
// bf16 x bf16 products are exact and accumulate in fp32.  P = exp2(s - m) is
// fed to the second product as two bf16 terms (P = hi + lo) so the weights
// keep about 16 significant bits.
//
// Work split: the attended set of each unit is cut into tiles of 16 rows;
// every warp owns a contiguous range of tiles (persistent grid, one CTA of 12
// warps per SM).  Each warp runs its own 2-stage shared-memory ring: 16-byte
// cp.async copies (one commit group per tile) fill a stage while the warp
// computes an earlier one, token ids are resolved NST + 1 tiles ahead, and rows
// sit at a 272-byte pitch so that ldmatrix is free of bank conflicts.  The warp keeps an online softmax (max, sum,
// O^T) per unit and writes one partial per (unit, warp) when it leaves a
// unit.  attn_mma_combine_kernel merges the partials of each unit in warp
// order (deterministic, no atomics).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "mma_sync.cuh"
#include "ptx.cuh"

namespace ckv {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int MW = 12;  // warps per CTA
constexpr int TR = 16;  // rows per tile

using namespace mmas;

struct MmaArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    const int32_t* idx;
    const int32_t* count;
    int max_len, sinks, clustered_end, cur_len, B;
    int tpu;    // tiles per unit
    int tpw;    // tiles per warp
    int total;  // units * tpu
    int max_slots;
    float qscale;  // log2(e) / sqrt(d)
    float* part;
    int32_t* dev_err;
};

constexpr int NST = 2;                       // ring stages per warp
constexpr int PITCH = D * 2 + 16;             // 272-byte row pitch: conflict-free ldmatrix
constexpr int TILE_BYTES = TR * PITCH;        // one 16-row K (or V) tile
constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K then V
constexpr size_t MMA_SMEM = (size_t)MW * NST * STAGE_BYTES;

template <int G>
__global__ void __launch_bounds__(MW * 32, 1) attn_mma_kernel(const MmaArgs a) {
    constexpr int PW = G * (D + 2);
    extern __shared__ __align__(128) unsigned char mma_smem[];
    ptx::grid_dependency_wait();  // idx and count come from the selection kernel
    ptx::allow_dependent_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * MW + warp;
    const int t_begin = gw * a.tpw;
    const int t_end = min(a.total, t_begin + a.tpw);
    if (t_begin >= t_end) return;
    unsigned char* wbase = mma_smem + (size_t)warp * NST * STAGE_BYTES;
    const uint32_t wbase_addr = ptx::smem_u32(wbase);
    const int pend = a.cur_len - a.clustered_end;

    // ---- token of row (lane & 15) of tile t, -1 if none (count cached per unit).
    // The idx entry is loaded before the count is known (any slot below B is
    // a valid address) so that both loads share one round trip; rows at or
    // past the count are discarded afterwards.
    int cu_ids = -1, r_ids = 0;
    auto ids_for = [&](int t) -> int {
        if (t >= t_end) return -1;
        const int u = t / a.tpu, k = t % a.tpu;
        const int r = k * TR + (lane & 15);
        const int j = r - a.sinks - pend;
        int tok;
        if (r < a.sinks) tok = r;
        else if (j < 0) tok = a.clustered_end + (r - a.sinks);
        else tok = j < a.B ? a.idx[(size_t)u * a.B + j] : -1;
        if (u != cu_ids) {
            int c = a.count[u];
            if (c < 0 || c > a.B) {
                if (lane == 0 && a.dev_err) atomicCAS(a.dev_err, 0, CKV_DEV_BAD_COUNT);
                c = c < 0 ? 0 : a.B;
            }
            r_ids = a.sinks + pend + c;
            cu_ids = u;
        }
        if (r >= r_ids) return -1;
        if (tok < 0 || tok >= a.cur_len) {
            if (a.dev_err) atomicCAS(a.dev_err, 0, CKV_DEV_BAD_INDEX);
            tok = -1;
        }
        return tok;
    };
    auto valid_bits = [&](int ids) -> unsigned { return __ballot_sync(FULL, ids >= 0) & 0xffffu; };
    // 16-byte asynchronous copies of the 16 K rows and 16 V rows of tile t
    // into stage st (lane l: chunk l % 16 of rows 2i + l / 16); a missing row
    // copies token 0 (a sink, always present) so the stage holds finite values,
    // and is masked later; one commit group per tile (empty past the range)
    const int sub = lane >> 4, li = lane & 15;
    auto issue = [&](int st, int t, int ids) {
        if (t < t_end) {
            const int u = t / a.tpu;
            const __nv_bfloat16* Ku = a.K + (size_t)u * a.max_len * D + li * 8;
            const __nv_bfloat16* Vu = a.V + (size_t)u * a.max_len * D + li * 8;
            unsigned char* dst = wbase + st * STAGE_BYTES + li * 16;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = 2 * j + sub;
                int tok = __shfl_sync(FULL, ids, r);
                tok = tok >= 0 ? tok : 0;
                ptx::cp_async16(dst + r * PITCH, Ku + (size_t)tok * D);
                ptx::cp_async16(dst + TILE_BYTES + r * PITCH, Vu + (size_t)tok * D);
            }
        }
        ptx::cp_async_commit();
    };

    // ---- per-unit state (S^T layout: head = lane / 4; O^T accumulators:
    // channel 16 mt + lane / 4 (+8), heads 2 (lane % 4) and 2 (lane % 4) + 1)
    uint32_t qa[8][2];
    float o[8][4];
    float mrun = -INFINITY, lrun = 0.f;
    int cur_u = -1;
    const int qh = lane >> 2;

    auto reset = [&](int u) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            if (qh < G) {
                const uint32_t* qp = reinterpret_cast<const uint32_t*>(a.q + ((size_t)u * G + qh) * D + 16 * ks) + (lane & 3);
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

    auto flush = [&](int u) {
        float lt = lrun;
        lt += __shfl_xor_sync(FULL, lt, 1);
        lt += __shfl_xor_sync(FULL, lt, 2);
        const int w0 = (u * a.tpu) / a.tpw;
        float* pp = a.part + ((size_t)u * a.max_slots + (gw - w0)) * PW;
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
    unsigned vb[NST];  // valid-row bits of the tiles in the ring, oldest first
#pragma unroll
    for (int j = 0; j < NST; ++j) {
        const int ids = ids_for(t_begin + j);
        vb[j] = valid_bits(ids);
        issue(j, t_begin + j, ids);  // tiles past t_end have no rows: empty groups
    }
    int ids_pend = ids_for(t_begin + NST);
    // the first unit's query while the first tiles are in flight
    cur_u = t_begin / a.tpu;
    reset(cur_u);

    for (int i = 0, t = t_begin; t < t_end; ++i, ++t) {
        const int st = i % NST;
        const int ids_next = ids_for(t + NST + 1);  // in flight during this tile
        ptx::cp_async_wait_group<NST - 1>();  // this lane's copies of tile t have landed
        __syncwarp();                          // ... and every other lane's
        const unsigned valid = vb[0];
        const int u = t / a.tpu;
        if (u != cur_u) {
            if (cur_u >= 0) flush(cur_u);
            cur_u = u;
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
            // -inf - -inf is avoided: ex2(-inf) = 0 covers masked rows
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
            // rescale the O^T columns only when some head's running max moved
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
        // the stage is free again: tile t + NST into it (an empty group past the end)
        issue(st, t + NST, ids_pend);
#pragma unroll
        for (int j = 0; j + 1 < NST; ++j) vb[j] = vb[j + 1];
        vb[NST - 1] = valid_bits(ids_pend);
        ids_pend = ids_next;
    }
    ptx::cp_async_wait_all();
    if (cur_u >= 0) flush(cur_u);
}

// One CTA per unit, one thread per output (head, channel): merge the unit's
// per-warp partials (in warp order) into
//   o_h = sum_w acc_w 2^(m_w - M) / sum_w l_w 2^(m_w - M),  M = max_w m_w.
// The warps that hold partials of unit u are those whose tile ranges meet u's
// tiles: (u*tpu)/tpw .. (u*tpu + tpu - 1)/tpw.  The per-slot weights are
// computed once into shared memory; the accumulator loads of all slots are
// independent, so they are in flight together.
constexpr int CMB_MAX_SLOTS = 256;
constexpr int CMB_REG_SLOTS = 12;  // units with at most this many partials merge in registers
// dynamic shared memory of a combine CTA: with the attention CTA's 209 KB it
// exceeds an SM's 228 KB
constexpr int CMB_BLOCK_SMEM = 64 * 1024;

template <int G>
__global__ void __launch_bounds__(G * D) attn_mma_combine_kernel(const float* __restrict__ part, int tpu, int tpw,
                                                                 int max_slots, float* __restrict__ out) {
    constexpr int PW = G * (D + 2);
    __shared__ float wt[CMB_MAX_SLOTS][G];
    __shared__ float lw[CMB_MAX_SLOTS][G];
    __shared__ float Ls[G];
    const int u = blockIdx.x, tid = threadIdx.x;
    ptx::grid_dependency_wait();  // the partials come from the attention kernel
    const int w0 = (u * tpu) / tpw, w1 = (u * tpu + tpu - 1) / tpw;
    const int ns = min(w1 - w0 + 1, CMB_MAX_SLOTS);
    const float* pu = part + (size_t)u * max_slots * PW;
    if (ns <= CMB_REG_SLOTS) {
        // the usual case: each thread loads its head's (max, sum) of every slot
        // with its own accumulator entries in one round trip and merges them in
        // registers (the same operations in the same order as below)
        const int h = tid / D, c = tid % D;
        float mv[CMB_REG_SLOTS], lv[CMB_REG_SLOTS], av[CMB_REG_SLOTS];
#pragma unroll
        for (int t = 0; t < CMB_REG_SLOTS; ++t)
            if (t < ns) {
                const float* sp = pu + (size_t)t * PW + h * (D + 2);
                mv[t] = sp[D];
                lv[t] = sp[D + 1];
                av[t] = sp[c];
            }
        float M = -INFINITY;
#pragma unroll
        for (int t = 0; t < CMB_REG_SLOTS; ++t)
            if (t < ns) M = fmaxf(M, mv[t]);
        float l = 0.f, acc = 0.f;
#pragma unroll
        for (int t = 0; t < CMB_REG_SLOTS; ++t)
            if (t < ns) {
                const float f = (mv[t] == -INFINITY) ? 0.f : exp2f(mv[t] - M);
                l += lv[t] * f;
                acc += av[t] * f;
            }
        out[((size_t)u * G + h) * D + c] = l > 0.f ? acc / l : 0.f;
        return;
    }
    // every slot's (max, sum) pair at once; the serial part below reads smem only
    for (int e = tid; e < ns * G; e += G * D) {
        const float* ms = pu + (size_t)(e / G) * PW + (e % G) * (D + 2) + D;
        wt[e / G][e % G] = ms[0];
        lw[e / G][e % G] = ms[1];
    }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int t = 0; t < ns; ++t) M = fmaxf(M, wt[t][tid]);
        float l = 0.f;
        for (int t = 0; t < ns; ++t) {
            const float f = (wt[t][tid] == -INFINITY) ? 0.f : exp2f(wt[t][tid] - M);
            l += lw[t][tid] * f;
            wt[t][tid] = f;
        }
        Ls[tid] = l;
    }
    __syncthreads();
    const int h = tid / D, c = tid % D;
    const float* src = pu + h * (D + 2) + c;
    float acc = 0.f;
    int t = 0;
    for (; t + 8 <= ns; t += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = src[(size_t)(t + j) * PW];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc += v[j] * wt[t + j][h];
    }
    for (; t < ns; ++t) acc += src[(size_t)t * PW] * wt[t][h];
    out[((size_t)u * G + h) * D + c] = Ls[h] > 0.f ? acc / Ls[h] : 0.f;
}

template <int G>
cudaError_t launch_mma_t(const void* q, const void* K, const void* V, const int32_t* idx, const int32_t* count,
                         int units, int max_len, int sinks, int clustered_end, int cur_len, int B, float* out,
                         float* part, int max_slots, int32_t* dev_err, int num_sms, cudaStream_t st) {
    MmaArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.K = static_cast<const __nv_bfloat16*>(K);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.idx = idx;
    a.count = count;
    a.max_len = max_len;
    a.sinks = sinks;
    a.clustered_end = clustered_end;
    a.cur_len = cur_len;
    a.B = B;
    a.tpu = (sinks + (cur_len - clustered_end) + B + TR - 1) / TR;
    if (a.tpu < 1) a.tpu = 1;
    if (a.tpu > max_slots) return cudaErrorInvalidValue;
    a.total = a.tpu * units;
    const int sms = num_sms > 0 ? num_sms : 152;
    const int warps = sms * MW;
    a.tpw = (a.total + warps - 1) / warps;
    if (a.tpw * (CMB_MAX_SLOTS - 1) < a.tpu) a.tpw = (a.tpu + CMB_MAX_SLOTS - 2) / (CMB_MAX_SLOTS - 1);
    const int grid = (a.total + a.tpw * MW - 1) / (a.tpw * MW);
    a.max_slots = max_slots;
    a.qscale = 1.4426950408889634f / sqrtf((float)D);
    a.part = part;
    a.dev_err = dev_err;
    const size_t smem = MMA_SMEM;
    auto kern = attn_mma_kernel<G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if ((e = launch_dependent(kern, dim3(grid), dim3(MW * 32), smem, st, a)) != cudaSuccess) return e;
    // the combine is a dependent launch too, so its CTAs are resident as soon
    // as SMs free up; its (unused) dynamic shared memory keeps it off any SM
    // that still holds an attention CTA, whose warps it would slow
    auto ck = attn_mma_combine_kernel<G>;
    if ((e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, CMB_BLOCK_SMEM)) != cudaSuccess)
        return e;
    return launch_dependent(ck, dim3(units), dim3(G * D), (size_t)CMB_BLOCK_SMEM, st, (const float*)part, a.tpu,
                            a.tpw, max_slots, out);
}

}  // namespace

int attention_mma_rows_per_tile() { return TR; }

cudaError_t launch_attention_mma(const void* q, const void* K, const void* V, const int32_t* idx,
                                 const int32_t* count, int units, int g, int max_len, int sinks, int clustered_end,
                                 int cur_len, int B, float* out, float* part, int max_slots, int32_t* dev_err,
                                 int num_sms, cudaStream_t s) {
#define CKV_MMA(G)                                                                                            \
    return launch_mma_t<G>(q, K, V, idx, count, units, max_len, sinks, clustered_end, cur_len, B, out, part, \
                           max_slots, dev_err, num_sms, s)
    switch (g) {
        case 1: CKV_MMA(1);
        case 2: CKV_MMA(2);
        case 4: CKV_MMA(4);
        case 8: CKV_MMA(8);
    }
#undef CKV_MMA
    return cudaErrorInvalidValue;
}

}  // namespace ckv
