// K-means assignment on the fifth-generation tensor cores (ClusterKV page,
// section "Clustering in semantic space", clustering process: every key joins
// the centroid of largest cosine similarity; section "Semantic clustering
// optimisation": the assignment is a batched keys x centroids product followed
// by an arg-max).
//
// cos(k, mu_c) = (k . mu_hat_c) / ||k|| and ||k|| > 0 is the same for every c,
// so the arg-max over c of k . mu_hat_c is the cosine arg-max: the key
// normalisation is folded away and the raw bf16 keys feed the MMA directly.
//
// One persistent CTA per SM walks a contiguous range of 128-token tiles
// (flattened over units).  The unit's centroid directions stay resident in
// shared memory while its tiles stream by; when there are too many of them
// (more than 640 rows), they are split into passes of at most 512 rows: the
// CTA walks its tiles of the unit once per pass, and the running maximum of a
// token and its column are kept in global memory between passes (a later pass
// wins only with a strictly larger dot, so ties still go to the lower index).
// Warp roles:
//   warp 0     TMA producer: the pass's rows of mu_hat [<= 640 x 128] once per
//              (unit, pass), key tiles [128 x 128] through a ring;
//   warp 1     TMEM owner and MMA issuer: per tile and per column chunk of at
//              most 256 centroids, 8 x tcgen05.mma (K = 16 each) into one of
//              two 256-column TMEM slots;
//   warps 2-17 epilogue: tcgen05.ld of the fp32 dots (one TMEM lane = one
//              token; four warps per lane quarter split the 32-column groups),
//              running arg-max in increasing centroid order with a strict '>'
//              (ties keep the lower index), merge of the four, label store.
// All mbarrier waits are bounded; a timeout sets the device error word and
// every role leaves its loop.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace ckv {
namespace {

constexpr int A_STAGE_BYTES = ASSIGN_TILE * D * 2;  // 32 KB: two 64-column panels
constexpr int A_PANEL_BYTES = ASSIGN_TILE * 128;    // 16 KB
constexpr int B_BOX_ROWS = 32;
constexpr int EPI_PER_Q = 4;                    // epilogue warps per TMEM lane quarter
constexpr int EPI_WARPS = 4 * EPI_PER_Q;
constexpr int THREADS = 64 + 32 * EPI_WARPS;     // producer, MMA issuer, epilogue warps
constexpr int GROUPS_PER_WARP = 8 / EPI_PER_Q;   // 32-column groups of a 256-column chunk

struct AssignArgs {
    int n;              // clustered tokens per unit
    int C;              // centroids
    int cpad;           // C rounded up to 32
    int pw;             // centroid rows per pass (multiple of 32)
    int npass;          // passes over a unit's tiles: ceil(cpad / pw)
    int tiles_per_unit;
    int total_tiles;
    int tiles_per_cta;
    int sinks;
    int stages;
    int32_t* labels;
    float* best;        // [units][n] running maxima between passes (npass > 1)
    int32_t* dev_err;
    long long wait_limit;  // SM cycles before a wait gives up
    int stall;          // failure detection test: the MMA issuer first waits on a barrier nothing completes
};

struct __align__(8) Bars {
    uint64_t a_full[4];
    uint64_t a_empty[4];
    uint64_t b_full;
    uint64_t b_empty;
    uint64_t tm_full[2];
    uint64_t tm_empty[2];
    uint64_t part_full[4];   // per TMEM lane quarter: the other warps' partials written
    uint64_t part_free[4];   // ... and consumed
    float xbest[4][EPI_PER_Q - 1][32];
    int xarg[4][EPI_PER_Q - 1][32];
    uint64_t never;          // no thread or copy ever arrives (failure detection test)
    uint64_t drain;          // completion of every MMA the issuer started, after an abort
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* bs,
                                              int32_t* dev_err, long long limit) {
    if (ptx::mbar_wait(bar, parity, limit, &bs->abort)) return true;
    if (atomicExch(&bs->abort, 1) == 0 && dev_err) atomicCAS(dev_err, 0, CKV_DEV_TIMEOUT);
    return false;
}

__global__ void __launch_bounds__(THREADS, 1)
    assign_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmMu,
                     const AssignArgs p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char* A = smem;                                     // stages x 32 KB
    unsigned char* Bm = smem + (size_t)p.stages * A_STAGE_BYTES;  // 2 panels x pw x 128 B
    Bars* bs = reinterpret_cast<Bars*>(Bm + (size_t)p.pw * 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t_begin = blockIdx.x * p.tiles_per_cta;
    const int t_end = min(p.total_tiles, t_begin + p.tiles_per_cta);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            ptx::mbar_init(&bs->a_full[s], 1);
            ptx::mbar_init(&bs->a_empty[s], 1);
        }
        ptx::mbar_init(&bs->b_full, 1);
        ptx::mbar_init(&bs->b_empty, 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&bs->tm_full[s], 1);
            ptx::mbar_init(&bs->tm_empty[s], EPI_WARPS);
        }
        for (int qq = 0; qq < 4; ++qq) {
            ptx::mbar_init(&bs->part_full[qq], EPI_PER_Q - 1);
            ptx::mbar_init(&bs->part_free[qq], 1);
        }
        ptx::mbar_init(&bs->never, 1);
        ptx::mbar_init(&bs->drain, 1);
        bs->abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&bs->tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bs->tmem_base;

    int p_loads = 0, p_bloads = 0;  // copies the producer issued (for the drain after an abort)
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tmK);
            ptx::prefetch_tmap(&tmMu);
            int b_loads = 0, it = 0;
            bool alive = true;
            for (int t0 = t_begin; t0 < t_end && alive;) {
                const int u = t0 / p.tiles_per_unit;
                const int t1 = min(t_end, (u + 1) * p.tiles_per_unit);
                for (int ps = 0; ps < p.npass && alive; ++ps) {
                    const int prow = ps * p.pw;
                    const int rows = min(p.pw, p.cpad - prow);
                    if (b_loads > 0 && !wait_or_abort(&bs->b_empty, (b_loads - 1) & 1, bs, p.dev_err, p.wait_limit)) {
                        alive = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&bs->b_full, (uint32_t)rows * 256u);
                    for (int pn = 0; pn < 2; ++pn)
                        for (int r0 = 0; r0 < rows; r0 += B_BOX_ROWS)
                            ptx::tma_load_3d(Bm + (size_t)pn * p.pw * 128 + (size_t)r0 * 128, &tmMu, pn * 64,
                                             prow + r0, u, &bs->b_full);
                    ++b_loads;
                    for (int t = t0; t < t1; ++t, ++it) {
                        const int s = it % p.stages;
                        if (it >= p.stages &&
                            !wait_or_abort(&bs->a_empty[s], ((it / p.stages) - 1) & 1, bs, p.dev_err, p.wait_limit)) {
                            alive = false;
                            break;
                        }
                        unsigned char* a = A + (size_t)s * A_STAGE_BYTES;
                        ptx::mbar_arrive_expect_tx(&bs->a_full[s], A_STAGE_BYTES);
                        const int row = p.sinks + (t - u * p.tiles_per_unit) * ASSIGN_TILE;
                        ptx::tma_load_3d(a, &tmK, 0, row, u, &bs->a_full[s]);
                        ptx::tma_load_3d(a + A_PANEL_BYTES, &tmK, 64, row, u, &bs->a_full[s]);
                    }
                }
                t0 = t1;
            }
            p_loads = it;
            p_bloads = b_loads;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t a_base = ptx::smem_u32(A);
            const uint32_t b_base = ptx::smem_u32(Bm);
            int b_loads = 0, it = 0, item = 0;
            bool alive = true;
            if (p.stall && !wait_or_abort(&bs->never, 0, bs, p.dev_err, p.wait_limit)) alive = false;
            for (int t0 = t_begin; t0 < t_end && alive;) {
                const int u = t0 / p.tiles_per_unit;
                const int t1 = min(t_end, (u + 1) * p.tiles_per_unit);
                for (int ps = 0; ps < p.npass && alive; ++ps) {
                    const int rows = min(p.pw, p.cpad - ps * p.pw);
                    const int nch = (rows + 255) >> 8;
                    // the previous pass's centroid rows may be overwritten once
                    // every MMA issued so far has completed
                    if (b_loads > 0) ptx::mma_commit(&bs->b_empty);
                    if (!wait_or_abort(&bs->b_full, b_loads & 1, bs, p.dev_err, p.wait_limit)) {
                        alive = false;
                        break;
                    }
                    ++b_loads;
                    for (int t = t0; t < t1 && alive; ++t, ++it) {
                        const int s = it % p.stages;
                        if (!wait_or_abort(&bs->a_full[s], (it / p.stages) & 1, bs, p.dev_err, p.wait_limit)) {
                            alive = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t a_st = a_base + (uint32_t)s * A_STAGE_BYTES;
                        for (int ch = 0; ch < nch; ++ch, ++item) {
                            const int slot = item & 1;
                            if (item >= 2 &&
                                !wait_or_abort(&bs->tm_empty[slot], ((item >> 1) - 1) & 1, bs, p.dev_err, p.wait_limit)) {
                                alive = false;
                                break;
                            }
                            ptx::tc_fence_after();
                            const int ncols = min(256, rows - 256 * ch);
                            const uint32_t idesc = ptx::idesc_bf16_f32(128, ncols);
                            const uint32_t d_tmem = tmem + (uint32_t)slot * 256u;
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const uint32_t koff = (uint32_t)(k & 3) * 32u;
                                const uint64_t ad =
                                    ptx::smem_desc_sw128(a_st + (uint32_t)(k >> 2) * A_PANEL_BYTES + koff);
                                const uint64_t bd = ptx::smem_desc_sw128(
                                    b_base + (uint32_t)(k >> 2) * (uint32_t)p.pw * 128u + (uint32_t)ch * 256u * 128u +
                                    koff);
                                ptx::mma_bf16(d_tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
                            }
                            ptx::mma_commit(&bs->tm_full[slot]);
                        }
                        ptx::mma_commit(&bs->a_empty[s]);
                    }
                }
                t0 = t1;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // EPI_PER_Q warps per TMEM lane quarter (warp % 4); warp `sub` of a
        // quarter takes the 32-column groups sub, sub + EPI_PER_Q, ... of every
        // chunk and issues all its TMEM loads of a chunk before one wait.  Per
        // row the partial arg-maxes are merged through shared memory by the
        // quarter's first warp; ties keep the lower column.
        const int q = warp & 3;
        const int sub = (warp - 2) >> 2;  // rank among the quarter's epilogue warps
        int item = 0, ntile = 0;
        bool alive = true;
        for (int t0 = t_begin; t0 < t_end && alive;) {
            const int u = t0 / p.tiles_per_unit;
            const int t1 = min(t_end, (u + 1) * p.tiles_per_unit);
            for (int ps = 0; ps < p.npass && alive; ++ps) {
                const int prow = ps * p.pw;
                const int rows = min(p.pw, p.cpad - prow);
                const int nch = (rows + 255) >> 8;
                for (int t = t0; t < t1; ++t, ++ntile) {
                    const int tl = t - u * p.tiles_per_unit;
                    // four independent running maxima (columns j mod 4) break the
                    // compare-select dependency chain; merged below
                    float bk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                    int ak[4] = {0, 0, 0, 0};
                    for (int ch = 0; ch < nch; ++ch, ++item) {
                        const int slot = item & 1;
                        const bool ok = __all_sync(
                            0xffffffffu, wait_or_abort(&bs->tm_full[slot], (item >> 1) & 1, bs, p.dev_err, p.wait_limit));
                        if (!ok) {
                            alive = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        // chunk columns [c0, c0 + ncols); rows is a multiple of 32 and
                        // cpad - C < 32, so every chunk holds at least one real column
                        const int c0 = prow + 256 * ch;
                        const int nvalid = min(min(256, rows - 256 * ch), p.C - c0);
                        const int ngroups = (nvalid + 31) >> 5;
                        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)slot * 256u;
                        uint32_t r[GROUPS_PER_WARP][32];
#pragma unroll
                        for (int k = 0; k < GROUPS_PER_WARP; ++k) {
                            const int g = EPI_PER_Q * k + sub;
                            if (g < ngroups) ptx::tmem_ld32(taddr + (uint32_t)(g * 32), r[k]);
                        }
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < GROUPS_PER_WARP; ++k) {
                            const int g = EPI_PER_Q * k + sub;
                            if (g >= ngroups) break;
                            const int lim = nvalid - g * 32;
                            const int cb = c0 + g * 32;
                            if (lim >= 32) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    const float v = __uint_as_float(r[k][j]);
                                    if (v > bk[j & 3]) {
                                        bk[j & 3] = v;
                                        ak[j & 3] = cb + j;
                                    }
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    const float v = __uint_as_float(r[k][j]);
                                    if (j < lim && v > bk[j & 3]) {
                                        bk[j & 3] = v;
                                        ak[j & 3] = cb + j;
                                    }
                                }
                            }
                        }
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(&bs->tm_empty[slot]);
                    }
                    if (!alive) break;
                    // each chain holds its first maximum; (larger value, then lower
                    // column) over chains and over the pair picks the row's first maximum
                    float best = bk[0];
                    int arg = ak[0];
#pragma unroll
                    for (int k = 1; k < 4; ++k)
                        if (bk[k] > best || (bk[k] == best && ak[k] < arg)) {
                            best = bk[k];
                            arg = ak[k];
                        }
                    if (sub > 0) {
                        if (ntile > 0 && !__all_sync(0xffffffffu, wait_or_abort(&bs->part_free[q], (ntile - 1) & 1,
                                                                                 bs, p.dev_err, p.wait_limit))) {
                            alive = false;
                            break;
                        }
                        bs->xbest[q][sub - 1][lane] = best;
                        bs->xarg[q][sub - 1][lane] = arg;
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(&bs->part_full[q]);
                    } else {
                        if (!__all_sync(0xffffffffu,
                                        wait_or_abort(&bs->part_full[q], ntile & 1, bs, p.dev_err, p.wait_limit))) {
                            alive = false;
                            break;
                        }
                        float ob[EPI_PER_Q - 1];
                        int oa[EPI_PER_Q - 1];
#pragma unroll
                        for (int w = 0; w < EPI_PER_Q - 1; ++w) {
                            ob[w] = bs->xbest[q][w][lane];
                            oa[w] = bs->xarg[q][w][lane];
                        }
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(&bs->part_free[q]);
#pragma unroll
                        for (int w = 0; w < EPI_PER_Q - 1; ++w)
                            if (ob[w] > best || (ob[w] == best && oa[w] < arg)) {
                                best = ob[w];
                                arg = oa[w];
                            }
                        const int row = tl * ASSIGN_TILE + q * 32 + lane;
                        if (row < p.n) {
                            const size_t o = (size_t)u * p.n + row;
                            // earlier passes hold lower columns: they keep ties.
                            // This thread wrote them itself (same tile row).
                            if (ps > 0) {
                                const float pb = p.best[o];
                                if (!(best > pb)) {
                                    best = pb;
                                    arg = p.labels[o];
                                }
                            }
                            p.labels[o] = arg;
                            if (ps + 1 < p.npass) p.best[o] = best;
                        }
                    }
                }
            }
            t0 = t1;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (bs->abort) {
        // a wait gave up, so some copies or MMAs may not have been consumed:
        // the producer waits (bounded) for the last phase of every stage and
        // of the centroid panel it armed, the MMA issuer for every MMA it
        // started, before the CTA's shared memory and TMEM are released
        if (warp == 0 && lane == 0) {
            for (int j = p_loads > p.stages ? p_loads - p.stages : 0; j < p_loads; ++j)
                if (!ptx::mbar_wait(&bs->a_full[j % p.stages], (j / p.stages) & 1, p.wait_limit, nullptr) && p.dev_err)
                    atomicCAS(p.dev_err, 0, CKV_DEV_TIMEOUT);
            if (p_bloads > 0 && !ptx::mbar_wait(&bs->b_full, (p_bloads - 1) & 1, p.wait_limit, nullptr) && p.dev_err)
                atomicCAS(p.dev_err, 0, CKV_DEV_TIMEOUT);
        }
        if (warp == 1 && lane == 0) {
            ptx::mma_commit(&bs->drain);
            if (!ptx::mbar_wait(&bs->drain, 0, p.wait_limit, nullptr) && p.dev_err) atomicCAS(p.dev_err, 0, CKV_DEV_TIMEOUT);
        }
    }
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3-D bf16 tensor [units][rows][128], box {64, box_rows, 1}, 128-byte swizzle.
bool encode_3d(CUtensorMap* m, const void* base, int rows, int units, int box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)units};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

// Centroid rows per pass: all of them up to MAX_ASSIGN_CPAD, else equal passes
// of at most 512 rows (which leaves room for three key stages).
void assign_tc_passes(int cpad, int* pw, int* npass) {
    int np = 1, w = cpad;
    if (cpad > MAX_ASSIGN_CPAD) {
        np = ceil_div(cpad, 512);
        w = round_up(ceil_div(cpad, np), 32);
    }
    *pw = w;
    *npass = np;
}

size_t assign_tc_smem(int cpad, int* stages_out) {
    int pw = 0, npass = 0;
    assign_tc_passes(cpad, &pw, &npass);
    const size_t fixed = (size_t)pw * 256 + sizeof(Bars) + 1024;
    const size_t cap = 232448;
    int stages = 4;
    while (stages > 2 && fixed + (size_t)stages * A_STAGE_BYTES > cap) --stages;
    if (stages_out) *stages_out = stages;
    return fixed + (size_t)stages * A_STAGE_BYTES;
}

cudaError_t launch_assign_tc(const ckv_ctx* ctx, const void* K, int n, int C, int32_t* labels,
                             cudaStream_t s) {
    const int cpad = round_up(C, 32);
    int stages = 0;
    const size_t smem = assign_tc_smem(cpad, &stages);
    if (smem > 232448 || cpad > ctx->cmax_pad) return cudaErrorInvalidValue;
    int pw = 0, npass = 0;
    assign_tc_passes(cpad, &pw, &npass);
    if (npass > 1 && !ctx->assign_best) return cudaErrorInvalidValue;
    CUtensorMap tmK, tmMu;
    if (!encode_3d(&tmK, K, ctx->cfg.max_len, ctx->cfg.units, ASSIGN_TILE)) return cudaErrorInvalidValue;
    if (!encode_3d(&tmMu, ctx->mu_hat, ctx->cmax_pad, ctx->cfg.units, B_BOX_ROWS))
        return cudaErrorInvalidValue;
    AssignArgs a;
    a.n = n;
    a.C = C;
    a.cpad = cpad;
    a.pw = pw;
    a.npass = npass;
    a.tiles_per_unit = ceil_div(n, ASSIGN_TILE);
    a.total_tiles = a.tiles_per_unit * ctx->cfg.units;
    const int grid = a.total_tiles < ctx->num_sms ? a.total_tiles : ctx->num_sms;
    a.tiles_per_cta = ceil_div(a.total_tiles, grid);
    const int used = ceil_div(a.total_tiles, a.tiles_per_cta);
    a.sinks = ctx->cfg.sinks;
    a.stages = stages;
    a.labels = labels;
    a.best = ctx->assign_best;
    a.dev_err = ctx->dev_err;
    a.wait_limit = ctx->wait_limit;
    a.stall = ctx->stall;
    cudaError_t e = cudaFuncSetAttribute(assign_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    assign_tc_kernel<<<used, THREADS, smem, s>>>(tmK, tmMu, a);
    return cudaGetLastError();
}

}  // namespace ckv
