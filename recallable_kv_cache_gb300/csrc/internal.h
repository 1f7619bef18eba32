// Internal declarations shared by the C-ABI layer and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ckv.h"

// NVTX range over one C-ABI call (header-only NVTX 3: without a profiler
// attached a push / pop costs a few nanoseconds)
#include <nvtx3/nvToolsExt.h>
struct CkvTraceRange {
    explicit CkvTraceRange(const char* name) { nvtxRangePushA(name); }
    ~CkvTraceRange() { nvtxRangePop(); }
    CkvTraceRange(const CkvTraceRange&) = delete;
    CkvTraceRange& operator=(const CkvTraceRange&) = delete;
};
#define CKV_TRACE(name) CkvTraceRange ckv_trace_range_(name)

namespace ckv {

constexpr int D = 128;             // head dimension the kernels support
constexpr int CSR_CHUNK = 1024;    // tokens per block in the CSR count/scatter passes
constexpr int SEG_ROWS = 64;       // rows per centroid-update task
constexpr int ASSIGN_TILE = 128;   // tokens per tcgen05 assignment tile (MMA M)
constexpr int MAX_ASSIGN_CPAD = 640;  // centroid rows the assignment keeps resident in smem
constexpr long long WAIT_LIMIT = 2000000000LL;  // SM cycles before a bounded wait gives up (default)
constexpr long long MAX_WAIT_LIMIT = 4000000000LL;  // largest limit ckv_set_wait_limit accepts
constexpr int QUEST_PAGE = 16;     // tokens per page of the page-granular comparator

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel of the stream is still running; it must call
// ptx::grid_dependency_wait() before touching memory that kernel writes.
template <typename... P, typename... A>
cudaError_t launch_dependent_win(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 const cudaAccessPolicyWindow* win, A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (win) {
        // accesses of this launch inside the window: hits persist in L2
        at[1].id = cudaLaunchAttributeAccessPolicyWindow;
        at[1].val.accessPolicyWindow = *win;
        cfg.numAttrs = 2;
    }
    cfg.attrs = at;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}
template <typename... P, typename... A>
cudaError_t launch_dependent(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A&&... args) {
    return launch_dependent_win(kern, grid, block, smem, s, nullptr, static_cast<A&&>(args)...);
}
inline int ceil_div(int x, int m) { return (x + m - 1) / m; }

}  // namespace ckv

struct ckv_ctx {
    ckv_config cfg;
    int device;
    int num_sms;
    int cmax;        // centroid capacity per unit
    int cmax_pad;    // rows of the assignment operand per unit (multiple of 16)
    int ntok;        // max_len - sinks: capacity of labels / perm per unit
    int nchunk;      // ceil(ntok / CSR_CHUNK)
    int max_tasks;   // centroid-update tasks per unit
    int max_splits;  // attention splits per unit
    int attn_rows;   // rows an attention call may cover per unit
    size_t elem;     // bytes per K/V element

    int n_clusters;
    int prefill_clusters;
    int prefill_len;
    int clustered_end;
    cudaStream_t last_stream;
    // an incremental clustering launched but not yet visible (begin / commit)
    int pend_c_plus, pend_m;
    cudaEvent_t pend_done;

    // state
    float* mu32;        // [U][cmax][D] centroids (fp32 master)
    void* mu_s;         // [U][cmax][D] scoring operand (bf16 copy, or == mu32 for f32)
    void* mu_hat;       // [U][cmax_pad][D] normalised directions (bf16 or f32)
    int32_t* sizes;     // [U][cmax]
    int32_t* offsets;   // [U][cmax + 1]
    int32_t* perm;      // [U][ntok]
    // workspace
    int32_t* labels;    // [U][ntok]
    int32_t* chunk_cnt; // [U][nchunk][cmax]
    int32_t* task_off;  // [U][cmax + 1]
    int32_t* task_cl;   // [U][max_tasks]
    float* seg_part;    // [U][max_tasks][D]
    float* scores;      // [U][cmax]
    float* attn_part;   // [U][max_splits][g * (D + 2)]
    int32_t* dev_err;   // device error word
    float* assign_best; // [U][ntok] running arg-max values between assignment passes (large C only)
    long long wait_limit; // SM cycles before a bounded device wait gives up
    int stall;            // failure detection test: kernels first wait on something nothing completes
    // L2 persistence (ckv_set_l2_persistence): windows for the scoring copy
    // and perm while l2_on; the context limit found before the first call
    int l2_on;
    int l2_saved;
    size_t l2_prev_limit;
    cudaAccessPolicyWindow l2_mu, l2_perm;
};

namespace ckv {

// centroid operand copies for centroids [c0, c1) of every unit
cudaError_t launch_shadows(const ckv_ctx* ctx, int c0, int c1, cudaStream_t s);
// mu[j] = K[sinks + base + j * stride], j in [0, C), then shadows
cudaError_t launch_seed(const ckv_ctx* ctx, const void* K, int C, int stride, cudaStream_t s);
// labels[u][i] = argmax_c cos(k_{sinks+i}, mu_c), i < n
cudaError_t launch_assign(const ckv_ctx* ctx, const void* K, int n, int C, int32_t* labels,
                          cudaStream_t s);
// CSR of labels over tokens [sinks, sinks+n) + centroid means + shadows
cudaError_t launch_update(const ckv_ctx* ctx, const void* K, int n, int C, const int32_t* labels,
                          cudaStream_t s);
// incremental clustering of [start, start+m) into c_plus clusters appended at C_old
cudaError_t launch_incremental(const ckv_ctx* ctx, const void* K, int start, int m, int c_plus,
                               int C_old, int csr_base, cudaStream_t s);
// scores[u][c] = sum_h q_h . mu_c, written with row stride `stride`
cudaError_t launch_score(const ckv_ctx* ctx, const void* q, int C, float* scores, int stride,
                         cudaStream_t s, bool prefetch_csr = false);
// selection for every unit: scores from q and the centroids (scores == null)
// or from caller-given scores [units][stride]
cudaError_t launch_select(const ckv_ctx* ctx, const void* q, const float* scores, int stride, int C, int B,
                          int32_t* idx, int32_t* count, cudaStream_t s);
constexpr int MAX_SELECT_CLUSTERS = 8192;
// split-K sparse decode attention; the partials are caller-provided scratch
// ([units][max_splits][g * (D + 2)] floats)
cudaError_t launch_attention(const void* q, const void* K, const void* V, const int32_t* idx,
                             const int32_t* count, int units, int g, int kv_dtype, int max_len,
                             int sinks, int clustered_end, int cur_len, int B, float* out,
                             float* part, int max_splits, int32_t* dev_err,
                             int num_sms, long long wait_limit, int stall, cudaStream_t s);
// rows of the attended set one attention work item covers (partials per unit
// are bounded by ceil(rows / this))
int attention_rows_per_split(int kv_dtype, int g);
int attention_mma_rows_per_tile();
cudaError_t launch_attention_mma(const void* q, const void* K, const void* V, const int32_t* idx,
                                 const int32_t* count, int units, int g, int max_len, int sinks, int clustered_end,
                                 int cur_len, int B, float* out, float* part, int max_slots, int32_t* dev_err,
                                 int num_sms, cudaStream_t s);

}  // namespace ckv
