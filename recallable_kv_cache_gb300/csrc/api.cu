// C ABI of the ClusterKV decode path: argument validation, the context that
// owns the cluster state, and the order of kernel launches per call.  All
// validation happens on the host before anything is launched.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include "internal.h"

namespace ckv {
size_t assign_tc_smem(int cpad, int* stages_out);
}  // namespace ckv

using namespace ckv;

namespace {

constexpr int32_t VERSION = 100;  // 0.1.0
constexpr int MAX_INCR_M = 400;   // keys of one incremental clustering kept in smem

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ckv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CKV_OK : CKV_ERR_CUDA; }

template <typename T>
cudaError_t alloc(T** p, size_t count) {
    *p = nullptr;
    if (count == 0) count = 1;
    return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
}

void free_all(ckv_ctx* c) {
    void* ptrs[] = {c->mu32,   c->mu_s == c->mu32 ? nullptr : c->mu_s, c->mu_hat, c->sizes,
                    c->offsets, c->perm, c->labels, c->chunk_cnt, c->task_off, c->task_cl,
                    c->seg_part, c->scores, c->attn_part, c->dev_err, c->assign_best};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    if (c->pend_done) cudaEventDestroy(c->pend_done);
}

// turns the persisting set-aside off and puts back the limit found before
cudaError_t l2_release(ckv_ctx* ctx) {
    if (!ctx->l2_saved) return cudaSuccess;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaCtxResetPersistingL2Cache();
    if (e == cudaSuccess) e = cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, ctx->l2_prev_limit);
    ctx->l2_on = 0;
    ctx->l2_saved = 0;
    return e;
}

ckv_status check_kv(const ckv_ctx* ctx, const void* K) {
    if (!ctx || !K) return CKV_ERR_ARG;
    if (!aligned16(K)) return CKV_ERR_ALIGN;
    return CKV_OK;
}

ckv_status check_L(const ckv_ctx* ctx, int32_t L) {
    if (L <= ctx->cfg.sinks || L > ctx->cfg.max_len) return CKV_ERR_ARG;
    return CKV_OK;
}

}  // namespace

extern "C" {

const char* ckv_status_str(int32_t status) {
    switch (status) {
        case CKV_OK: return "CKV_OK";
        case CKV_ERR_ARG: return "CKV_ERR_ARG: bad argument";
        case CKV_ERR_DTYPE: return "CKV_ERR_DTYPE: unsupported or mismatched dtype";
        case CKV_ERR_CAPACITY: return "CKV_ERR_CAPACITY: exceeds a capacity fixed at ckv_create";
        case CKV_ERR_CUDA: return "CKV_ERR_CUDA: a CUDA runtime call failed";
        case CKV_ERR_TIMEOUT: return "CKV_ERR_TIMEOUT: a bounded device wait gave up";
        case CKV_ERR_DEVICE_CHECK: return "CKV_ERR_DEVICE_CHECK: a device-side check failed";
        case CKV_ERR_UNIMPLEMENTED: return "CKV_ERR_UNIMPLEMENTED: configuration not supported";
        case CKV_ERR_ALIGN: return "CKV_ERR_ALIGN: pointer not 16-byte aligned";
        case CKV_ERR_STATE: return "CKV_ERR_STATE: call out of order";
        default: return "unknown ckv_status";
    }
}

int32_t ckv_version(void) { return VERSION; }

ckv_status ckv_create(const ckv_config* cfg, ckv_ctx** out) {
    CKV_TRACE("ckv_create");
    if (!out) return CKV_ERR_ARG;
    *out = nullptr;
    if (!cfg) return CKV_ERR_ARG;
    if (cfg->d != D) return CKV_ERR_ARG;
    if (cfg->g != 1 && cfg->g != 2 && cfg->g != 4 && cfg->g != 8) return CKV_ERR_ARG;
    if (cfg->kv_dtype != CKV_F32 && cfg->kv_dtype != CKV_BF16) return CKV_ERR_DTYPE;
    if (cfg->units < 1 || cfg->sinks < 0 || cfg->ratio < 1 || cfg->m < 1 || cfg->c_plus < 1 ||
        cfg->c_plus > 16 || cfg->iters < 1 || cfg->max_len <= cfg->sinks || cfg->max_clusters < 1 ||
        cfg->max_budget < 1)
        return CKV_ERR_ARG;

    ckv_ctx* c = new (std::nothrow) ckv_ctx;
    if (!c) return CKV_ERR_CUDA;
    memset(c, 0, sizeof(*c));
    c->cfg = *cfg;
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        delete c;
        return CKV_ERR_CUDA;
    }
    const size_t U = (size_t)cfg->units;
    c->cmax = cfg->max_clusters;
    c->cmax_pad = round_up(cfg->max_clusters, 32);
    c->ntok = cfg->max_len - cfg->sinks;
    c->nchunk = ceil_div(c->ntok, CSR_CHUNK);
    c->max_tasks = ceil_div(c->ntok, SEG_ROWS) + c->cmax;
    c->attn_rows = cfg->sinks + cfg->max_budget + 2 * cfg->m;
    c->max_splits = ceil_div(c->attn_rows, attention_rows_per_split(cfg->kv_dtype, cfg->g));
    c->wait_limit = WAIT_LIMIT;
    c->stall = 0;
    c->elem = cfg->kv_dtype == CKV_BF16 ? 2 : 4;
    c->last_stream = nullptr;
    c->pend_m = 0;
    c->pend_c_plus = 0;
    c->pend_done = nullptr;

    const size_t cd = (size_t)c->cmax * D;
    bool ok = alloc(&c->mu32, U * cd) == cudaSuccess;
    if (cfg->kv_dtype == CKV_BF16) {
        ok = ok && cudaMalloc(&c->mu_s, U * cd * 2) == cudaSuccess;
        ok = ok && cudaMalloc(&c->mu_hat, U * (size_t)c->cmax_pad * D * 2) == cudaSuccess;
    } else {
        c->mu_s = c->mu32;
        ok = ok && cudaMalloc(&c->mu_hat, U * (size_t)c->cmax_pad * D * 4) == cudaSuccess;
    }
    ok = ok && alloc(&c->sizes, U * c->cmax) == cudaSuccess;
    ok = ok && alloc(&c->offsets, U * (c->cmax + 1)) == cudaSuccess;
    ok = ok && alloc(&c->perm, U * c->ntok) == cudaSuccess;
    ok = ok && alloc(&c->labels, U * c->ntok) == cudaSuccess;
    ok = ok && alloc(&c->chunk_cnt, U * c->nchunk * c->cmax) == cudaSuccess;
    ok = ok && alloc(&c->task_off, U * (c->cmax + 1)) == cudaSuccess;
    ok = ok && alloc(&c->task_cl, U * c->max_tasks) == cudaSuccess;
    ok = ok && alloc(&c->seg_part, U * c->max_tasks * D) == cudaSuccess;
    ok = ok && alloc(&c->scores, U * c->cmax) == cudaSuccess;
    ok = ok && alloc(&c->attn_part, U * c->max_splits * cfg->g * (D + 2)) == cudaSuccess;
    ok = ok && alloc(&c->dev_err, 1) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&c->pend_done, cudaEventDisableTiming) == cudaSuccess;
    if (cfg->kv_dtype == CKV_BF16 && c->cmax_pad > MAX_ASSIGN_CPAD)
        ok = ok && alloc(&c->assign_best, U * c->ntok) == cudaSuccess;
    if (ok) {
        const size_t hat = U * (size_t)c->cmax_pad * D * c->elem;
        ok = cudaMemset(c->mu_hat, 0, hat) == cudaSuccess &&
             cudaMemset(c->dev_err, 0, 4) == cudaSuccess && cudaMemset(c->sizes, 0, U * c->cmax * 4) == cudaSuccess &&
             cudaDeviceSynchronize() == cudaSuccess;
    }
    if (!ok) {
        free_all(c);
        delete c;
        cudaGetLastError();
        return CKV_ERR_CUDA;
    }
    *out = c;
    return CKV_OK;
}

ckv_status ckv_destroy(ckv_ctx* ctx) {
    CKV_TRACE("ckv_destroy");
    if (!ctx) return CKV_ERR_ARG;
    cudaDeviceSynchronize();
    l2_release(ctx);
    free_all(ctx);
    delete ctx;
    return CKV_OK;
}

ckv_status ckv_cluster_prefill(ckv_ctx* ctx, const void* K, int32_t L, int32_t n_clusters, void* stream) {
    CKV_TRACE("ckv_cluster_prefill");
    ckv_status st = check_kv(ctx, K);
    if (st != CKV_OK) return st;
    if ((st = check_L(ctx, L)) != CKV_OK) return st;
    const int n = L - ctx->cfg.sinks;
    int C = n_clusters > 0 ? n_clusters : n / ctx->cfg.ratio;
    if (C < 1) C = 1;
    if (n_clusters < 0 || C > n) return CKV_ERR_ARG;
    if (C > ctx->cmax) return CKV_ERR_CAPACITY;
    if (ctx->cfg.kv_dtype == CKV_BF16 && assign_tc_smem(round_up(C, 32), nullptr) > 232448)
        return CKV_ERR_UNIMPLEMENTED;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    int stride = n / C;
    if (stride > ctx->cfg.ratio) stride = ctx->cfg.ratio;
    if (stride < 1) stride = 1;
    cudaError_t e = launch_seed(ctx, K, C, stride, s);
    for (int it = 0; it < ctx->cfg.iters && e == cudaSuccess; ++it) {
        e = launch_assign(ctx, K, n, C, ctx->labels, s);
        if (e == cudaSuccess) e = launch_update(ctx, K, n, C, ctx->labels, s);
    }
    if (e != cudaSuccess) return CKV_ERR_CUDA;
    ctx->n_clusters = C;
    ctx->prefill_clusters = C;
    ctx->prefill_len = L;
    ctx->clustered_end = L;
    return CKV_OK;
}

ckv_status ckv_cluster_incremental(ckv_ctx* ctx, const void* K, int32_t start, int32_t m, int32_t c_plus,
                                   void* stream) {
    CKV_TRACE("ckv_cluster_incremental");
    ckv_status st = check_kv(ctx, K);
    if (st != CKV_OK) return st;
    if (ctx->pend_m > 0) return CKV_ERR_STATE;
    if (ctx->n_clusters <= 0 || start != ctx->clustered_end) return CKV_ERR_STATE;
    if (c_plus < 1 || c_plus > 16 || m < c_plus || m > MAX_INCR_M || start + m > ctx->cfg.max_len)
        return CKV_ERR_ARG;
    if (ctx->n_clusters + c_plus > ctx->cmax) return CKV_ERR_CAPACITY;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    const int csr_base = ctx->clustered_end - ctx->cfg.sinks;
    cudaError_t e = launch_incremental(ctx, K, start, m, c_plus, ctx->n_clusters, csr_base, s);
    if (e != cudaSuccess) return CKV_ERR_CUDA;
    ctx->n_clusters += c_plus;
    ctx->clustered_end += m;
    return CKV_OK;
}

ckv_status ckv_cluster_incremental_begin(ckv_ctx* ctx, const void* K, int32_t start, int32_t m, int32_t c_plus,
                                         void* stream) {
    CKV_TRACE("ckv_cluster_incremental_begin");
    ckv_status st = check_kv(ctx, K);
    if (st != CKV_OK) return st;
    if (ctx->pend_m > 0) return CKV_ERR_STATE;
    if (ctx->n_clusters <= 0 || start != ctx->clustered_end) return CKV_ERR_STATE;
    if (c_plus < 1 || c_plus > 16 || m < c_plus || m > MAX_INCR_M || start + m > ctx->cfg.max_len)
        return CKV_ERR_ARG;
    if (ctx->n_clusters + c_plus > ctx->cmax) return CKV_ERR_CAPACITY;
    cudaStream_t s = (cudaStream_t)stream;
    // the new clusters go to slots [n_clusters, n_clusters + c_plus) and the
    // perm segment after the clustered tokens: nothing the decode calls read
    // until the commit advances the counters
    const int csr_base = ctx->clustered_end - ctx->cfg.sinks;
    cudaError_t e = launch_incremental(ctx, K, start, m, c_plus, ctx->n_clusters, csr_base, s);
    if (e == cudaSuccess) e = cudaEventRecord(ctx->pend_done, s);
    if (e != cudaSuccess) return CKV_ERR_CUDA;
    ctx->pend_m = m;
    ctx->pend_c_plus = c_plus;
    return CKV_OK;
}

ckv_status ckv_cluster_incremental_commit(ckv_ctx* ctx, void* stream) {
    CKV_TRACE("ckv_cluster_incremental_commit");
    if (!ctx) return CKV_ERR_ARG;
    if (ctx->pend_m <= 0) return CKV_ERR_STATE;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamWaitEvent(s, ctx->pend_done, 0) != cudaSuccess) return CKV_ERR_CUDA;
    ctx->last_stream = s;
    ctx->n_clusters += ctx->pend_c_plus;
    ctx->clustered_end += ctx->pend_m;
    ctx->pend_m = 0;
    ctx->pend_c_plus = 0;
    return CKV_OK;
}

ckv_status ckv_kmeans_assign(ckv_ctx* ctx, const void* K, int32_t L, int32_t* labels, void* stream) {
    CKV_TRACE("ckv_kmeans_assign");
    ckv_status st = check_kv(ctx, K);
    if (st != CKV_OK) return st;
    if ((st = check_L(ctx, L)) != CKV_OK) return st;
    if (!labels) return CKV_ERR_ARG;
    if (ctx->n_clusters <= 0) return CKV_ERR_STATE;
    if (ctx->cfg.kv_dtype == CKV_BF16 && assign_tc_smem(round_up(ctx->n_clusters, 32), nullptr) > 232448)
        return CKV_ERR_UNIMPLEMENTED;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    return cuda_status(launch_assign(ctx, K, L - ctx->cfg.sinks, ctx->n_clusters, labels, s));
}

ckv_status ckv_kmeans_update(ckv_ctx* ctx, const void* K, int32_t L, const int32_t* labels, void* stream) {
    CKV_TRACE("ckv_kmeans_update");
    ckv_status st = check_kv(ctx, K);
    if (st != CKV_OK) return st;
    if ((st = check_L(ctx, L)) != CKV_OK) return st;
    if (!labels) return CKV_ERR_ARG;
    if (ctx->n_clusters <= 0) return CKV_ERR_STATE;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    cudaError_t e = launch_update(ctx, K, L - ctx->cfg.sinks, ctx->n_clusters, labels, s);
    if (e != cudaSuccess) return CKV_ERR_CUDA;
    ctx->prefill_clusters = ctx->n_clusters;
    ctx->prefill_len = L;
    ctx->clustered_end = L;
    return CKV_OK;
}

ckv_status ckv_score(ckv_ctx* ctx, const void* q, int32_t q_dtype, float* scores, void* stream) {
    CKV_TRACE("ckv_score");
    if (!ctx || !q || !scores) return CKV_ERR_ARG;
    if (q_dtype != ctx->cfg.kv_dtype) return CKV_ERR_DTYPE;
    if (!aligned16(q)) return CKV_ERR_ALIGN;
    if (ctx->n_clusters <= 0) return CKV_ERR_STATE;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    return cuda_status(launch_score(ctx, q, ctx->n_clusters, scores, ctx->n_clusters, s));
}

ckv_status ckv_select_scored(ckv_ctx* ctx, const float* scores, int32_t B, int32_t* idx, int32_t* count,
                             void* stream) {
    CKV_TRACE("ckv_select_scored");
    if (!ctx || !scores || !idx || !count) return CKV_ERR_ARG;
    if (B < 0) return CKV_ERR_ARG;
    if (B > ctx->cfg.max_budget) return CKV_ERR_CAPACITY;
    if (ctx->n_clusters <= 0 || ctx->clustered_end <= ctx->cfg.sinks) return CKV_ERR_STATE;
    if (ctx->n_clusters > MAX_SELECT_CLUSTERS) return CKV_ERR_UNIMPLEMENTED;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    return cuda_status(launch_select(ctx, nullptr, scores, ctx->n_clusters, ctx->n_clusters, B, idx, count, s));
}

ckv_status ckv_select(ckv_ctx* ctx, const void* q, int32_t q_dtype, int32_t B, int32_t* idx, int32_t* count,
                      void* stream) {
    CKV_TRACE("ckv_select");
    if (!ctx || !q || !idx || !count) return CKV_ERR_ARG;
    if (q_dtype != ctx->cfg.kv_dtype) return CKV_ERR_DTYPE;
    if (!aligned16(q)) return CKV_ERR_ALIGN;
    if (B < 0) return CKV_ERR_ARG;
    if (B > ctx->cfg.max_budget) return CKV_ERR_CAPACITY;
    if (ctx->n_clusters <= 0 || ctx->clustered_end <= ctx->cfg.sinks) return CKV_ERR_STATE;
    if (ctx->n_clusters > MAX_SELECT_CLUSTERS) return CKV_ERR_UNIMPLEMENTED;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    return cuda_status(launch_select(ctx, q, nullptr, 0, ctx->n_clusters, B, idx, count, s));
}

ckv_status ckv_sparse_decode_attn(ckv_ctx* ctx, const void* q, int32_t q_dtype, const void* K, const void* V,
                                  const int32_t* idx, const int32_t* count, int32_t B, int32_t cur_len, float* out,
                                  void* stream) {
    CKV_TRACE("ckv_sparse_decode_attn");
    if (!ctx || !q || !K || !V || !idx || !count || !out) return CKV_ERR_ARG;
    if (q_dtype != ctx->cfg.kv_dtype) return CKV_ERR_DTYPE;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return CKV_ERR_ALIGN;
    if (ctx->clustered_end <= ctx->cfg.sinks) return CKV_ERR_STATE;
    if (B < 0) return CKV_ERR_ARG;
    if (B > ctx->cfg.max_budget) return CKV_ERR_CAPACITY;
    if (cur_len < ctx->clustered_end || cur_len > ctx->cfg.max_len) return CKV_ERR_ARG;
    if (cur_len - ctx->clustered_end > 2 * ctx->cfg.m) return CKV_ERR_CAPACITY;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    cudaError_t e = launch_attention(q, K, V, idx, count, ctx->cfg.units, ctx->cfg.g, ctx->cfg.kv_dtype,
                                     ctx->cfg.max_len, ctx->cfg.sinks, ctx->clustered_end, cur_len, B, out,
                                     ctx->attn_part, ctx->max_splits, ctx->dev_err, ctx->num_sms,
                                     ctx->wait_limit, ctx->stall, s);
    return cuda_status(e);
}

ckv_status ckv_decode_step(ckv_ctx* ctx, const void* q, int32_t q_dtype, const void* K, const void* V, int32_t B,
                           int32_t cur_len, int32_t* idx, int32_t* count, float* out, void* stream) {
    CKV_TRACE("ckv_decode_step");
    if (!ctx || !q || !K || !V || !idx || !count || !out) return CKV_ERR_ARG;
    if (q_dtype != ctx->cfg.kv_dtype) return CKV_ERR_DTYPE;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return CKV_ERR_ALIGN;
    if (ctx->n_clusters <= 0 || ctx->clustered_end <= ctx->cfg.sinks) return CKV_ERR_STATE;
    if (B < 0) return CKV_ERR_ARG;
    if (B > ctx->cfg.max_budget) return CKV_ERR_CAPACITY;
    if (cur_len < ctx->clustered_end || cur_len > ctx->cfg.max_len) return CKV_ERR_ARG;
    if (cur_len - ctx->clustered_end > 2 * ctx->cfg.m) return CKV_ERR_CAPACITY;
    if (ctx->n_clusters > MAX_SELECT_CLUSTERS) return CKV_ERR_UNIMPLEMENTED;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    // selection, then attention (a dependent launch: it is scheduled while the
    // selection drains and waits for it on the device)
    cudaError_t e = launch_select(ctx, q, nullptr, 0, ctx->n_clusters, B, idx, count, s);
    if (e == cudaSuccess)
        e = launch_attention(q, K, V, idx, count, ctx->cfg.units, ctx->cfg.g, ctx->cfg.kv_dtype, ctx->cfg.max_len,
                             ctx->cfg.sinks, ctx->clustered_end, cur_len, B, out, ctx->attn_part,
                             ctx->max_splits, ctx->dev_err, ctx->num_sms, ctx->wait_limit, ctx->stall, s);
    return cuda_status(e);
}

ckv_status ckv_get_info(ckv_ctx* ctx, ckv_info* info) {
    CKV_TRACE("ckv_get_info");
    if (!ctx || !info) return CKV_ERR_ARG;
    info->n_clusters = ctx->n_clusters;
    info->prefill_clusters = ctx->prefill_clusters;
    info->prefill_len = ctx->prefill_len;
    info->clustered_end = ctx->clustered_end;
    return CKV_OK;
}

ckv_status ckv_export_clusters(ckv_ctx* ctx, float* mu, void* mu_hat, int32_t* sizes, int32_t* offsets,
                               int32_t* perm, void* stream) {
    CKV_TRACE("ckv_export_clusters");
    if (!ctx) return CKV_ERR_ARG;
    const int C = ctx->n_clusters;
    if (C <= 0) return CKV_ERR_STATE;
    const size_t U = (size_t)ctx->cfg.units;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    cudaError_t e = cudaSuccess;
    if (mu && e == cudaSuccess)
        e = cudaMemcpy2DAsync(mu, (size_t)C * D * 4, ctx->mu32, (size_t)ctx->cmax * D * 4, (size_t)C * D * 4, U,
                              cudaMemcpyDeviceToDevice, s);
    if (mu_hat && e == cudaSuccess)
        e = cudaMemcpy2DAsync(mu_hat, (size_t)C * D * ctx->elem, ctx->mu_hat, (size_t)ctx->cmax_pad * D * ctx->elem,
                              (size_t)C * D * ctx->elem, U, cudaMemcpyDeviceToDevice, s);
    if (sizes && e == cudaSuccess)
        e = cudaMemcpy2DAsync(sizes, (size_t)C * 4, ctx->sizes, (size_t)ctx->cmax * 4, (size_t)C * 4, U,
                              cudaMemcpyDeviceToDevice, s);
    if (offsets && e == cudaSuccess)
        e = cudaMemcpy2DAsync(offsets, (size_t)(C + 1) * 4, ctx->offsets, (size_t)(ctx->cmax + 1) * 4,
                              (size_t)(C + 1) * 4, U, cudaMemcpyDeviceToDevice, s);
    const int np = ctx->clustered_end - ctx->cfg.sinks;
    if (perm && np > 0 && e == cudaSuccess)
        e = cudaMemcpy2DAsync(perm, (size_t)np * 4, ctx->perm, (size_t)ctx->ntok * 4, (size_t)np * 4, U,
                              cudaMemcpyDeviceToDevice, s);
    return cuda_status(e);
}

ckv_status ckv_import_clusters(ckv_ctx* ctx, int32_t n_clusters, int32_t clustered_end, const float* mu,
                               const int32_t* sizes, const int32_t* offsets, const int32_t* perm, void* stream) {
    CKV_TRACE("ckv_import_clusters");
    if (!ctx || !mu) return CKV_ERR_ARG;
    if (n_clusters < 1) return CKV_ERR_ARG;
    if (n_clusters > ctx->cmax) return CKV_ERR_CAPACITY;
    const bool csr = sizes || offsets || perm;
    if (csr && !(sizes && offsets && perm)) return CKV_ERR_ARG;
    if (csr && (clustered_end <= ctx->cfg.sinks || clustered_end > ctx->cfg.max_len)) return CKV_ERR_ARG;
    const size_t U = (size_t)ctx->cfg.units;
    const int C = n_clusters;
    cudaStream_t s = (cudaStream_t)stream;
    ctx->last_stream = s;
    cudaError_t e = cudaMemcpy2DAsync(ctx->mu32, (size_t)ctx->cmax * D * 4, mu, (size_t)C * D * 4,
                                      (size_t)C * D * 4, U, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = launch_shadows(ctx, 0, C, s);
    if (csr) {
        const int np = clustered_end - ctx->cfg.sinks;
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(ctx->sizes, (size_t)ctx->cmax * 4, sizes, (size_t)C * 4, (size_t)C * 4, U,
                                  cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(ctx->offsets, (size_t)(ctx->cmax + 1) * 4, offsets, (size_t)(C + 1) * 4,
                                  (size_t)(C + 1) * 4, U, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(ctx->perm, (size_t)ctx->ntok * 4, perm, (size_t)np * 4, (size_t)np * 4, U,
                                  cudaMemcpyDeviceToDevice, s);
    }
    if (e != cudaSuccess) return CKV_ERR_CUDA;
    ctx->n_clusters = C;
    ctx->prefill_clusters = C;
    if (csr) {
        ctx->clustered_end = clustered_end;
        ctx->prefill_len = clustered_end;
    }
    return CKV_OK;
}

ckv_status ckv_set_wait_limit(ckv_ctx* ctx, int64_t cycles, int32_t stall) {
    CKV_TRACE("ckv_set_wait_limit");
    if (!ctx) return CKV_ERR_ARG;
    if (cycles < 1 || cycles > MAX_WAIT_LIMIT || (stall != 0 && stall != 1)) return CKV_ERR_ARG;
    ctx->wait_limit = cycles;
    ctx->stall = stall;
    return CKV_OK;
}

ckv_status ckv_set_l2_persistence(ckv_ctx* ctx, int64_t bytes) {
    CKV_TRACE("ckv_set_l2_persistence");
    if (!ctx) return CKV_ERR_ARG;
    if (bytes == 0) return cuda_status(l2_release(ctx));
    int maxp = 0, maxw = 0;
    cudaError_t e = cudaDeviceGetAttribute(&maxp, cudaDevAttrMaxPersistingL2CacheSize, ctx->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&maxw, cudaDevAttrMaxAccessPolicyWindowSize, ctx->device);
    if (e != cudaSuccess || maxp <= 0 || maxw <= 0) return CKV_ERR_CUDA;
    const size_t U = (size_t)ctx->cfg.units;
    const size_t mu_bytes = U * ctx->cmax * D * ctx->elem;
    const size_t perm_bytes = U * ctx->ntok * sizeof(int32_t);
    // what the context needs: the centroid copy (a selection that scores its
    // own unit reads only it through its window), and only when all of it
    // fits: a partial set-aside keeps little of it and takes L2 from the
    // K-means passes
    if (bytes < 0 && mu_bytes > (size_t)maxp) return cuda_status(l2_release(ctx));
    size_t want = bytes < 0 ? mu_bytes : (size_t)bytes;
    if (want > (size_t)maxp) want = (size_t)maxp;
    if (!ctx->l2_saved) {
        if ((e = cudaDeviceGetLimit(&ctx->l2_prev_limit, cudaLimitPersistingL2CacheSize)) != cudaSuccess)
            return CKV_ERR_CUDA;
        ctx->l2_saved = 1;
    }
    if ((e = cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, want)) != cudaSuccess) return CKV_ERR_CUDA;
    size_t got = 0;
    if ((e = cudaDeviceGetLimit(&got, cudaLimitPersistingL2CacheSize)) != cudaSuccess) return CKV_ERR_CUDA;
    // the centroid copy first (every step reads all of it), perm from what is
    // left (a step reads ~B entries of each unit's perm): hit ratio = the part
    // of each window the set-aside can hold
    auto ratio = [](size_t have, size_t n) {
        return have >= n ? 1.0f : (float)((double)have / (double)n);
    };
    const size_t left = got > mu_bytes ? got - mu_bytes : 0;
    auto window = [&](void* base, size_t n, float hit) {
        cudaAccessPolicyWindow w = {};
        w.base_ptr = base;
        w.num_bytes = n < (size_t)maxw ? n : (size_t)maxw;
        w.hitRatio = hit;
        w.hitProp = cudaAccessPropertyPersisting;
        w.missProp = cudaAccessPropertyStreaming;
        return w;
    };
    ctx->l2_mu = window(ctx->mu_s, mu_bytes, ratio(got, mu_bytes));
    ctx->l2_perm = window(ctx->perm, perm_bytes, ratio(left, perm_bytes));
    ctx->l2_on = 1;
    return CKV_OK;
}

ckv_status ckv_get_device_error(ckv_ctx* ctx, int32_t* code) {
    CKV_TRACE("ckv_get_device_error");
    if (!ctx || !code) return CKV_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(ctx->last_stream);
    int32_t v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, ctx->dev_err, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(ctx->dev_err, 0, 4);
    if (e != cudaSuccess) return CKV_ERR_CUDA;
    *code = v;
    return CKV_OK;
}

}  // extern "C"
