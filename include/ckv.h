/*
 * ckv.h - C ABI of the GB300-native ClusterKV decode path.
 *
 * ClusterKV ("ClusterKV: Manipulating LLM KV Cache in Semantic Space for
 * Recallable Compression", arXiv 2412.03213) recalls KV-cache tokens at the
 * granularity of semantic clusters: the keys of each attention head are
 * grouped by cosine K-means, every decode step scores the cluster centroids
 * against the query, takes whole clusters in descending score order up to a
 * token budget B, and runs attention over the selected, non-contiguous K/V.
 *
 * Terms used below
 *   unit      one (sequence, layer, KV head); units are independent.
 *   d         head dimension; this library is built for d = 128.
 *   g         query heads sharing one KV head (GQA group), 1, 2, 4 or 8.
 *   sinks     leading tokens never clustered and always attended (16).
 *   L         prompt length; the prompt's clustered tokens are [sinks, L).
 *   clustered_end   end of the clustered token range: L after prefill, then
 *             +m after each incremental clustering.
 *   pending   tokens [clustered_end, cur_len): generated but not yet
 *             clustered; always attended.
 *
 * Buffers (all pointers are DEVICE pointers unless stated, 16-byte aligned,
 * row-contiguous, owned by the caller; the library never frees them).  A
 * device pointer is any address the kernels can access: device memory, or
 * pinned host memory the device maps (with unified addressing its host
 * address), for the small per-step inputs and outputs (q, out, the appended
 * K/V rows), which then cross the host link inside the kernels:
 *   K, V      [units][max_len][d] of kv_dtype.  Row t of unit u starts at
 *             element (u * max_len + t) * d.
 *   q         [units][g][d] of kv_dtype (q_dtype must equal kv_dtype).
 *   labels    [units][L - sinks] int32.
 *   scores    [units][n_clusters] float.
 *   idx       [units][B] int32; count [units] int32.
 *   out       [units][g][d] float.
 * The library owns the cluster state (centroids, sizes, prefix offsets, the
 * label-sorted token permutation) and a workspace, all allocated on the
 * device current at ckv_create and freed by ckv_destroy.
 *
 * Calls are asynchronous on the given stream (a cudaStream_t passed as
 * void*, NULL = legacy default stream).  Argument, dtype, alignment and
 * capacity errors are detected on the host before any launch and returned;
 * nothing is launched then.  Device-side checks (an index out of range) set
 * a device error word instead of trapping; ckv_get_device_error reads it.
 * Bounded device waits that give up report CKV_ERR_TIMEOUT the same way.
 * One context must not be used from two streams at the same time.
 */
#ifndef CKV_H
#define CKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ckv_ctx ckv_ctx;

typedef enum {
    CKV_OK = 0,
    CKV_ERR_ARG = -1,           /* bad argument (null, out of range, wrong shape) */
    CKV_ERR_DTYPE = -2,         /* unsupported or mismatched dtype */
    CKV_ERR_CAPACITY = -3,      /* exceeds a capacity fixed at ckv_create */
    CKV_ERR_CUDA = -4,          /* a CUDA runtime call failed */
    CKV_ERR_TIMEOUT = -5,       /* a bounded device wait gave up */
    CKV_ERR_DEVICE_CHECK = -6,  /* a device-side check failed (see ckv_get_device_error) */
    CKV_ERR_UNIMPLEMENTED = -7, /* configuration the library does not support */
    CKV_ERR_ALIGN = -8,         /* pointer not 16-byte aligned */
    CKV_ERR_STATE = -9          /* call out of order (e.g. select before clustering) */
} ckv_status;

typedef enum { CKV_F32 = 0, CKV_BF16 = 1 } ckv_dtype;

/* Device error word values (ckv_get_device_error). */
enum {
    CKV_DEV_OK = 0,
    CKV_DEV_TIMEOUT = 1,        /* an mbarrier wait ran past its iteration limit */
    CKV_DEV_BAD_INDEX = 2,      /* a selected token index outside [0, cur_len) */
    CKV_DEV_BAD_COUNT = 3,      /* a count outside [0, B] */
    CKV_DEV_BAD_LABEL = 4,      /* a label outside [0, n_clusters) (treated as 0) */
    CKV_DEV_BAD_CSR = 5         /* cluster offsets pointing outside the token permutation */
};

typedef struct {
    int32_t units;        /* independent (sequence, layer, KV head) triples, >= 1 */
    int32_t d;            /* head dimension; must be 128 */
    int32_t g;            /* query heads per KV head: 1, 2, 4 or 8 */
    int32_t sinks;        /* attention-sink tokens (ClusterKV: 16) */
    int32_t ratio;        /* prompt tokens per cluster (ClusterKV: 80) */
    int32_t m;            /* incremental clustering period (ClusterKV: 320) */
    int32_t c_plus;       /* clusters per incremental clustering (ClusterKV: 4) */
    int32_t iters;        /* Lloyd iterations per clustering (10) */
    int32_t max_len;      /* tokens per unit in the caller's K/V buffers */
    int32_t max_clusters; /* centroid capacity per unit (prefill + incremental) */
    int32_t max_budget;   /* largest B passed to ckv_select / ckv_sparse_decode_attn */
    int32_t kv_dtype;     /* ckv_dtype of K, V and q */
} ckv_config;

typedef struct {
    int32_t n_clusters;       /* clusters per unit now (prefill + incremental) */
    int32_t prefill_clusters; /* clusters made by the last ckv_cluster_prefill */
    int32_t prefill_len;      /* L of the last ckv_cluster_prefill */
    int32_t clustered_end;    /* end of the clustered token range */
} ckv_info;

/* Human-readable name of a ckv_status value (static string). */
const char* ckv_status_str(int32_t status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t ckv_version(void);

/* Validates cfg and allocates the cluster state and workspace on the current
 * device.  *out receives the context; on error *out is NULL and nothing stays
 * allocated.  Errors: CKV_ERR_ARG (null, d != 128, g not in {1,2,4,8},
 * sizes <= 0), CKV_ERR_DTYPE, CKV_ERR_CUDA (allocation failed). */
ckv_status ckv_create(const ckv_config* cfg, ckv_ctx** out);

/* Frees everything ckv_create allocated.  Synchronises the device first. */
ckv_status ckv_destroy(ckv_ctx* ctx);

/* Prefill clustering (ClusterKV page, section "Clustering in semantic space":
 * clustering process, Fig. 4, and clustering strategy during inference).
 * For every unit: keep tokens [0, sinks) as attention sinks; seed
 * n_clusters centroids with the keys at stride s = min(ratio, n / n_clusters)
 * of the n = L - sinks clustered keys; then run `iters` Lloyd iterations of
 * (assignment to the centroid of largest cosine similarity, ties to the
 * lower index) and (centroid = mean of the raw assigned keys, an empty
 * cluster keeping its centroid).  The final assignment becomes the cluster
 * metadata: sizes, prefix offsets and the token ids sorted by label (section
 * "Selection and indexing mechanism", Fig. 8).  Replaces any earlier state.
 * n_clusters = 0 selects (L - sinks) / ratio.
 * Errors: CKV_ERR_ARG (L <= sinks, L > max_len, n_clusters > L - sinks),
 * CKV_ERR_CAPACITY (n_clusters > max_clusters), CKV_ERR_ALIGN. */
ckv_status ckv_cluster_prefill(ckv_ctx* ctx, const void* K, int32_t L, int32_t n_clusters,
                               void* stream);

/* Incremental clustering (section "Clustering in semantic space": every m
 * decode steps the m newest keys are clustered among themselves into C+
 * clusters, never together with the prompt's keys).  Clusters the keys of
 * tokens [start, start + m) of every unit into c_plus new clusters with the
 * same seeding (stride min(ratio, m / c_plus)) and Lloyd iterations, and
 * appends their centroids and CSR segments after the existing ones.  start
 * must equal the current clustered_end, which then advances by m.
 * Errors: CKV_ERR_STATE (no prefill yet, start != clustered_end),
 * CKV_ERR_ARG (m < c_plus, start + m > max_len, m > 400, c_plus > 16),
 * CKV_ERR_CAPACITY (n_clusters + c_plus > max_clusters). */
ckv_status ckv_cluster_incremental(ckv_ctx* ctx, const void* K, int32_t start, int32_t m,
                                   int32_t c_plus, void* stream);

/* The same incremental clustering split in two, so that it can overlap decode
 * work (ClusterKV page, section "Semantic clustering optimisation", Fig. 6:
 * clustering runs asynchronously, overlapped with the model's other work).
 * _begin launches the clustering on `stream` (typically a side stream forked
 * from the decode stream) and writes the new centroids and perm segment where
 * no decode call reads them; until _commit, ckv_select, ckv_sparse_decode_attn
 * and ckv_decode_step keep using the previous clusters and treat the m tokens
 * as pending (attended in full).  _commit makes `stream` wait for the
 * clustering and then publishes it (n_clusters += c_plus, clustered_end +=
 * m).  Errors as for ckv_cluster_incremental; CKV_ERR_STATE for a second
 * _begin before _commit, a _commit with nothing begun, or
 * ckv_cluster_incremental while one is pending. */
ckv_status ckv_cluster_incremental_begin(ckv_ctx* ctx, const void* K, int32_t start, int32_t m,
                                         int32_t c_plus, void* stream);
ckv_status ckv_cluster_incremental_commit(ckv_ctx* ctx, void* stream);

/* One assignment step with the context's current n_clusters centroids:
 * labels[u][i] = argmax_c cos(k_{sinks+i}, mu_c) for i < L - sinks, ties to
 * the lower index (section "Clustering in semantic space", clustering
 * process).  The cosine is taken against the centroid direction rounded to
 * the operand type (bf16 for bf16 keys).  Does not change the state. */
ckv_status ckv_kmeans_assign(ckv_ctx* ctx, const void* K, int32_t L, int32_t* labels,
                             void* stream);

/* One update step from caller-given labels (same layout as above, each in
 * [0, n_clusters)): builds sizes, prefix offsets and the label-sorted token
 * permutation of tokens [sinks, L), and sets every centroid with a non-empty
 * cluster to the mean of its raw keys (section "Clustering in semantic
 * space", clustering process; section "Semantic clustering optimisation",
 * Fig. 7).  Sums are per cluster in a fixed order (deterministic, no float
 * atomics).  Sets clustered_end = L and prefill_len = L. */
ckv_status ckv_kmeans_update(ckv_ctx* ctx, const void* K, int32_t L, const int32_t* labels,
                             void* stream);

/* Centroid scores (section "Selection at semantic-cluster granularity"):
 * scores[u][c] = sum over the g query heads h of q_h . mu_c (inner product,
 * not cosine).  For bf16 the centroids are read as bf16; sums are fp32. */
ckv_status ckv_score(ckv_ctx* ctx, const void* q, int32_t q_dtype, float* scores, void* stream);

/* Selection and indexing from given scores (section "Selection and indexing
 * mechanism", Fig. 8): rank clusters by (score descending, index ascending),
 * prefix-sum their sizes in that order, take every cluster that starts before
 * the budget and trim the last one.  idx[u][0..count) receives the token ids
 * in rank order, ascending inside a cluster (the trimmed cluster keeps its
 * lowest ids); count[u] = min(B, clustered tokens).  Entries past count are
 * left unchanged.  Errors: CKV_ERR_STATE (no clusters), CKV_ERR_ARG (B < 0),
 * CKV_ERR_CAPACITY (B > max_budget), CKV_ERR_UNIMPLEMENTED (more than 8192
 * clusters per unit: the ranking keeps one CTA's shared memory). */
ckv_status ckv_select_scored(ckv_ctx* ctx, const float* scores, int32_t B, int32_t* idx,
                             int32_t* count, void* stream);

/* ckv_score followed by ckv_select_scored (scores kept in the workspace). */
ckv_status ckv_select(ckv_ctx* ctx, const void* q, int32_t q_dtype, int32_t B, int32_t* idx,
                      int32_t* count, void* stream);

/* Appends keys and values to the caches (section "Clustering in semantic
 * space", clustering strategy during inference: a generated token's K/V join
 * the cache and stay pending until their block is clustered; the prompt's K/V
 * are the cache the prefill clustering reads).  For every unit u and row
 * j < n: K[u][pos + j][:] = k_src[u][j][:] and V[u][pos + j][:] =
 * v_src[u][j][:]; k_src, v_src [units][src_len][d] of kv_dtype (src_len >= n
 * rows per unit; n = 1, src_len = 1 for one decode step).  The copy runs on
 * the SMs, so the sources may be mapped pinned host memory.  Touches no
 * context: the attention calls see the rows through cur_len.
 * Errors: CKV_ERR_ARG (n < 1, src_len < n, [pos, pos + n) outside
 * [0, max_len)), CKV_ERR_DTYPE, CKV_ERR_ALIGN. */
ckv_status ckv_append_kv(const void* k_src, const void* v_src, int32_t src_len, int32_t kv_dtype, int32_t units,
                         int32_t max_len, int32_t pos, int32_t n, void* K, void* V, void* stream);

/* Sparse decode attention (section "Background": softmax(q K_S^T / sqrt(d))
 * V_S).  For every unit and query head h: o_h = softmax over the attended
 * set S of (q_h . k_t / sqrt(d)) times v_t, where S = sinks [0, sinks) +
 * pending [clustered_end, cur_len) + idx[u][0..count[u]).  Each K/V row is
 * read once for all g heads; fp32 arithmetic; out is fp32.  An index outside
 * [0, cur_len) is skipped and sets CKV_DEV_BAD_INDEX.  Errors: CKV_ERR_ARG
 * (cur_len < clustered_end or > max_len), CKV_ERR_CAPACITY (B > max_budget or
 * more than 2*m pending tokens). */
ckv_status ckv_sparse_decode_attn(ckv_ctx* ctx, const void* q, int32_t q_dtype, const void* K,
                                  const void* V, const int32_t* idx, const int32_t* count,
                                  int32_t B, int32_t cur_len, float* out, void* stream);

/* One whole decode step of every unit in one call: ckv_select followed by
 * ckv_sparse_decode_attn on the same stream (the attention kernel is a
 * dependent launch of the selection kernel).  Arguments, layouts and errors as
 * for those two calls; idx [units][B], count [units] and out are written. */
ckv_status ckv_decode_step(ckv_ctx* ctx, const void* q, int32_t q_dtype, const void* K, const void* V,
                           int32_t B, int32_t cur_len, int32_t* idx, int32_t* count, float* out,
                           void* stream);

/* ---------------------------------------------------------------------------
 * Page-granular comparator (Quest), the baseline the ClusterKV page compares
 * its recall against (section "Background and design principles", drawbacks
 * of existing recallable compression; pages of 16 tokens, Fig. 3b).
 *
 * The clustered tokens [sinks, L) form n_pages = ceil((L - sinks) / 16) pages
 * of consecutive tokens (the last may be short).  ckv_quest_pages writes each
 * page's per-channel maximum and minimum key, page_max / page_min
 * [units][n_pages][d] of kv_dtype (caller-owned, 16-byte aligned).
 * ckv_quest_score writes each page's weight, the upper bound of q . k over the
 * page summed over the g query heads, scores [units][n_pages] float:
 *   w_p = sum_h sum_i max(q_hi * max_pi, q_hi * min_pi).
 * The selection is ckv_select_scored on a context whose clusters are the
 * pages (sizes 16, offsets 16 p, the identity permutation, imported with
 * ckv_import_clusters), and the attention ckv_sparse_decode_attn.
 * Errors: CKV_ERR_ARG (L <= sinks, L > max_len, g not 1/2/4/8),
 * CKV_ERR_DTYPE, CKV_ERR_ALIGN. */
ckv_status ckv_quest_pages(const void* K, int32_t kv_dtype, int32_t units, int32_t max_len, int32_t sinks,
                           int32_t L, void* page_max, void* page_min, void* stream);
ckv_status ckv_quest_score(const void* q, int32_t q_dtype, const void* page_max, const void* page_min,
                           int32_t units, int32_t g, int32_t n_pages, float* scores, void* stream);

/* ---------------------------------------------------------------------------
 * Reuse of earlier selections (section "Caching the KV of selected tokens":
 * a cache of the KV selected in the last R decode steps, only clusters missing
 * from it are loaded; cache-effectiveness analysis, hit rates for R = 1, 2).
 *
 * For every unit u: hits[u] = the number of tokens idx_cur[u][p],
 * p < cnt_cur[u], that appear in at least one of the R previous selections
 * idx_prev[r][u][0 .. cnt_prev[r][u]).  Whole clusters are selected, so
 * hits[u] / cnt_cur[u] is the token-weighted cluster hit rate.  Nothing is
 * loaded: every K/V row is resident, so this is a measurement only.
 * idx_prev / cnt_prev are HOST arrays of R device pointers (idx [units][B_prev]
 * int32, cnt [units] int32); idx_cur [units][B_cur], cnt_cur [units] and hits
 * [units] are device pointers.  Counts are clamped to [0, B]; ids outside
 * [0, max_len) are ignored.  R = 0 gives hits = 0.
 * Errors: CKV_ERR_ARG (R outside [0, 8], null pointers, negative sizes),
 * CKV_ERR_CAPACITY (max_len above 1.6 M tokens: the bitmap is in shared
 * memory), CKV_ERR_CUDA. */
ckv_status ckv_selection_overlap(int32_t units, int32_t max_len, int32_t R, const int32_t* const* idx_prev,
                                 const int32_t* const* cnt_prev, int32_t B_prev, const int32_t* idx_cur,
                                 const int32_t* cnt_cur, int32_t B_cur, int32_t* hits, void* stream);

/* ---------------------------------------------------------------------------
 * Channel pre-score, an alternative cheap scorer over the centroid table after
 * TailorKV's channel contribution (TailorKV page, dynamic retrieval for
 * sparsity-friendly layers: s_i = |q_i| * max |K_i|; attention scores
 * approximated from the critical channels only).
 *
 * ckv_centroid_channels writes a channel-major copy of the context's scoring
 * centroids, muT [units][d][max_clusters] of kv_dtype (entries c < n_clusters
 * written), and chmax [units][d] float = max over the current clusters of
 * |mu_c,i|.  Rebuild both whenever the clusters change (prefill, incremental
 * commit, import).  Caller-owned, 16-byte aligned.
 *
 * ckv_channel_prescore, per unit: qs_i = sum_h q_h,i (fp32, heads in order),
 * s_i = |qs_i| * chmax_i (fp32); the r channels of largest s_i (ties: lower
 * channel) in descending order ch_0 .. ch_{r-1}; then for every current
 * cluster scores[u][c] = sum_{j<r} qs_{ch_j} * muT[u][ch_j][c] (fp32, j in
 * order), row stride n_clusters like ckv_score, ready for ckv_select_scored.
 * channels [units][r] int32 receives ch_j when not null.  r in [1, 32].
 * Errors: CKV_ERR_ARG, CKV_ERR_DTYPE (q_dtype != kv_dtype), CKV_ERR_ALIGN,
 * CKV_ERR_STATE (no clusters). */
ckv_status ckv_centroid_channels(ckv_ctx* ctx, void* muT, float* chmax, void* stream);
ckv_status ckv_channel_prescore(ckv_ctx* ctx, const void* q, int32_t q_dtype, const void* muT, const float* chmax,
                                int32_t r, float* scores, int32_t* channels, void* stream);

/* Sparse decode attention that allocates nothing and needs no context.
 * The ClusterKV paper has no counterpart of this call; it exists for callers
 * that cannot allocate device memory: code running while a CUDA graph is
 * being captured, engines whose memory planner owns the whole device, or
 * processes that handed all free memory to a pooling allocator.  (Creating a
 * ckv_ctx allocates, so those callers cannot use ckv_sparse_decode_attn.)
 * It computes exactly what ckv_sparse_decode_attn computes, with the same
 * kernel, for caller-given state: the attended set of unit u is tokens
 * [0, sinks) + [clustered_end, cur_len) + idx[u][0..count[u]); q, K, V, idx,
 * count and out have the layouts given at the top of this file (K and V with
 * max_len rows per unit).  dev_err is an optional device int32 (NULL = none)
 * that receives CKV_DEV_* codes.
 * Scratch: the split partials live in one fixed 8 MiB device array inside
 * the library (held on every device that loads the library until the process
 * exits).  A call needs
 *   units * ceil((sinks + cur_len - clustered_end + B) / R) * g * 130 * 4
 * bytes, where R is the rows of one attention work item: 16 for bf16, 64 for
 * fp32 with g <= 4 and 32 for fp32 with g = 8; larger calls return
 * CKV_ERR_CAPACITY before launching anything.  The first call on each device
 * looks the array's device address up (cudaGetSymbolAddress) in that device's
 * primary context (the one the CUDA runtime uses) and keeps it: make that
 * first call before any stream capture, and do not use the entry point across
 * a cudaDeviceReset (the cached address would be stale).  Every call reuses
 * the same array and overwrites what the previous call left in it (nothing is
 * read before the same call writes it), so calls that can overlap on the GPU
 * (different streams without ordering) race and must not be issued.
 * Errors: CKV_ERR_ARG, CKV_ERR_DTYPE,
 * CKV_ERR_ALIGN, CKV_ERR_CAPACITY, CKV_ERR_CUDA. */
ckv_status ckv_sparse_decode_attn_noalloc(const void* q, int32_t q_dtype, const void* K,
                                          const void* V, const int32_t* idx, const int32_t* count,
                                          int32_t units, int32_t g, int32_t max_len, int32_t sinks,
                                          int32_t clustered_end, int32_t cur_len, int32_t B,
                                          float* out, int32_t* dev_err, void* stream);

/* Host-side copy of the context's counters. */
ckv_status ckv_get_info(ckv_ctx* ctx, ckv_info* info);

/* Copies the cluster state out to caller device buffers (any may be NULL):
 * mu [units][n_clusters][d] float centroids; mu_hat [units][n_clusters][d]
 * normalised centroid directions in the assignment operand type (bf16 for
 * bf16 keys, else float); sizes [units][n_clusters]; offsets
 * [units][n_clusters + 1]; perm [units][clustered_end - sinks]. */
ckv_status ckv_export_clusters(ckv_ctx* ctx, float* mu, void* mu_hat, int32_t* sizes,
                               int32_t* offsets, int32_t* perm, void* stream);

/* Replaces the cluster state from caller device buffers (same layouts as
 * ckv_export_clusters).  mu is required and the derived operand copies are
 * recomputed from it; sizes, offsets and perm may all be NULL (centroids only,
 * e.g. before ckv_kmeans_assign), else all three are required and
 * clustered_end gives the perm length (+ sinks). */
ckv_status ckv_import_clusters(ckv_ctx* ctx, int32_t n_clusters, int32_t clustered_end,
                               const float* mu, const int32_t* sizes, const int32_t* offsets,
                               const int32_t* perm, void* stream);

/* Failure detection.  Every wait inside the library's kernels (an mbarrier
 * phase, a flag another warp sets) is bounded: after `cycles` SM clock cycles
 * (default 2e9, about one second at 2 GHz) the waiting warp gives up, records
 * CKV_DEV_TIMEOUT in the device error word, the kernel lets the copies and
 * tensor-core operations it already started complete (each of those waits
 * bounded the same way), releases its tensor memory and returns; the context
 * stays usable.  ckv_set_wait_limit sets that limit for this context's later
 * launches (1 <= cycles <= 4e9).  stall = 1 makes the next launches of two
 * kernels wait once on a barrier nothing ever completes, so that their
 * failure path runs: the tensor-core K-means assignment (bf16 keys) and the
 * fp32 sparse attention (whose outputs are then not valid).  stall = 0
 * restores normal operation.  This exists to test failure detection (see
 * ckv_get_device_error) without faulting or hanging a GPU.
 * Errors: CKV_ERR_ARG. */
ckv_status ckv_set_wait_limit(ckv_ctx* ctx, int64_t cycles, int32_t stall);

/* L2 residency of the data every decode step re-reads (a GB300 has 129 MB of
 * L2; the gathered K/V rows of one step are larger and have no reuse, so
 * without this they evict the rest each step).  bytes > 0 sets aside up to
 * that many bytes of L2 for persisting lines (capped at the device maximum),
 * bytes < 0 sets aside the size of the bf16 / fp32 scoring copy of the
 * centroids, [units][max_clusters][d], when all of it fits the device's
 * maximum (and otherwise leaves persistence off: a set-aside holding a
 * fraction of it would mostly take L2 from the K-means passes), bytes = 0
 * turns it off.  While it is on, the kernels that score (the selection, up
 * to 1024 clusters, or the scoring kernel) read the centroid copy through an
 * access-policy window whose hits persist (hit ratio = set-aside / its
 * bytes, at most 1), and a selection from given scores reads perm through
 * one holding what is left of the set-aside.  The set-aside is the calling
 * process's CUDA-context limit cudaLimitPersistingL2CacheSize on the current
 * device: it is released with that context, the value found before the first
 * call is restored by bytes = 0 and by ckv_destroy, and the persisting lines
 * are reset then.  Results do not change.
 * Errors: CKV_ERR_ARG (ctx null), CKV_ERR_CUDA (the limit could not be set,
 * e.g. the device has no persisting L2). */
ckv_status ckv_set_l2_persistence(ckv_ctx* ctx, int64_t bytes);

/* Synchronises the context's last stream and reads then clears the device
 * error word (CKV_DEV_*). */
ckv_status ckv_get_device_error(ckv_ctx* ctx, int32_t* code);

#ifdef __cplusplus
}
#endif

#endif /* CKV_H */
