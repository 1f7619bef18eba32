// Plain C++ oracle for ClusterKV's cluster-granular recallable KV selection.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
// Python binding) links, loads or calls this file; only tests/, the smoke
// check in __graft_entry__ and the CPU-baseline leg of bench.py do, through
// oracle/cpp.py.  It shares no code with the CUDA path.
//
// Source: "ClusterKV: Manipulating LLM KV Cache in Semantic Space for Recallable
// Compression" (papercache summary page, arXiv 2412.03213).  The algorithm is
// written out step by step in float64, one function per step, in the order the
// page gives it, with the same readings as the float64 numpy oracle in
// oracle/clusterkv.py (each function below names that function):
//   * cosine K-means over keys: section "Clustering in semantic space"
//     (semantic distance, clustering process, strategy during inference);
//   * centroid scoring and cluster selection: section "Selection at
//     semantic-cluster granularity" and section "Selection and indexing
//     mechanism" (Fig. 8);
//   * sparse attention: section "Background: long-context inference and
//     KV-cache compression".
// Readings of points the page leaves open: C = floor((L - 16) / 80); the seeds
// are keys at stride s = min(80, floor(n / C)); the update is the mean of the
// raw keys and an empty cluster keeps its centroid; a zero key has cosine 0
// with every centroid; arg-max ties go to the lower cluster index, clusters
// rank by (score desc, index asc), tokens inside a cluster ascend, and the
// trimmed last cluster keeps its lowest token ids; the arg-max is taken with
// the centroid directions rounded to the kernel's operand precision (bf16 for
// bf16 keys), dots exact in float64.
//
// ckvo_unit_jobs runs whole per-unit jobs (prefill clustering, then every
// decode step) on a pool of std::threads, one unit per thread at a time; the
// units are independent.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <numeric>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- operand rounding
// round-to-nearest-even to 8 significant bits (bfloat16), in float64
double round_bf16(double x) {
    int e = 0;
    const double m = frexp(x, &e);            // x = m 2^e, 0.5 <= |m| < 1
    return ldexp(nearbyint(m * 256.0), e - 8);  // default rounding: ties to even
}

// clusterkv.normalize_centroids: mu_c / ||mu_c|| (0 for a zero centroid), rounded
// to bf16 if requested; amb = the bf16 step wherever a relative change of
// rel_err can round the other way, else 0
void normalize(const double* mu, int C, int d, bool bf16, double rel_err, double* mu_hat, double* amb) {
    for (int c = 0; c < C; ++c) {
        double ss = 0.0;
        for (int j = 0; j < d; ++j) ss += mu[(size_t)c * d + j] * mu[(size_t)c * d + j];
        const double nrm = sqrt(ss);
        for (int j = 0; j < d; ++j) {
            const double x = nrm > 0.0 ? mu[(size_t)c * d + j] / nrm : 0.0;
            if (bf16) {
                mu_hat[(size_t)c * d + j] = round_bf16(x);
                if (amb) amb[(size_t)c * d + j] = fabs(round_bf16(x * (1.0 + rel_err)) - round_bf16(x * (1.0 - rel_err)));
            } else {
                mu_hat[(size_t)c * d + j] = x;
                if (amb) amb[(size_t)c * d + j] = 0.0;
            }
        }
    }
}

// dot product in float64 with four running partial sums (channels j mod 4),
// added at the end
double dot(const double* a, const double* b, int d) {
    double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
    int j = 0;
    for (; j + 4 <= d; j += 4) {
        s0 += a[j] * b[j];
        s1 += a[j + 1] * b[j + 1];
        s2 += a[j + 2] * b[j + 2];
        s3 += a[j + 3] * b[j + 3];
    }
    for (; j < d; ++j) s0 += a[j] * b[j];
    return (s0 + s1) + (s2 + s3);
}

// clusterkv.assign: each key joins the centroid of largest cosine
// <k, mu_hat_c> / ||k||; the first maximum (lowest index) wins; zero key -> 0
void assign(const double* keys, int n, int d, const double* mu_hat, int C, int32_t* labels) {
    for (int i = 0; i < n; ++i) {
        const double* k = keys + (size_t)i * d;
        const double nrm = sqrt(dot(k, k, d));
        int arg = 0;
        if (nrm > 0.0) {
            double best = -INFINITY;
            for (int c = 0; c < C; ++c) {
                const double cs = dot(k, mu_hat + (size_t)c * d, d) / nrm;
                if (cs > best) {
                    best = cs;
                    arg = c;
                }
            }
        }
        labels[i] = arg;
    }
}

// clusterkv.update: mean of the raw keys of each cluster; empty keeps mu_old
void update(const double* keys, int n, int d, const int32_t* labels, const double* mu_old, int C, double* mu) {
    std::vector<double> sum((size_t)C * d, 0.0);
    std::vector<int64_t> cnt(C, 0);
    for (int i = 0; i < n; ++i) {
        const int c = labels[i];
        ++cnt[c];
        for (int j = 0; j < d; ++j) sum[(size_t)c * d + j] += keys[(size_t)i * d + j];
    }
    for (int c = 0; c < C; ++c)
        for (int j = 0; j < d; ++j)
            mu[(size_t)c * d + j] = cnt[c] ? sum[(size_t)c * d + j] / (double)cnt[c] : mu_old[(size_t)c * d + j];
}

// clusterkv.build_csr: sizes, exclusive prefix sums, token ids stably sorted by label
void build_csr(const int32_t* labels, int n, int C, int32_t base, int32_t* sizes, int32_t* offsets, int32_t* perm) {
    for (int c = 0; c < C; ++c) sizes[c] = 0;
    for (int i = 0; i < n; ++i) ++sizes[labels[i]];
    offsets[0] = 0;
    for (int c = 0; c < C; ++c) offsets[c + 1] = offsets[c] + sizes[c];
    std::vector<int32_t> fill(offsets, offsets + C);
    for (int i = 0; i < n; ++i) perm[fill[labels[i]]++] = base + i;  // ascending i: stable
}

// clusterkv.objective: J = sum_i (1 - cos(k_i, mu_c(i))), exact cosines
double objective(const double* keys, int n, int d, const int32_t* labels, const double* mu, int C) {
    std::vector<double> mh((size_t)C * d);
    normalize(mu, C, d, false, 0.0, mh.data(), nullptr);
    double J = 0.0;
    for (int i = 0; i < n; ++i) {
        const double* k = keys + (size_t)i * d;
        const double nrm = sqrt(dot(k, k, d));
        const double cs = nrm > 0.0 ? dot(k, mh.data() + (size_t)labels[i] * d, d) / nrm : 0.0;
        J += 1.0 - cs;
    }
    return J;
}

int seed_stride(int n, int C, int ratio) { return std::max(1, std::min(ratio, n / C)); }

// clusterkv.kmeans: seed, then `iters` x (assignment, update); the CSR of the
// last assignment
void kmeans(const double* keys, int n, int d, int C, int iters, bool bf16, int ratio, int32_t base, double* mu,
            int32_t* labels, int32_t* sizes, int32_t* offsets, int32_t* perm) {
    const int s = seed_stride(n, C, ratio);
    for (int c = 0; c < C; ++c) memcpy(mu + (size_t)c * d, keys + (size_t)c * s * d, sizeof(double) * d);
    for (int i = 0; i < n; ++i) labels[i] = 0;
    std::vector<double> mh((size_t)C * d), mn((size_t)C * d);
    for (int it = 0; it < iters; ++it) {
        normalize(mu, C, d, bf16, 0.0, mh.data(), nullptr);
        assign(keys, n, d, mh.data(), C, labels);
        update(keys, n, d, labels, mu, C, mn.data());
        memcpy(mu, mn.data(), sizeof(double) * C * d);
    }
    build_csr(labels, n, C, base, sizes, offsets, perm);
}

// clusterkv.score: score_c = sum_h q_h . mu_c
void score(const double* q, int g, int d, const double* mu, int C, double* out) {
    for (int c = 0; c < C; ++c) {
        double s = 0.0;
        for (int h = 0; h < g; ++h) s += dot(q + (size_t)h * d, mu + (size_t)c * d, d);
        out[c] = s;
    }
}

// clusterkv.select: clusters by (score desc, index asc); whole clusters in that
// order, the last trimmed, until min(B, clustered) tokens; idx in rank order
int select(const double* scores, const int32_t* sizes, const int32_t* offsets, const int32_t* perm, int C, int B,
           int32_t* idx) {
    std::vector<int> order(C);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return scores[a] > scores[b]; });
    int cnt = 0;
    for (int r = 0; r < C && cnt < B; ++r) {
        const int c = order[r];
        for (int t = 0; t < sizes[c] && cnt < B; ++t) idx[cnt++] = perm[offsets[c] + t];
    }
    return cnt;
}

// clusterkv.sparse_attention: softmax(q K_S^T / sqrt(d)) V_S, max-subtracted
void sparse_attention(const double* q, int g, int d, const double* K, const double* V, const int64_t* tok, int nt,
                      double* out) {
    std::vector<double> w(nt);
    const double scale = 1.0 / sqrt((double)d);
    for (int h = 0; h < g; ++h) {
        double mx = -INFINITY;
        for (int i = 0; i < nt; ++i) {
            w[i] = dot(q + (size_t)h * d, K + (size_t)tok[i] * d, d) * scale;
            mx = std::max(mx, w[i]);
        }
        double sum = 0.0;
        for (int i = 0; i < nt; ++i) {
            w[i] = exp(w[i] - mx);
            sum += w[i];
        }
        for (int j = 0; j < d; ++j) out[(size_t)h * d + j] = 0.0;
        for (int i = 0; i < nt; ++i) {
            const double p = w[i] / sum;
            const double* v = V + (size_t)tok[i] * d;
            for (int j = 0; j < d; ++j) out[(size_t)h * d + j] += p * v[j];
        }
    }
}

}  // namespace

extern "C" {

double ckvo_round_bf16(double x) { return round_bf16(x); }

void ckvo_round_bf16_n(const double* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = round_bf16(x[i]);
}

void ckvo_normalize(const double* mu, int C, int d, int bf16, double rel_err, double* mu_hat, double* amb) {
    normalize(mu, C, d, bf16 != 0, rel_err, mu_hat, amb);
}

void ckvo_cosines(const double* keys, int n, int d, const double* mu_hat, int C, double* cos) {
    for (int i = 0; i < n; ++i) {
        const double* k = keys + (size_t)i * d;
        const double nrm = sqrt(dot(k, k, d));
        for (int c = 0; c < C; ++c) cos[(size_t)i * C + c] = nrm > 0.0 ? dot(k, mu_hat + (size_t)c * d, d) / nrm : 0.0;
    }
}

void ckvo_assign(const double* keys, int n, int d, const double* mu_hat, int C, int32_t* labels) {
    assign(keys, n, d, mu_hat, C, labels);
}

void ckvo_update(const double* keys, int n, int d, const int32_t* labels, const double* mu_old, int C, double* mu) {
    update(keys, n, d, labels, mu_old, C, mu);
}

void ckvo_build_csr(const int32_t* labels, int n, int C, int32_t base, int32_t* sizes, int32_t* offsets,
                    int32_t* perm) {
    build_csr(labels, n, C, base, sizes, offsets, perm);
}

double ckvo_objective(const double* keys, int n, int d, const int32_t* labels, const double* mu, int C) {
    return objective(keys, n, d, labels, mu, C);
}

int ckvo_seed_stride(int n, int C, int ratio) { return seed_stride(n, C, ratio); }

void ckvo_kmeans(const double* keys, int n, int d, int C, int iters, int bf16, int ratio, int32_t base, double* mu,
                 int32_t* labels, int32_t* sizes, int32_t* offsets, int32_t* perm) {
    kmeans(keys, n, d, C, iters, bf16 != 0, ratio, base, mu, labels, sizes, offsets, perm);
}

void ckvo_score(const double* q, int g, int d, const double* mu, int C, double* out) { score(q, g, d, mu, C, out); }

int ckvo_select(const double* scores, const int32_t* sizes, const int32_t* offsets, const int32_t* perm, int C, int B,
                int32_t* idx) {
    return select(scores, sizes, offsets, perm, C, B, idx);
}

void ckvo_sparse_attention(const double* q, int g, int d, const double* K, const double* V, const int64_t* tok,
                           int nt, double* out) {
    sparse_attention(q, g, d, K, V, tok, nt, out);
}

// Whole jobs of `units` independent units on `threads` std::threads.  Unit u:
// K_u, V_u [max_len][d] and Q_u [T][g][d] (float64).  Prefill clustering of
// tokens [sinks, L) into C clusters (`iters` iterations); then T decode steps:
// before steps m, 2m, ... the m newest tokens are clustered into c_plus
// appended clusters; each step scores, selects B tokens and attends to sinks +
// pending + selected (tokens [0, L + t + 1)).  out_u [T][g][d] receives the
// attention outputs; times_u[2] the prefill and decode seconds of the unit.
void ckvo_unit_jobs(int units, const double* const* K, const double* const* V, const double* const* Q,
                    double* const* out, int L, int T, int C, int B, int iters, int m, int c_plus, int sinks, int ratio,
                    int g, int d, int bf16, int threads, double* times) {
    std::atomic<int> next(0);
    auto worker = [&]() {
        for (int u = next.fetch_add(1); u < units; u = next.fetch_add(1)) {
            const auto t0 = std::chrono::steady_clock::now();
            const int n = L - sinks;
            const int cmax = C + c_plus * (T / m + 1);
            std::vector<double> mu((size_t)cmax * d);
            std::vector<int32_t> sizes(cmax), offsets(cmax + 1), perm((size_t)n + (size_t)T), lab((size_t)n);
            kmeans(K[u] + (size_t)sinks * d, n, d, C, iters, bf16 != 0, ratio, sinks, mu.data(), lab.data(),
                   sizes.data(), offsets.data(), perm.data());
            int nc = C, end = L;
            const auto t1 = std::chrono::steady_clock::now();
            std::vector<double> sc(cmax), mi((size_t)c_plus * d);
            std::vector<int32_t> idx(B), li(m), si(c_plus), oi(c_plus + 1), pi(m);
            std::vector<int64_t> tok;
            for (int t = 0; t < T; ++t) {
                if (t > 0 && t % m == 0) {
                    // incremental clustering of [end, end + m), appended
                    kmeans(K[u] + (size_t)end * d, m, d, c_plus, iters, bf16 != 0, ratio, end, mi.data(), li.data(),
                           si.data(), oi.data(), pi.data());
                    const int base = offsets[nc];
                    for (int j = 0; j < c_plus; ++j) {
                        memcpy(mu.data() + (size_t)(nc + j) * d, mi.data() + (size_t)j * d, sizeof(double) * d);
                        sizes[nc + j] = si[j];
                        offsets[nc + j + 1] = base + oi[j + 1];
                    }
                    memcpy(perm.data() + base, pi.data(), sizeof(int32_t) * m);
                    nc += c_plus;
                    end += m;
                }
                const double* q = Q[u] + (size_t)t * g * d;
                score(q, g, d, mu.data(), nc, sc.data());
                const int cnt = select(sc.data(), sizes.data(), offsets.data(), perm.data(), nc, B, idx.data());
                const int cur = L + t + 1;
                tok.clear();
                for (int i = 0; i < sinks; ++i) tok.push_back(i);
                for (int i = end; i < cur; ++i) tok.push_back(i);
                for (int i = 0; i < cnt; ++i) tok.push_back(idx[i]);
                sparse_attention(q, g, d, K[u], V[u], tok.data(), (int)tok.size(), out[u] + (size_t)t * g * d);
            }
            const auto t2 = std::chrono::steady_clock::now();
            times[2 * u] = std::chrono::duration<double>(t1 - t0).count();
            times[2 * u + 1] = std::chrono::duration<double>(t2 - t1).count();
        }
    };
    const int nt = std::max(1, std::min(threads, units));
    std::vector<std::thread> pool;
    for (int i = 0; i < nt; ++i) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
}

}  // extern "C"
