"""Plain CPU oracle for ClusterKV's cluster-granular recallable KV selection.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) imports, links or calls this module; only ``tests/``, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` do.

Source: "ClusterKV: Manipulating LLM KV Cache in Semantic Space for Recallable
Compression" (papercache summary page, arXiv 2412.03213).  Every function below
names the section of that page it follows.  ClusterKV is a heuristic: it does not
compute the exact top-B tokens, it approximates them.  So this module writes the
algorithm out step by step, in float64, in the order the page gives it:

  * semantic distance and K-means over keys  - section "Clustering in semantic
    space" (semantic distance, clustering process, clustering strategy during
    inference);
  * centroid scoring and selection           - section "Selection at semantic-
    cluster granularity" and section "Selection and indexing mechanism" (Fig. 8);
  * sparse attention                         - section "Background: long-context
    inference and KV-cache compression";
  * the exact objective (top-B by q.k)       - section "Problem formulation and
    design principle".

Readings of points the page leaves open:
  * C = floor((L - 16) / 80): the 16 sink tokens are not counted in L/80.
  * Seeding ("randomly sample keys as initial centroids") is read as the
    deterministic stride pick mu_j = k[s*j], s = min(80, floor(n / C)).
  * The update is the mean of the RAW assigned keys (not of normalised keys).
  * An empty cluster keeps its old centroid and has size 0.
  * A zero-norm key has cosine 0 with every centroid, so it joins cluster 0.
  * Ties: lowest cluster index wins an argmax; clusters rank by (score desc,
    index asc); tokens inside a cluster are in ascending token id; the trimmed
    last cluster keeps its lowest token ids.
  * The argmax over cosines is taken with the centroid directions rounded to the
    kernel's operand precision (bf16 for bf16 keys), since floating point here
    decides an integer label.  Dots are then exact (float64 of bf16 values).

Parity pins for every function live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

# Constants of the method (section "Clustering in semantic space", clustering
# strategy during inference): 16 attention-sink tokens are always kept, the
# prompt is clustered into C0 = L/80 clusters, and every m = 320 decode steps the
# new tokens are clustered among themselves into C+ = 4 clusters.
SINKS = 16
RATIO = 80
M_INCR = 320
C_PLUS = 4


# --------------------------------------------------------------------------
# cluster count and seeding
# --------------------------------------------------------------------------
def cluster_count(L: int, sinks: int = SINKS, ratio: int = RATIO) -> int:
    """C0 = L/80 over the clustered (non-sink) prompt tokens.

    Section "Clustering in semantic space": the first 16 tokens are kept and
    the remaining prompt tokens are grouped into C0 = L/80 clusters.  Reading:
    C = floor((L - sinks) / ratio), at least 1.
    """
    return max(1, (L - sinks) // ratio)


def seed_stride(n: int, C: int, ratio: int = RATIO) -> int:
    """Stride of the deterministic seeding: s = min(ratio, floor(n / C)), >= 1."""
    return max(1, min(ratio, n // C))


def seed_centroids(keys: np.ndarray, C: int, ratio: int = RATIO) -> np.ndarray:
    """Initial centroids: sampled keys (section "Clustering in semantic space",
    clustering process; Fig. 4).  Read as mu_j = k[s * j], j < C."""
    s = seed_stride(len(keys), C, ratio)
    return np.asarray(keys, dtype=np.float64)[np.arange(C) * s].copy()


# --------------------------------------------------------------------------
# operand rounding (precision of the argmax decision)
# --------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significant bits), ties
    to even; the result is returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def normalize_centroids(mu: np.ndarray, operand: str = "bf16", rel_err: float = 2.0 ** -20):
    """Centroid directions mu_c / ||mu_c|| used by the cosine assignment.

    Returns (mu_hat, amb).  For ``operand == "bf16"`` mu_hat is rounded to
    bfloat16 (the kernel's operand precision).  ``amb[c, j]`` is the size of the
    rounding step where the exact value lies within ``rel_err`` of a rounding
    midpoint, i.e. where an implementation that normalises in float32 may round
    the other way; 0 elsewhere.  For ``operand == "f64"`` mu_hat is unrounded and
    amb is all zero.  A zero centroid has mu_hat = 0.
    """
    mu = np.asarray(mu, dtype=np.float64)
    nrm = np.sqrt(np.sum(mu * mu, axis=1, keepdims=True))
    x = np.divide(mu, nrm, out=np.zeros_like(mu), where=nrm > 0)
    if operand == "f64":
        return x, np.zeros_like(x)
    if operand != "bf16":
        raise ValueError(operand)
    lo = round_to_bf16(x * (1.0 - rel_err))
    hi = round_to_bf16(x * (1.0 + rel_err))
    return round_to_bf16(x), np.abs(hi - lo)


# --------------------------------------------------------------------------
# K-means in semantic space
# --------------------------------------------------------------------------
def cosine_to_centroids(keys: np.ndarray, mu_hat: np.ndarray) -> np.ndarray:
    """cos(k_i, mu_c) = <k_i, mu_hat_c> / ||k_i||  (semantic distance
    D(i, j) = 1 - cos, section "Clustering in semantic space").  Zero keys: 0."""
    k = np.asarray(keys, dtype=np.float64)
    dots = k @ np.asarray(mu_hat, dtype=np.float64).T
    nrm = np.sqrt(np.sum(k * k, axis=1, keepdims=True))
    return np.divide(dots, nrm, out=np.zeros_like(dots), where=nrm > 0)


def assign(keys: np.ndarray, mu_hat: np.ndarray) -> np.ndarray:
    """Assignment step: each key joins the centroid nearest by D, i.e. with the
    largest cosine similarity (section "Clustering in semantic space",
    clustering process).  Ties go to the lowest cluster index."""
    cos = cosine_to_centroids(keys, mu_hat)
    return np.argmax(cos, axis=1).astype(np.int32)   # first maximum = lowest index


def update(keys: np.ndarray, labels: np.ndarray, mu_old: np.ndarray) -> np.ndarray:
    """Update step: the new centroid is the mean of the keys assigned to it
    (section "Clustering in semantic space", clustering process; section
    "Semantic clustering optimisation", Fig. 7).  Raw keys are averaged; an
    empty cluster keeps its previous centroid."""
    k = np.asarray(keys, dtype=np.float64)
    mu = np.array(mu_old, dtype=np.float64, copy=True)
    for c in range(mu.shape[0]):
        members = k[labels == c]
        if len(members):
            mu[c] = members.sum(axis=0) / len(members)
    return mu


def build_csr(labels: np.ndarray, C: int, token_base: int = 0):
    """Cluster metadata: sizes, their prefix sums, and the key indices sorted
    by label (section "Selection and indexing mechanism", Fig. 8).  Within a
    cluster the token ids stay ascending (stable sort).  Returns
    (sizes[C], offsets[C+1], perm[n]) with perm holding global token ids."""
    labels = np.asarray(labels)
    sizes = np.bincount(labels, minlength=C).astype(np.int32)[:C]
    offsets = np.zeros(C + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(sizes)
    perm = (np.argsort(labels, kind="stable") + token_base).astype(np.int32)
    return sizes, offsets.astype(np.int32), perm


def objective(keys: np.ndarray, labels: np.ndarray, mu: np.ndarray) -> float:
    """J = sum_i D(k_i, mu_{c(i)}) = sum_i (1 - cos(k_i, mu_{c(i)})), exact
    cosines (no operand rounding)."""
    mu_hat, _ = normalize_centroids(mu, "f64")
    cos = cosine_to_centroids(keys, mu_hat)
    return float(np.sum(1.0 - cos[np.arange(len(labels)), labels]))


def kmeans(keys: np.ndarray, C: int, iters: int, operand: str = "bf16",
           ratio: int = RATIO, token_base: int = 0, trace: bool = False):
    """Lloyd's K-means with the cosine distance (section "Clustering in semantic
    space", clustering process; Fig. 4): seed, then alternate assignment and
    update ``iters`` times.  The CSR of the last assignment is the cluster
    metadata kept for selection.

    Returns a dict with mu (float64 [C, d]), labels, sizes, offsets, perm and,
    if ``trace``, the per-iteration list of (mu_in, labels, mu_out, J_after_
    assign, J_after_update).
    """
    mu = seed_centroids(keys, C, ratio)
    labels = np.zeros(len(keys), dtype=np.int32)
    steps = []
    for _ in range(iters):
        mu_hat, _amb = normalize_centroids(mu, operand)
        labels = assign(keys, mu_hat)
        mu_new = update(keys, labels, mu)
        if trace:
            steps.append(dict(mu_in=mu, labels=labels, mu_out=mu_new,
                              J_assign=objective(keys, labels, mu),
                              J_update=objective(keys, labels, mu_new)))
        mu = mu_new
    sizes, offsets, perm = build_csr(labels, C, token_base)
    out = dict(mu=mu, labels=labels, sizes=sizes, offsets=offsets, perm=perm)
    if trace:
        out["trace"] = steps
    return out


def cluster_prefill(K: np.ndarray, L: int, C: int | None = None, iters: int = 10,
                    operand: str = "bf16", sinks: int = SINKS, ratio: int = RATIO,
                    trace: bool = False):
    """Prefill clustering of one unit (one KV head): keep tokens [0, sinks) as
    attention sinks and cluster the keys of tokens [sinks, L) into C clusters
    (section "Clustering in semantic space", clustering strategy during
    inference).  Token ids in ``perm`` are global (>= sinks)."""
    if C is None or C == 0:
        C = cluster_count(L, sinks, ratio)
    keys = np.asarray(K[sinks:L], dtype=np.float64)
    return kmeans(keys, C, iters, operand, ratio, token_base=sinks, trace=trace)


def cluster_incremental(K: np.ndarray, start: int, m: int = M_INCR, c_plus: int = C_PLUS,
                        iters: int = 10, operand: str = "bf16", ratio: int = RATIO,
                        trace: bool = False):
    """Incremental clustering of the m newest tokens [start, start+m) among
    themselves into C+ clusters (section "Clustering in semantic space",
    clustering strategy during inference: every m = 320 steps, C+ = 4)."""
    keys = np.asarray(K[start:start + m], dtype=np.float64)
    return kmeans(keys, c_plus, iters, operand, ratio, token_base=start, trace=trace)


def append_clusters(state: dict, new: dict) -> dict:
    """Append an incremental clustering result to a unit's cluster metadata:
    the new centroids follow the old ones and their CSR segment follows the old
    segments (section "Selection and indexing mechanism" metadata, extended by
    the incremental clusters of section "Clustering in semantic space")."""
    n_old = int(state["offsets"][-1])
    return dict(
        mu=np.concatenate([state["mu"], new["mu"]]),
        sizes=np.concatenate([state["sizes"], new["sizes"]]).astype(np.int32),
        offsets=np.concatenate([state["offsets"][:-1], new["offsets"] + n_old]).astype(np.int32),
        perm=np.concatenate([state["perm"], new["perm"]]).astype(np.int32),
    )


# --------------------------------------------------------------------------
# selection
# --------------------------------------------------------------------------
def score(q: np.ndarray, mu: np.ndarray) -> np.ndarray:
    """Cluster importance q . mu_c^T (section "Selection at semantic-cluster
    granularity": the inner product, not the cosine, to match the attention
    weights).  With grouped-query attention the g query heads that share a KV
    head each contribute: score_c = sum_h q_h . mu_c."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    return (q @ np.asarray(mu, dtype=np.float64).T).sum(axis=0)


def rank_clusters(scores: np.ndarray) -> np.ndarray:
    """Clusters in descending score order, ties by ascending cluster index."""
    scores = np.asarray(scores)
    return np.lexsort((np.arange(len(scores)), -scores.astype(np.float64)))


def select(scores: np.ndarray, sizes: np.ndarray, offsets: np.ndarray, perm: np.ndarray,
           B: int):
    """Selection and indexing (section "Selection and indexing mechanism",
    Fig. 8): sort the clusters by score, gather their sizes in that order,
    take clusters while their prefix sum stays within the budget, and trim the
    last selected cluster so exactly min(B, clustered tokens) tokens are taken.
    Returns (idx[count] in rank order, count)."""
    order = rank_clusters(scores)
    out = []
    for c in order:
        need = B - len(out)
        if need <= 0:
            break
        seg = perm[offsets[c]:offsets[c] + sizes[c]]
        out.extend(int(t) for t in seg[:need])
    return np.asarray(out, dtype=np.int32), len(out)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def attention_tokens(sinks: int, clustered_end: int, cur_len: int, idx: np.ndarray) -> np.ndarray:
    """Tokens attended at a decode step: the sinks (always kept), the tokens
    not yet clustered (positions [clustered_end, cur_len)), and the selected
    clustered tokens."""
    return np.concatenate([np.arange(sinks), np.arange(clustered_end, cur_len),
                           np.asarray(idx, dtype=np.int64)]).astype(np.int64)


def sparse_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    """softmax(q K_S^T / sqrt(d)) V_S over the selected tokens S (section
    "Background", long-context inference and KV-cache compression).  One
    output row per query head; float64 with a max-subtracted softmax."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    Ks = np.asarray(K, dtype=np.float64)[tokens]
    Vs = np.asarray(V, dtype=np.float64)[tokens]
    logits = (q @ Ks.T) / np.sqrt(q.shape[1])
    logits -= logits.max(axis=1, keepdims=True)
    w = np.exp(logits)
    w /= w.sum(axis=1, keepdims=True)
    return w @ Vs


def full_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, cur_len: int) -> np.ndarray:
    """softmax(q K^T / sqrt(d)) V over every token (section "Background")."""
    return sparse_attention(q, K, V, np.arange(cur_len))


# --------------------------------------------------------------------------
# the exact objective and recall
# --------------------------------------------------------------------------
def exact_top_b(q: np.ndarray, K: np.ndarray, candidates: np.ndarray, B: int) -> np.ndarray:
    """I_T = argmax over |I_T| = B of sum_{i in I_T} q k_i^T (section "Problem
    formulation and design principle"): the B candidates with the largest
    q . k_i (summed over the query heads of a group), ties by lower token id."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    cand = np.asarray(candidates, dtype=np.int64)
    w = (q @ np.asarray(K, dtype=np.float64)[cand].T).sum(axis=0)
    order = np.lexsort((cand, -w))
    return cand[order[:B]]


def recall(selected: np.ndarray, q: np.ndarray, K: np.ndarray, candidates: np.ndarray, B: int):
    """Recall of the selection against the exact top-B (section "Experiments",
    recall of important tokens).  Returns (token recall |S n TopB| / |TopB|,
    attention-mass recall sum_{S} a / sum_{TopB} a), where a is the full
    softmax over the candidates, averaged over the query heads."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    cand = np.asarray(candidates, dtype=np.int64)
    top = exact_top_b(q, K, cand, B)
    sel = np.asarray(selected, dtype=np.int64)
    tok = len(np.intersect1d(sel, top)) / max(1, len(top))
    logits = (q @ np.asarray(K, dtype=np.float64)[cand].T) / np.sqrt(q.shape[1])
    logits -= logits.max(axis=1, keepdims=True)
    a = np.exp(logits)
    a /= a.sum(axis=1, keepdims=True)
    pos = {int(t): i for i, t in enumerate(cand)}
    s_idx = np.array([pos[int(t)] for t in sel if int(t) in pos], dtype=np.int64)
    t_idx = np.array([pos[int(t)] for t in top], dtype=np.int64)
    mass = a[:, s_idx].sum(axis=1) / np.maximum(a[:, t_idx].sum(axis=1), 1e-300)
    return tok, float(mass.mean())
