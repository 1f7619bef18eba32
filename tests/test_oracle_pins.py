"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function checks the oracle module it is given against something
the ClusterKV page or plain mathematics fixes: the page's selection example,
closed forms, invariants, special cases that reduce to a library routine, and
brute force on tiny inputs.  The ``test_mutant_*`` tests plant one plausible
mistake in a copy of the oracle (on the CPU) and check that a pin catches it.
"""
import importlib.util
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.clusterkv as ck
import oracle.cpp as cc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------
def pin_selection_worked_example(m):
    """Section "Selection and indexing mechanism", Fig. 8 (hand-built toy)."""
    g = json.load(open(os.path.join(GOLDEN, "selection_fig8.json")))
    cl = g["clusters"]
    for case in g["cases"]:
        idx, count = m.select(np.array(cl["scores"]), np.array(cl["sizes"]),
                              np.array(cl["offsets"]), np.array(cl["perm"]), case["B"])
        assert count == case["count"], case
        assert list(idx) == case["idx"], case


def pin_cluster_count(m):
    """C0 = L/80 over the non-sink tokens gives the cluster counts printed in
    the workload descriptions: 25 at 2k, 409 at 32k, 1638 at 128k."""
    assert m.cluster_count(2048) == 25
    assert m.cluster_count(32768) == 409
    assert m.cluster_count(131072) == 1638


def pin_bf16_rounding(m):
    """bf16 round-to-nearest-even agrees with torch's float32 -> bfloat16 cast
    (a library routine) on float32-representable inputs, including ties."""
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-3).astype(np.float32)])
    # exact ties: 8 significant bits plus a half ulp
    ties = (np.arange(1, 300, dtype=np.float64) * 2 + 1) * 2.0 ** -9 + 1.0
    x = np.concatenate([x, ties.astype(np.float32), -ties.astype(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = m.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def pin_assign_vs_scipy_cosine(m):
    """The assignment is the arg-min of the semantic distance D(i, j) =
    1 - cos(k_i, mu_j), here computed by scipy's cosine distance."""
    from scipy.spatial.distance import cdist
    rng = np.random.default_rng(2)
    for n, C, d in [(50, 7, 16), (200, 25, 128), (33, 3, 5)]:
        keys = rng.standard_normal((n, d)) * rng.uniform(0.1, 5.0, size=(n, 1))
        keys[:, 0] *= 20.0                       # an outlier channel
        mu = rng.standard_normal((C, d))
        mu_hat, amb = m.normalize_centroids(mu, "f64")
        assert not amb.any()
        got = m.assign(keys, mu_hat)
        D = cdist(keys, mu, metric="cosine")
        srt = np.sort(D, axis=1)
        clear = (srt[:, 1] - srt[:, 0]) > 1e-12
        assert clear.all()
        assert np.array_equal(got, np.argmin(D, axis=1))


def pin_assign_brute_force(m):
    """Brute force on tiny inputs: python loops over every (key, centroid)
    pair with math.sqrt, ties to the lowest cluster index; zero key -> 0."""
    rng = np.random.default_rng(3)
    for trial in range(30):
        n, C, d = rng.integers(1, 12), rng.integers(1, 4), rng.integers(1, 6)
        keys = rng.integers(-3, 4, size=(n, d)).astype(np.float64)
        mu = rng.integers(-3, 4, size=(C, d)).astype(np.float64)
        mu_hat, _ = m.normalize_centroids(mu, "f64")
        got = m.assign(keys, mu_hat)
        for i in range(n):
            kn = math.sqrt(sum(v * v for v in keys[i]))
            best, arg = -math.inf, 0
            for c in range(C):
                mn = math.sqrt(sum(v * v for v in mu[c]))
                cos = 0.0 if kn == 0 or mn == 0 else sum(a * b for a, b in zip(keys[i], mu[c])) / (kn * mn)
                if cos > best + 1e-12:
                    best, arg = cos, c
            assert got[i] == arg, (trial, i, keys[i], mu)


def pin_update_closed_form(m):
    """Keys placed symmetrically around known points have exactly those points
    as means; an empty cluster keeps its previous centroid."""
    rng = np.random.default_rng(4)
    C, d = 5, 8
    centres = rng.integers(-8, 8, size=(C, d)).astype(np.float64)
    keys, labels = [], []
    for c in range(C - 1):                   # cluster C-1 stays empty
        for _ in range(3):
            delta = rng.integers(-4, 4, size=d).astype(np.float64)
            keys += [centres[c] + delta, centres[c] - delta]
            labels += [c, c]
    keys, labels = np.array(keys), np.array(labels, dtype=np.int32)
    old = rng.standard_normal((C, d))
    mu = m.update(keys, labels, old)
    assert np.array_equal(mu[:C - 1], centres[:C - 1])
    assert np.array_equal(mu[C - 1], old[C - 1])


def pin_update_is_mean_logit(m):
    """Mean update <=> q . mu_c is the average of q . k_i over the cluster, for
    any q (the property that makes q . mu a cluster's mean attention logit)."""
    rng = np.random.default_rng(5)
    keys = rng.standard_normal((300, 16)) * 3
    labels = rng.integers(0, 9, size=300).astype(np.int32)
    mu = m.update(keys, labels, np.zeros((9, 16)))
    q = rng.standard_normal(16)
    for c in range(9):
        sel = labels == c
        if sel.any():
            assert abs(q @ mu[c] - np.mean(keys[sel] @ q)) < 1e-9


def pin_planted_partition(m):
    """Incremental clustering of 320 tokens in 4 contiguous blocks of 80 keys
    that point in 4 well-separated directions: seeding picks one key per block
    (stride 80), and the clusters recover the blocks exactly; token ids in the
    CSR are global; the centroids are the block means."""
    rng = np.random.default_rng(6)
    d, start = 128, 5000
    dirs = np.linalg.qr(rng.standard_normal((d, 4)))[0].T * 10
    K = rng.standard_normal((start + 400, d)) * 0.05
    for b in range(4):
        K[start + 80 * b: start + 80 * (b + 1)] += dirs[b] * rng.uniform(0.5, 2.0, size=(80, 1))
    for operand in ("bf16", "f64"):
        r = m.cluster_incremental(K, start, m=320, c_plus=4, iters=10, operand=operand)
        assert list(r["sizes"]) == [80, 80, 80, 80]
        assert list(r["offsets"]) == [0, 80, 160, 240, 320]
        assert np.array_equal(r["perm"], np.arange(start, start + 320))
        for b in range(4):
            assert np.allclose(r["mu"][b], K[start + 80 * b: start + 80 * (b + 1)].mean(axis=0),
                               rtol=0, atol=1e-12)


def pin_one_token_per_cluster_is_exact_top_b(m):
    """With C = n (one token per cluster) selection equals the exact top-B by
    q . k (the objective of section "Problem formulation"), found here by
    Python's sort over tokens."""
    rng = np.random.default_rng(7)
    L, d, g = 16 + 200, 32, 4
    K = rng.standard_normal((L, d))
    q = rng.standard_normal((g, d))
    st = m.cluster_prefill(K, L, C=L - 16, iters=3, operand="f64")
    assert list(st["sizes"]) == [1] * (L - 16)
    sc = m.score(q, st["mu"])
    w = {t: float(sum(q[h] @ K[t] for h in range(g))) for t in range(16, L)}
    for B in (1, 17, 64, 199, 200, 500):
        idx, count = m.select(sc, st["sizes"], st["offsets"], st["perm"], B)
        want = sorted(w, key=lambda t: (-w[t], t))[:B]
        assert count == min(B, L - 16)
        assert list(idx) == want


def pin_selection_vs_token_sort(m):
    """Selecting whole clusters by descending score, then trimming, equals
    sorting the tokens by (cluster score desc, cluster id asc, token id asc)
    and taking the first B."""
    rng = np.random.default_rng(8)
    for trial in range(40):
        C = int(rng.integers(1, 30))
        labels = rng.integers(0, C, size=int(rng.integers(1, 200)))
        sizes = np.bincount(labels, minlength=C)
        offsets = np.concatenate([[0], np.cumsum(sizes)])
        tokens = np.arange(100, 100 + len(labels))
        perm = tokens[np.argsort(labels, kind="stable")]
        scores = rng.integers(-5, 5, size=C).astype(np.float64)   # many ties
        B = int(rng.integers(0, len(labels) + 20))
        idx, count = m.select(scores, sizes, offsets, perm, B)
        lab = dict(zip(tokens.tolist(), labels.tolist()))
        want = sorted(tokens.tolist(), key=lambda t: (-scores[lab[t]], lab[t], t))[:B]
        assert count == len(want) and list(idx) == want, trial


def pin_attention_vs_torch_sdpa(m):
    """Sparse attention over a token subset equals torch's scaled-dot-product
    attention (float64, CPU) on the gathered rows; with every token selected it
    equals full attention; with B >= clustered tokens the sparse set is all."""
    rng = np.random.default_rng(9)
    L, d, g = 300, 128, 4
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    q = rng.standard_normal((g, d)) * 2
    tok = np.sort(rng.choice(L, size=77, replace=False))
    got = m.sparse_attention(q, K, V, tok)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(K[tok])[None],
        torch.from_numpy(V[tok])[None])[0].numpy()
    assert np.abs(got - ref).max() < 1e-12
    full = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None])[0].numpy()
    assert np.abs(m.full_attention(q, K, V, L) - full).max() < 1e-12
    st = m.cluster_prefill(K, L, C=10, iters=2, operand="f64")
    idx, count = m.select(m.score(q, st["mu"]), st["sizes"], st["offsets"], st["perm"], B=L)
    assert count == L - 16
    toks = m.attention_tokens(16, L, L, idx)
    assert np.abs(m.sparse_attention(q, K, V, toks) - full).max() < 1e-12


def pin_assignment_never_increases_objective(m):
    """With exact cosines the assignment step cannot increase
    J = sum_i (1 - cos(k_i, mu_c(i))) (each key takes its best centroid)."""
    rng = np.random.default_rng(10)
    keys = rng.standard_normal((600, 32)) + 2 * rng.standard_normal((1, 32))
    keys[:, 3] *= 20
    r = m.kmeans(keys, 12, 8, operand="f64", trace=True)
    tr = r["trace"]
    for t in range(1, len(tr)):
        assert tr[t]["J_assign"] <= tr[t - 1]["J_update"] + 1e-9


def pin_recall_properties(m):
    """Recall of the exact top-B is 1; a disjoint set of tokens has token recall 0."""
    rng = np.random.default_rng(11)
    K = rng.standard_normal((120, 16))
    q = rng.standard_normal((2, 16))
    cand = np.arange(16, 120)
    top = m.exact_top_b(q, K, cand, 20)
    tok, mass = m.recall(top, q, K, cand, 20)
    assert tok == 1.0 and abs(mass - 1.0) < 1e-12
    other = np.setdiff1d(cand, top)[:20]
    tok, mass = m.recall(other, q, K, cand, 20)
    assert tok == 0.0 and mass < 1.0


def pin_append_clusters(m):
    """Appending incremental clusters extends sizes/offsets/perm so that every
    cluster's token segment is unchanged and the new tokens follow."""
    rng = np.random.default_rng(12)
    K = rng.standard_normal((16 + 400 + 320, 16))
    st = m.cluster_prefill(K, 416, C=5, iters=3)
    inc = m.cluster_incremental(K, 416, 320, 4, iters=3)
    s2 = m.append_clusters(st, inc)
    assert len(s2["sizes"]) == 9 and s2["offsets"][-1] == 720 and len(s2["perm"]) == 720
    for c in range(9):
        seg = s2["perm"][s2["offsets"][c]: s2["offsets"][c] + s2["sizes"][c]]
        src = st if c < 5 else inc
        cc = c if c < 5 else c - 5
        want = src["perm"][src["offsets"][cc]: src["offsets"][cc] + src["sizes"][cc]]
        assert np.array_equal(seg, want)


def pin_attention_tokens_with_pending(m):
    """The attended set while decode tokens are pending (section "Clustering
    in semantic space", clustering strategy during inference: tokens are
    clustered in blocks of m, so the newest ones are not yet in any cluster):
    the sinks, every position in [clustered_end, cur_len) and the selected
    tokens, listed here by hand.  Attention over that set is checked against
    torch's scaled-dot-product attention over the same hand-listed rows."""
    idx = np.array([50, 17, 99, 23])
    got = m.attention_tokens(16, 100, 104, idx)
    want = list(range(16)) + [100, 101, 102, 103] + [50, 17, 99, 23]
    assert list(got) == want
    # nothing pending: sinks and the selection only
    assert list(m.attention_tokens(16, 100, 100, idx)) == list(range(16)) + [50, 17, 99, 23]
    # one pending token (the usual decode step right after a clustering)
    assert list(m.attention_tokens(4, 9, 10, np.array([5]))) == [0, 1, 2, 3, 9, 5]
    # no selection (budget 0): sinks and pending only
    assert list(m.attention_tokens(2, 7, 9, np.array([], dtype=np.int64))) == [0, 1, 7, 8]
    rng = np.random.default_rng(13)
    K = rng.standard_normal((110, 128))
    V = rng.standard_normal((110, 128))
    q = rng.standard_normal((4, 128))
    rows = want
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(K[rows])[None], torch.from_numpy(V[rows])[None])[0].numpy()
    out = m.sparse_attention(q, K, V, m.attention_tokens(16, 100, 104, idx))
    assert np.abs(out - ref).max() < 1e-12


def _f32_normalisations(mu):
    """Float32 normalisations of the rows of mu the way a GPU may compute
    them: the sum of squares as 32 lanes of 4 sequential terms followed by a
    butterfly over the lanes, or numpy's pairwise float32 sum; then sqrt and a
    division, or a multiplication by the reciprocal (all float32)."""
    m32 = np.asarray(mu, dtype=np.float32)
    sq = m32 * m32
    lanes = sq.reshape(len(m32), 32, -1)
    acc = lanes[:, :, 0].copy()
    for j in range(1, lanes.shape[2]):
        acc = (acc + lanes[:, :, j]).astype(np.float32)
    w = 16
    while w >= 1:
        acc = (acc + np.roll(acc, -w, axis=1)).astype(np.float32)
        w //= 2
    tree = acc[:, 0]
    pair = sq.sum(axis=1, dtype=np.float32)
    outs = []
    for ss in (tree, pair):
        nrm = np.sqrt(ss.astype(np.float32)).astype(np.float32)[:, None]
        outs.append((m32 / nrm).astype(np.float32))
        outs.append((m32 * (np.float32(1.0) / nrm).astype(np.float32)).astype(np.float32))
    return outs


def pin_rounding_band(m):
    """The ambiguity band of the bf16 centroid directions (used by the GPU
    acceptance rule for arg-max decisions): wherever any float32
    normalisation, or any relative perturbation of the exact unit vector up to
    2^-20, rounds to another bfloat16 than the exact value, the band holds
    that difference; the band is one bfloat16 step exactly where the exact
    value lies within 2^-20 (relative) of a rounding midpoint, and 0
    everywhere else."""
    rng = np.random.default_rng(14)
    mu = rng.standard_normal((64, 128)) * rng.uniform(0.01, 50.0, size=(64, 1))
    mu[:, 5] *= 20.0
    # rows with one component of the unit vector planted next to a bf16
    # midpoint (relative offsets 2^-26 .. 2^-18 from a (k + 1/2) step, both
    # sides): y_j = t sqrt(S / (1 - t^2)) gives y_j / ||y|| = t, S = the sum of
    # the other squares
    planted = []
    for r in range(160):
        y = rng.standard_normal(128)
        j = int(rng.integers(0, 128))
        y[j] = 0.0
        S = float(y @ y)
        t0 = rng.uniform(0.05, 0.9) * rng.choice([-1, 1])
        mant, ex = np.frexp(t0)
        t = float(np.ldexp(np.floor(mant * 256.0) + 0.5, ex - 8))
        t *= 1.0 + rng.choice([-1, 1]) * 2.0 ** rng.uniform(-26, -18)
        y[j] = t * math.sqrt(S / (1.0 - t * t))
        planted.append(y * rng.uniform(0.5, 3.0))
    mu = np.concatenate([mu, np.array(planted)])
    rel = 2.0 ** -20
    mh, amb = m.normalize_centroids(mu, "bf16", rel_err=rel)
    xe = mu / np.linalg.norm(mu, axis=1, keepdims=True)
    # 1. the band is 0 or exactly one bf16 step of the exact value
    mant, ex = np.frexp(xe)
    step = np.ldexp(np.ones_like(xe), ex - 8)
    assert np.all((amb == 0) | np.isclose(amb, step, rtol=0, atol=0) | np.isclose(amb, step / 2, rtol=0, atol=0))
    # 2. non-zero exactly where the exact value is within rel of a midpoint
    #    (strictly inside, or strictly outside by a margin: skip the knife edge)
    t = mant * 256.0
    dist = np.abs(t - (np.floor(t) + 0.5)) / np.abs(t)   # relative distance to the midpoint
    inside, outside = dist < rel * 0.999, dist > rel * 1.001
    assert np.all(amb[inside] > 0) and np.all(amb[outside] == 0)
    assert inside.sum() >= 50 and outside.sum() >= 1000
    # 3. every float32 normalisation and every perturbation within rel rounds
    #    to the exact rounding or to the other side of the band
    for x32 in _f32_normalisations(mu):
        got = m.round_to_bf16(x32.astype(np.float64))
        assert np.all(np.abs(got - mh) <= amb), np.abs(got - mh)[np.abs(got - mh) > amb][:5]
    for k in range(-16, 17):
        got = m.round_to_bf16(xe * (1.0 + rel * k / 16.0))
        assert np.all(np.abs(got - mh) <= amb)
    # 4. far from midpoints, the band is empty (float64 operands: always empty)
    assert not m.normalize_centroids(mu, "f64")[1].any()


def pin_objective_hand_value(m):
    """J = sum_i (1 - cos(k_i, mu_c(i))) on a hand-computed example: k = (1,0),
    (0,1), (1,1), (0,0) with labels 0, 0, 1, 1 and centroids (3,0), (0,2):
    cosines 1, 0, 1/sqrt(2) and 0 (a zero key), so J = 3 - 1/sqrt(2)."""
    keys = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [0.0, 0.0]])
    labels = np.array([0, 0, 1, 1], dtype=np.int32)
    mu = np.array([[3.0, 0.0], [0.0, 2.0]])
    assert abs(m.objective(keys, labels, mu) - (3.0 - 1.0 / math.sqrt(2.0))) < 1e-15
    # perfect clusters: J = 0; opposite centroid: D = 2
    assert m.objective(keys[:1], labels[:1], mu) == 0.0
    assert abs(m.objective(np.array([[-1.0, 0.0]]), np.array([0], dtype=np.int32), mu) - 2.0) < 1e-15


PINS = [pin_selection_worked_example, pin_cluster_count, pin_bf16_rounding,
        pin_assign_vs_scipy_cosine, pin_assign_brute_force, pin_update_closed_form,
        pin_update_is_mean_logit, pin_planted_partition,
        pin_one_token_per_cluster_is_exact_top_b, pin_selection_vs_token_sort,
        pin_attention_vs_torch_sdpa, pin_assignment_never_increases_objective,
        pin_recall_properties, pin_append_clusters, pin_attention_tokens_with_pending,
        pin_rounding_band, pin_objective_hand_value]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(ck)


# the same pins against the C++ oracle (the recall helpers are measurement
# code of the numpy oracle only)
@pytest.mark.parametrize("pin", [p for p in PINS if p is not pin_recall_properties], ids=lambda f: f.__name__)
def test_cpp_oracle_pin(pin):
    pin(cc)


# ----------------------------------------------------------------------------
# planted mistakes: a copy of the oracle with one plausible error must fail a pin
# ----------------------------------------------------------------------------
def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("ck_mutant", ck.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_argmin(mod):
    mod.assign = lambda keys, mu_hat: np.argmin(mod.cosine_to_centroids(keys, mu_hat), axis=1).astype(np.int32)


def _mut_sum_update(mod):
    def update(keys, labels, mu_old):
        mu = np.array(mu_old, dtype=np.float64, copy=True)
        for c in range(mu.shape[0]):
            if (labels == c).any():
                mu[c] = np.asarray(keys, dtype=np.float64)[labels == c].sum(axis=0)
        return mu
    mod.update = update


def _mut_normalised_mean(mod):
    def update(keys, labels, mu_old):
        k = np.asarray(keys, dtype=np.float64)
        k = k / np.linalg.norm(k, axis=1, keepdims=True)
        mu = np.array(mu_old, dtype=np.float64, copy=True)
        for c in range(mu.shape[0]):
            if (labels == c).any():
                mu[c] = k[labels == c].mean(axis=0)
        return mu
    mod.update = update


def _mut_no_trim(mod):
    def select(scores, sizes, offsets, perm, B):
        out = []
        for c in mod.rank_clusters(scores):
            if len(out) >= B:
                break
            out.extend(int(t) for t in perm[offsets[c]:offsets[c] + sizes[c]])
        return np.asarray(out, dtype=np.int32), len(out)
    mod.select = select


def _mut_ascending_rank(mod):
    mod.rank_clusters = lambda s: np.lexsort((np.arange(len(s)), np.asarray(s, dtype=np.float64)))


def _mut_no_scale(mod):
    orig = mod.sparse_attention
    mod.sparse_attention = lambda q, K, V, t: orig(np.asarray(q) * math.sqrt(np.atleast_2d(q).shape[1]), K, V, t)


def _mut_cosine_score(mod):
    def score(q, mu):
        q = np.atleast_2d(np.asarray(q, dtype=np.float64))
        mu = np.asarray(mu, dtype=np.float64)
        return (q @ (mu / np.linalg.norm(mu, axis=1, keepdims=True)).T).sum(axis=0)
    mod.score = score


def _mut_seed_stride_one(mod):
    mod.seed_stride = lambda n, C, ratio=80: 1


def _mut_transposed_dot(mod):
    """A wrong index mapping: centroid c scored with the row of centroid C-1-c."""
    def cosine_to_centroids(keys, mu_hat):
        k = np.asarray(keys, dtype=np.float64)
        dots = k @ np.asarray(mu_hat, dtype=np.float64)[::-1].T
        nrm = np.sqrt(np.sum(k * k, axis=1, keepdims=True))
        return np.divide(dots, nrm, out=np.zeros_like(dots), where=nrm > 0)
    mod.cosine_to_centroids = cosine_to_centroids


def _mut_bf16_truncate(mod):
    def round_to_bf16(x):
        m_, e = np.frexp(np.asarray(x, dtype=np.float64))
        return np.ldexp(np.trunc(m_ * 256.0), e - 8)
    mod.round_to_bf16 = round_to_bf16


def _mut_pending_past_end(mod):
    def attention_tokens(sinks, clustered_end, cur_len, idx):
        return np.concatenate([np.arange(sinks), np.arange(clustered_end, cur_len + 1),
                               np.asarray(idx, dtype=np.int64)]).astype(np.int64)
    mod.attention_tokens = attention_tokens


def _mut_pending_from_one_early(mod):
    def attention_tokens(sinks, clustered_end, cur_len, idx):
        return np.concatenate([np.arange(sinks), np.arange(clustered_end - 1, cur_len),
                               np.asarray(idx, dtype=np.int64)]).astype(np.int64)
    mod.attention_tokens = attention_tokens


def _mut_pending_dropped(mod):
    def attention_tokens(sinks, clustered_end, cur_len, idx):
        return np.concatenate([np.arange(sinks), np.asarray(idx, dtype=np.int64)]).astype(np.int64)
    mod.attention_tokens = attention_tokens


def _mut_band_too_wide(mod):
    orig = mod.normalize_centroids
    mod.normalize_centroids = lambda mu, operand="bf16", rel_err=2.0 ** -20: orig(mu, operand, 2.0 ** -12)


def _mut_band_missing(mod):
    orig = mod.normalize_centroids
    mod.normalize_centroids = lambda mu, operand="bf16", rel_err=2.0 ** -20: (
        orig(mu, operand, rel_err)[0], np.zeros_like(np.asarray(mu, dtype=np.float64)))


def _mut_band_two_steps(mod):
    orig = mod.normalize_centroids
    mod.normalize_centroids = lambda mu, operand="bf16", rel_err=2.0 ** -20: (
        orig(mu, operand, rel_err)[0], 2.0 * orig(mu, operand, rel_err)[1])


def _mut_objective_offset(mod):
    orig = mod.objective
    mod.objective = lambda keys, labels, mu: orig(keys, labels, mu) + 1.0


def _mut_objective_plus_cos(mod):
    def objective(keys, labels, mu):
        mu_hat, _ = mod.normalize_centroids(mu, "f64")
        cos = mod.cosine_to_centroids(keys, mu_hat)
        return float(np.sum(1.0 + cos[np.arange(len(labels)), labels]))
    mod.objective = objective


MUTANTS = [_mut_argmin, _mut_sum_update, _mut_normalised_mean, _mut_no_trim,
           _mut_ascending_rank, _mut_no_scale, _mut_cosine_score, _mut_seed_stride_one,
           _mut_transposed_dot, _mut_bf16_truncate, _mut_pending_past_end, _mut_pending_from_one_early,
           _mut_pending_dropped, _mut_band_too_wide, _mut_band_missing, _mut_band_two_steps,
           _mut_objective_offset, _mut_objective_plus_cos]


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda f: f.__name__)
def test_mutant_caught(mutate):
    mod = _fresh_oracle()
    mutate(mod)
    failed = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception:  # a failed check, or a crash on the planted mistake
            failed.append(pin.__name__)
    assert failed, f"no pin caught {mutate.__name__}"
