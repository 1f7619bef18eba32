"""The C++ oracle (oracle/clusterkv_ref.cpp, the timed CPU baseline) against
the numpy oracle, on seeded inputs: integer results (labels, CSR, selected
token ids, counts) bit-exact, float64 results within 1e-12 relative (the two
sum in different orders).  Both are also pinned independently by
tests/test_oracle_pins.py."""
import numpy as np
import pytest

import oracle.clusterkv as ck
import oracle.cpp as cc
from recallable_kv_cache_gb300 import synth


def _close(a, b, rel=1e-12):
    scale = max(np.abs(b).max(), 1e-300)
    assert np.abs(np.asarray(a) - np.asarray(b)).max() <= rel * scale


@pytest.mark.parametrize("operand", ["bf16", "f64"])
@pytest.mark.parametrize("n,C,iters", [(500, 7, 3), (2032, 25, 10), (3000, 37, 4)])
def test_kmeans_matches(operand, n, C, iters):
    rng = np.random.default_rng(n + C)
    centres = rng.standard_normal((C, 128))
    keys = centres[rng.integers(0, C, n)] * 3 + rng.standard_normal((n, 128))
    keys[:, [2, 9]] *= 20
    keys[5] = 0.0  # a zero key
    a = ck.kmeans(keys, C, iters, operand, token_base=16)
    b = cc.kmeans(keys, C, iters, operand, token_base=16)
    for k in ("labels", "sizes", "offsets", "perm"):
        assert np.array_equal(a[k], b[k]), k
    _close(b["mu"], a["mu"])


def test_rounding_band_matches():
    rng = np.random.default_rng(3)
    mu = rng.standard_normal((50, 128)) * rng.uniform(0.1, 10, (50, 1))
    for rel in (2.0 ** -20, 2.0 ** -12):
        a, b = ck.normalize_centroids(mu, "bf16", rel), cc.normalize_centroids(mu, "bf16", rel)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("B", [0, 1, 100, 999, 5000])
def test_score_select_attention_match(B):
    rng = np.random.default_rng(B)
    L, C, d = 16 + 1500, 40, 128
    K = rng.standard_normal((L + 30, d))
    V = rng.standard_normal((L + 30, d))
    st = ck.cluster_prefill(K, L, C, iters=2)
    q = rng.standard_normal((4, d))
    sa, sb = ck.score(q, st["mu"]), cc.score(q, st["mu"])
    _close(sb, sa)
    tied = np.round(sa, 0)  # many ties: rank by cluster index
    for sc in (sa, tied):
        ia, na = ck.select(sc, st["sizes"], st["offsets"], st["perm"], B)
        ib, nb = cc.select(sc, st["sizes"], st["offsets"], st["perm"], B)
        assert na == nb and np.array_equal(ia, ib)
    toks = ck.attention_tokens(16, L, L + 30, ia)
    _close(cc.sparse_attention(q, K, V, toks), ck.sparse_attention(q, K, V, toks))


def test_whole_unit_jobs_match():
    """Whole jobs (prefill clustering, decode steps with an incremental
    clustering) of a few small units on the C++ thread pool against the numpy
    oracle's steps composed the same way."""
    w = synth.scaled(synth.WORKLOADS["layer_32k"], units=3, L=16 + 700, decode_steps=45, C=8, n_centres=8,
                     B=64, m=20, iters=3)
    K, V = synth.make_kv(w)
    Q = synth.make_queries(w, w.decode_steps)
    Ks = [K[u].double().numpy() for u in range(w.units)]
    Vs = [V[u].double().numpy() for u in range(w.units)]
    Qs = [Q[:, u].double().numpy() for u in range(w.units)]
    outs, times = cc.unit_jobs(Ks, Vs, Qs, w.L, w.C, w.B, iters=w.iters, m=w.m, c_plus=w.c_plus, threads=2)
    assert times.shape == (3, 2) and (times >= 0).all()
    for u in range(w.units):
        st = ck.cluster_prefill(Ks[u], w.L, w.C, iters=w.iters)
        end = w.L
        for t in range(w.decode_steps):
            if t > 0 and t % w.m == 0:
                st = ck.append_clusters(st, ck.cluster_incremental(Ks[u], end, w.m, w.c_plus, iters=w.iters))
                end += w.m
            idx, _ = ck.select(ck.score(Qs[u][t], st["mu"]), st["sizes"], st["offsets"], st["perm"], w.B)
            want = ck.sparse_attention(Qs[u][t], Ks[u], Vs[u], ck.attention_tokens(16, end, w.L + t + 1, idx))
            _close(outs[u, t], want)
