"""Pins of the reuse oracle against what the ClusterKV page and plain set
arithmetic fix: a selection repeated from the previous step is all hits, a
disjoint one none, the R = 2 count obeys inclusion-exclusion over the two
previous selections, and a hand-worked example."""
import numpy as np

import oracle.clusterkv as ck
import oracle.reuse as ro


def test_identical_and_disjoint():
    a = [5, 9, 17, 18, 40]
    assert ro.selection_hits([a], a) == 5
    assert ro.selection_hits([[1, 2, 3]], [4, 5, 6]) == 0
    assert ro.selection_hits([], a) == 0


def test_hand_example():
    # step t-2 took clusters {A: 20, 21} and {B: 30}; step t-1 took {B: 30} and
    # {C: 40, 41}; step t takes {B: 30}, {A: 20, 21} and {D: 50}
    prev2, prev1, cur = [20, 21, 30], [30, 40, 41], [30, 20, 21, 50]
    assert ro.selection_hits([prev1], cur) == 1          # R = 1: only B
    assert ro.selection_hits([prev2, prev1], cur) == 3   # R = 2: B and A
    assert np.isclose(ro.hit_rate([prev2, prev1, cur], 1), (1 / 3 + 1 / 4) / 2)


def test_inclusion_exclusion_and_monotone():
    rng = np.random.default_rng(3)
    for _ in range(20):
        p1 = rng.choice(200, 60, replace=False)
        p2 = rng.choice(200, 60, replace=False)
        cur = rng.choice(200, 70, replace=False)
        both = np.intersect1d(p1, p2)
        h1, h2 = ro.selection_hits([p1], cur), ro.selection_hits([p2], cur)
        h12 = ro.selection_hits([both], cur)
        assert ro.selection_hits([p1, p2], cur) == h1 + h2 - h12
        assert ro.selection_hits([p1, p2], cur) >= max(h1, h2)
        assert ro.selection_hits([p1, p2], cur) <= len(cur)


def test_whole_cluster_selections_hit_by_cluster():
    # selections made by the oracle's own cluster selection: when the same
    # clusters rank first at two steps, every token of the second is a hit
    rng = np.random.default_rng(4)
    labels = rng.integers(0, 12, size=300)
    sizes, offsets, perm = ck.build_csr(labels, 12, 16)
    s1 = rng.standard_normal(12)
    s2 = s1 + 1e-3 * rng.standard_normal(12)   # same order with a tiny perturbation
    assert (np.argsort(-s1, kind="stable") == np.argsort(-s2, kind="stable")).all()
    i1, c1 = ck.select(s1, sizes, offsets, perm, 80)
    i2, c2 = ck.select(s2, sizes, offsets, perm, 80)
    assert ro.selection_hits([i1[:c1]], i2[:c2]) == c2
