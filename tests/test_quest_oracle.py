"""Pins of the page-granular (Quest) oracle against what the ClusterKV page and
the mathematics fix: the page weight bounds every token's weight in the page,
pages of one token reduce to the exact top-B, and a hand-worked example."""
import numpy as np

import oracle.clusterkv as ck
import oracle.quest as qo


def test_page_weight_bounds_every_token():
    rng = np.random.default_rng(7)
    keys = rng.standard_normal((16 * 9 + 5, 32))
    q = rng.standard_normal((3, 32))
    kmax, kmin = qo.page_bounds(keys)
    s = qo.page_scores(q, kmax, kmin)
    w = (q @ keys.T).sum(axis=0)
    for p in range(len(s)):
        block = w[p * 16:(p + 1) * 16]
        assert block.max() <= s[p] + 1e-9
    assert len(kmax) == 10  # nine full pages and one of five tokens
    # a page of one token: the bound is that token's weight
    s1 = qo.page_scores(q, *qo.page_bounds(keys[:1], page=1))
    assert np.isclose(s1[0], w[0])


def test_pages_of_one_token_are_the_exact_top_b():
    rng = np.random.default_rng(8)
    n, d, B = 300, 16, 37
    keys = rng.standard_normal((n, d))
    q = rng.standard_normal((4, d))
    kmax, kmin = qo.page_bounds(keys, page=1)
    s = qo.page_scores(q, kmax, kmin)
    idx, c = qo.select_pages(s, n, B, page=1, token_base=16)
    K = np.vstack([np.zeros((16, d)), keys])
    want = ck.exact_top_b(q, K, np.arange(16, 16 + n), B)
    assert c == B
    assert np.array_equal(idx, want)


def test_hand_example():
    # two pages of two tokens in 2-d, one query head q = (1, -1):
    # page 0 holds (1, 0), (0, 1): max (1, 1), min (0, 0): bound 1*1 + (-1)*0 = 1
    # page 1 holds (2, 3), (-1, -2): max (2, 3), min (-1, -2): bound 2 + 2 = 4
    keys = np.array([[1.0, 0.0], [0.0, 1.0], [2.0, 3.0], [-1.0, -2.0]])
    kmax, kmin = qo.page_bounds(keys, page=2)
    s = qo.page_scores(np.array([1.0, -1.0]), kmax, kmin)
    assert np.allclose(s, [1.0, 4.0])
    idx, c = qo.select_pages(s, 4, 3, page=2, token_base=16)
    # page 1 first (tokens 18, 19), then page 0 trimmed to one token (16)
    assert c == 3 and list(idx) == [18, 19, 16]
