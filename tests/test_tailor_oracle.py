"""Pins of the channel pre-score oracle against what the TailorKV page and the
mathematics fix: with every channel kept it is the exact cluster score of the
ClusterKV oracle; the page's contribution |q_i| * max |K_i| ranks a hand-built
example as expected (including a channel with a large query but small keys);
the dropped channels bound the error."""
import numpy as np

import oracle.clusterkv as ck
import oracle.tailor as to


def test_all_channels_is_the_exact_score():
    rng = np.random.default_rng(11)
    # eighths: the fp32 head sum is exact, so only the fp64 dot products remain
    q = rng.integers(-64, 64, size=(4, 16)) / 8.0
    mu = rng.standard_normal((30, 16))
    sc, ch = to.prescore(q, mu, 16)
    assert sorted(ch.tolist()) == list(range(16))
    assert np.allclose(sc, ck.score(q, mu), rtol=1e-12, atol=1e-12)


def test_hand_example_ranking():
    # one head, 4 channels; contributions |q_i| * max_c |mu_c,i|:
    #   ch0: 1 * 3 = 3,  ch1: 10 * 0.1 = 1,  ch2: 2 * 2 = 4,  ch3: 0.5 * 6 = 3
    q = np.array([[1.0, -10.0, 2.0, 0.5]])
    mu = np.array([[3.0, 0.1, -2.0, 1.0],
                   [-1.0, 0.0, 1.0, -6.0]])
    ch = to.critical_channels(q, mu, 4)
    assert ch.tolist() == [2, 0, 3, 1]          # 4, then the tie 3 = 3 to the lower channel
    sc, ch2 = to.prescore(q, mu, 2)
    assert ch2.tolist() == [2, 0]
    assert np.allclose(sc, [2.0 * -2.0 + 1.0 * 3.0, 2.0 * 1.0 + 1.0 * -1.0])


def test_dropped_channels_bound_the_error():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((4, 32))
    mu = rng.standard_normal((50, 32))
    exact = ck.score(q, mu)
    qs = to.head_sum_f32(q).astype(np.float64)
    for r in (1, 4, 8, 16):
        sc, ch = to.prescore(q, mu, r)
        rest = np.setdiff1d(np.arange(32), ch)
        bound = (np.abs(qs[rest]) * to.channel_max(mu)[rest]).sum()
        assert (np.abs(sc - exact) <= bound + 1e-4).all()
