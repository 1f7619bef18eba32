"""Plain CPU oracle for the channel pre-score over the centroid table.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports, links or calls this
module; only ``tests/`` and the CPU-baseline leg of ``bench.py`` may.

Source: "TailorKV: A Hybrid Framework for Long-Context Inference via Tailored
KV Cache Optimization" (papercache summary page), dynamic retrieval for
sparsity-friendly layers: the contribution of channel i is
s_i = |q_i| * max |K_i|, and attention scores are approximated from the few
channels of largest contribution (8 or 12 in the page's settings).

Reading (also listed with the other readings): applied to ClusterKV's centroid
scoring, q is the sum of the g query heads (the exact cluster score sums q_h .
mu), K is the centroid table, and the approximate score of cluster c is the
dot product of q and mu_c over the r channels of largest s_i (ties: lower
channel).  The ranking is an integer decision taken from floating point, so
it is made as the kernel makes it: the head sum and the product in fp32 from
the bf16 (or fp32) inputs; the scores themselves are computed in fp64.
"""
from __future__ import annotations

import numpy as np


def channel_max(mu: np.ndarray) -> np.ndarray:
    """max over clusters of |mu_c,i| for every channel i (mu [C, d])."""
    return np.abs(np.asarray(mu, dtype=np.float64)).max(axis=0)


def head_sum_f32(q: np.ndarray) -> np.ndarray:
    """sum over the heads of q [g, d] in fp32, heads in order."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float32))
    acc = np.zeros(q.shape[1], dtype=np.float32)
    for qh in q:
        acc = (acc + qh).astype(np.float32)
    return acc


def critical_channels(q: np.ndarray, mu: np.ndarray, r: int) -> np.ndarray:
    """The r channels of largest s_i = |qs_i| * max_c |mu_c,i|, descending, ties
    to the lower channel (s in fp32 as the kernel forms it)."""
    qs = head_sum_f32(q)
    s = (np.abs(qs) * channel_max(mu).astype(np.float32)).astype(np.float32)
    order = sorted(range(len(s)), key=lambda i: (-float(s[i]), i))
    return np.array(order[:r], dtype=np.int64)


def prescore(q: np.ndarray, mu: np.ndarray, r: int):
    """(scores [C], channels [r]): score_c = sum over the r critical channels of
    qs_i * mu_c,i, in fp64."""
    ch = critical_channels(q, mu, r)
    qs = head_sum_f32(q).astype(np.float64)
    mu = np.asarray(mu, dtype=np.float64)
    return mu[:, ch] @ qs[ch], ch
