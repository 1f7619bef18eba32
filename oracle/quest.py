"""Plain CPU oracle for the page-granular selection that the ClusterKV page
compares against (Quest).

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports, links or calls this
module; only ``tests/`` and the CPU-baseline leg of ``bench.py`` may.

Source: "ClusterKV: Manipulating LLM KV Cache in Semantic Space for Recallable
Compression" (papercache summary page, arXiv 2412.03213), section "Background
and design principles" (drawbacks of existing recallable compression): Quest
selects tokens at the granularity of pages of consecutive tokens, scoring each
page with the per-channel maximum key of its tokens, at cost O(L d /
page_size); its pages (page_size = 16 in the page's Fig. 3b) suffer internal
fragmentation.

Reading (also listed with the other readings): a page's weight is the upper
bound of q . k over its tokens, sum_i max(q_i * max_i, q_i * min_i) with the
per-channel maximum and minimum keys of the page (the per-channel maximum alone
is not a bound where q_i < 0).  Grouped-query attention sums the bound over the
g query heads, as the cluster score sums q_h . mu.  Pages cover the clustered
token range [sinks, L) from its start; the last page may be short.  Pages are
taken whole in descending weight order (ties: lower page index) up to the
budget B, the last one trimmed, exactly as clusters are (the selection of
``clusterkv.select`` with one "cluster" per page).
"""
from __future__ import annotations

import numpy as np

from . import clusterkv as ck

PAGE = 16


def page_bounds(keys: np.ndarray, page: int = PAGE):
    """Per-page, per-channel maximum and minimum of the keys [n, d] (the
    clustered tokens in order).  Returns (kmax [P, d], kmin [P, d])."""
    keys = np.asarray(keys, dtype=np.float64)
    n = len(keys)
    P = (n + page - 1) // page
    kmax = np.empty((P, keys.shape[1]))
    kmin = np.empty((P, keys.shape[1]))
    for p in range(P):
        block = keys[p * page:min(n, (p + 1) * page)]
        kmax[p] = block.max(axis=0)
        kmin[p] = block.min(axis=0)
    return kmax, kmin


def page_scores(q: np.ndarray, kmax: np.ndarray, kmin: np.ndarray) -> np.ndarray:
    """sum over heads h and channels i of max(q_hi * max_pi, q_hi * min_pi)."""
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    s = np.zeros(len(kmax))
    for qh in q:
        s += np.maximum(kmax * qh, kmin * qh).sum(axis=1)
    return s


def page_csr(n: int, page: int = PAGE, token_base: int = 0):
    """The pages as clusters: sizes, offsets and the identity permutation."""
    P = (n + page - 1) // page
    sizes = np.array([min(page, n - p * page) for p in range(P)], dtype=np.int32)
    offsets = np.zeros(P + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(sizes)
    perm = (np.arange(n) + token_base).astype(np.int32)
    return sizes, offsets, perm


def select_pages(scores: np.ndarray, n: int, B: int, page: int = PAGE, token_base: int = 0):
    """Whole pages in descending score order up to B tokens, the last trimmed.
    Returns (idx, count) like ``clusterkv.select``."""
    sizes, offsets, perm = page_csr(n, page, token_base)
    return ck.select(scores, sizes, offsets, perm, B)
