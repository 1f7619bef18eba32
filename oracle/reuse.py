"""Plain CPU oracle for the reuse measurement of earlier selections.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports, links or calls this
module; only ``tests/`` and the CPU-baseline leg of ``bench.py`` may.

Source: "ClusterKV: Manipulating LLM KV Cache in Semantic Space for Recallable
Compression" (papercache summary page, arXiv 2412.03213), section "Caching the
KV of selected tokens": the GPU keeps the KV of the tokens selected in the last
R decode steps together with the labels of their clusters; at a new step only
the selected clusters missing from that cache are loaded.  The page's cache
effectiveness analysis reports the hit rate for R = 1 and R = 2.

Reading (also listed with the other readings): the hit count of a step is the
number of tokens of its selection that were selected in at least one of the R
previous steps.  Selections are made of whole clusters (the last one trimmed),
so this is the token-weighted cluster hit rate: the share of the step's K/V
bytes that the cache would already hold.
"""
from __future__ import annotations

import numpy as np


def selection_hits(prev_sets, cur) -> int:
    """Tokens of ``cur`` (a sequence of token ids) present in the union of the
    sequences in ``prev_sets``."""
    cached = set()
    for s in prev_sets:
        cached.update(int(t) for t in s)
    return sum(1 for t in cur if int(t) in cached)


def hit_rate(history, R: int) -> float:
    """Mean over steps t >= R of selection_hits(history[t-R:t], history[t]) /
    len(history[t]) for a list of per-step selections of one unit."""
    rates = []
    for t in range(R, len(history)):
        n = len(history[t])
        if n:
            rates.append(selection_hits(history[t - R:t], history[t]) / n)
    return float(np.mean(rates)) if rates else 0.0
