"""Seeded synthetic workloads shaped like ClusterKV's evaluation setting.

This module only draws random numbers.  It holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle may take their inputs from
it.  Shapes follow the Llama-3.1-8B attention layout used in the ClusterKV
efficiency experiments (section "Experiments": 32 layers, 8 KV heads, GQA 4:1,
head dim 128, 32k prompts, 1024 decode steps, budget 1k-2k).  The page's
datasets are not used: keys are drawn from a mixture of random unit centres with
Gaussian noise and a few large outlier channels (the page motivates the cosine
distance by such channels, section "Clustering in semantic space").

A unit is one (sequence, layer, KV head).  Every unit draws from its own
``torch.Generator`` seeded from (workload seed, purpose, unit), so any subset of
units can be regenerated on its own.  CPU and CUDA generators give different
streams: parity tests draw on the CPU and upload the very same tensors.
"""
from __future__ import annotations

import dataclasses
import hashlib

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    units: int            # (sequence, layer, KV head) triples
    g: int                # query heads per KV head
    L: int                # prompt length (tokens)
    decode_steps: int     # decode steps after the prompt
    C: int                # prefill clusters per unit
    B: int                # token budget
    dtype: str            # "f32" or "bf16" for K, V and q
    n_centres: int        # mixture centres per unit
    centre_scale: float   # key = centre_scale * centre + sigma * noise
    sigma: float
    n_outlier: int        # outlier channels per unit (scaled after drawing)
    outlier_scale: float
    zipf: float = 0.0     # 0: uniform centre weights, else Zipf exponent
    q_scale: float = 3.0  # query = q_scale * centre + q_sigma * noise
    q_sigma: float = 0.5
    n_queries: int = 1    # independent queries per unit for select/attend tests
    iters: int = 10
    d: int = 128
    sinks: int = 16
    m: int = 320
    c_plus: int = 4
    seed: int = 0
    layers: int = 1
    kv_heads: int = 1
    batch: int = 1

    @property
    def max_len(self) -> int:
        return self.L + self.decode_steps

    @property
    def n_incremental(self) -> int:
        # clustering runs before decode steps m, 2m, ... (never before step 0)
        return max(0, (self.decode_steps - 1) // self.m)

    @property
    def max_clusters(self) -> int:
        return self.C + self.c_plus * self.n_incremental

    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The five workloads: a tiny single-head case, one Llama-3.1-8B layer at 32k,
# the 32-layer 32k decode loop, a batch-16 decode and a 128k stress case.
WORKLOADS = {
    "tiny_2k": Workload("tiny_2k", units=1, g=1, L=2048, decode_steps=0, C=25, B=256,
                        dtype="f32", n_centres=25, centre_scale=3.0, sigma=1.0,
                        n_outlier=4, outlier_scale=20.0, q_scale=3.0, q_sigma=0.3,
                        n_queries=8, seed=20241204, kv_heads=1),
    "layer_32k": Workload("layer_32k", units=8, g=4, L=32768, decode_steps=0, C=409, B=1024,
                          dtype="bf16", n_centres=409, centre_scale=1.0, sigma=0.3,
                          n_outlier=4, outlier_scale=20.0, seed=20241205, kv_heads=8),
    "decode_32k": Workload("decode_32k", units=256, g=4, L=32768, decode_steps=1024, C=409,
                           B=1024, dtype="bf16", n_centres=409, centre_scale=1.0, sigma=0.3,
                           n_outlier=4, outlier_scale=20.0, seed=20241206, layers=32,
                           kv_heads=8),
    "batch16_32k": Workload("batch16_32k", units=4096, g=4, L=32768, decode_steps=256, C=409,
                            B=2048, dtype="bf16", n_centres=409, centre_scale=1.0, sigma=0.3,
                            n_outlier=4, outlier_scale=20.0, seed=20241207, layers=32,
                            kv_heads=8, batch=16),
    "long_128k": Workload("long_128k", units=1024, g=4, L=131072, decode_steps=128, C=1638,
                          B=2048, dtype="bf16", n_centres=1638, centre_scale=1.0, sigma=0.3,
                          n_outlier=8, outlier_scale=30.0, zipf=1.1, seed=20241208,
                          layers=32, kv_heads=8, batch=4),
}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some fields changed (smaller test cases)."""
    return dataclasses.replace(w, **changes)


def _seed(*parts) -> int:
    h = hashlib.blake2b(repr(parts).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 62) - 1)


def _gen(w: Workload, purpose: str, unit: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(w.seed, purpose, unit))
    return g


def unit_structure(w: Workload, unit: int, device="cpu"):
    """Per-unit mixture: centres [n_centres, d] (unit vectors), centre weights
    [n_centres] and outlier channel ids [n_outlier]."""
    g = _gen(w, "structure", unit, device)
    c = torch.randn(w.n_centres, w.d, generator=g, device=device, dtype=torch.float32)
    c = c / c.norm(dim=1, keepdim=True)
    if w.zipf > 0:
        ranks = torch.arange(1, w.n_centres + 1, device=device, dtype=torch.float64)
        wts = ranks.pow(-w.zipf)
        wts = (wts / wts.sum()).to(torch.float32)
    else:
        wts = torch.full((w.n_centres,), 1.0 / w.n_centres, device=device)
    out = torch.randperm(w.d, generator=g, device=device)[: w.n_outlier]
    return c, wts, out


def unit_keys(w: Workload, unit: int, device="cpu", structure=None) -> torch.Tensor:
    """Keys of tokens [0, max_len) of one unit, in the workload dtype."""
    c, wts, out = structure if structure is not None else unit_structure(w, unit, device)
    g = _gen(w, "keys", unit, device)
    T = w.max_len
    if w.zipf > 0:
        z = torch.multinomial(wts, T, replacement=True, generator=g)
    else:
        z = torch.randint(0, w.n_centres, (T,), generator=g, device=device)
    noise = torch.randn(T, w.d, generator=g, device=device, dtype=torch.float32)
    k = c[z] * w.centre_scale + noise * w.sigma
    k[:, out] = k[:, out] * w.outlier_scale
    return k.to(w.torch_dtype())


def unit_values(w: Workload, unit: int, device="cpu") -> torch.Tensor:
    """Values of tokens [0, max_len) of one unit: N(0, 1)."""
    g = _gen(w, "values", unit, device)
    v = torch.randn(w.max_len, w.d, generator=g, device=device, dtype=torch.float32)
    return v.to(w.torch_dtype())


def unit_queries(w: Workload, unit: int, n: int, device="cpu", structure=None, topic_run: int = 1) -> torch.Tensor:
    """``n`` query groups [n, g, d] of one unit: every group picks one random
    centre j and its g heads are q_h = q_scale * c_j + q_sigma * noise.  With
    topic_run > 1 each drawn centre is kept for topic_run consecutive groups
    (fresh noise every group)."""
    c, _, _ = structure if structure is not None else unit_structure(w, unit, device)
    g = _gen(w, "queries", unit, device)
    j = torch.randint(0, w.n_centres, (n,), generator=g, device=device)
    if topic_run > 1:
        j = j[(torch.arange(n, device=device) // topic_run) * topic_run]
    noise = torch.randn(n, w.g, w.d, generator=g, device=device, dtype=torch.float32)
    q = c[j][:, None, :] * w.q_scale + noise * w.q_sigma
    return q.to(w.torch_dtype())


def make_kv(w: Workload, units=None, device="cpu"):
    """K, V [len(units), max_len, d] for the given units (default: all)."""
    units = range(w.units) if units is None else units
    units = list(units)
    K = torch.empty(len(units), w.max_len, w.d, dtype=w.torch_dtype(), device=device)
    V = torch.empty_like(K)
    for i, u in enumerate(units):
        s = unit_structure(w, u, device)
        K[i] = unit_keys(w, u, device, s)
        V[i] = unit_values(w, u, device)
    return K, V


def make_queries(w: Workload, n: int, units=None, device="cpu", topic_run: int = 1) -> torch.Tensor:
    """Queries [n, len(units), g, d]: ``n`` query groups per unit (a new random
    centre every group, or every topic_run groups)."""
    units = list(range(w.units) if units is None else units)
    Q = torch.empty(n, len(units), w.g, w.d, dtype=w.torch_dtype(), device=device)
    for i, u in enumerate(units):
        Q[:, i] = unit_queries(w, u, n, device, topic_run=topic_run)
    return Q
