"""Shared helpers of the GPU parity tests: building library contexts from
seeded inputs, uploading oracle state, and the acceptance rules.

Acceptance (per part):
  * assignment, given identical fp32 centroids: labels bit-exact, except rows
    whose two best oracle cosines lie within the floating-point band below of
    each other, where the GPU label must be one of the labels within the band;
  * update, given identical labels: sizes, offsets, perm bit-exact; centroids
    within 1e-5 relative (max |d mu_c| <= 1e-5 * max |mu_c| per centroid);
  * scores: |d| <= 2^-8 * sum_h sum_j |q_hj mu_cj| (bf16 operand copy of mu),
    2^-16 * the same sum for fp32;
  * selection, given identical fp32 scores: idx and count bit-exact;
  * attention, given identical idx: max abs error 2e-3 (bf16 K/V), 1e-5 (fp32).

The assignment band: the GPU accumulates 128 exact bf16 x bf16 products in
fp32 (tensor cores) and normalises the centroids in fp32 before rounding them
to bf16.  Its dot for (key i, centroid c) differs from the exact one by at most
EPS * S_ic + A_ic, where S_ic = sum_j |k_ij mu_hat_cj| and A_ic = sum_j |k_ij| *
amb_cj (amb = rounding steps where fp32 normalisation may round the other way,
from the oracle).  EPS = 2^-14 is 8x the bound of sequential fp32 summation of
128 terms (127 * 2^-24 < 2^-17).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.clusterkv as ck
from recallable_kv_cache_gb300 import ckv

EPS_BF16 = 2.0 ** -14
EPS_F32 = 2.0 ** -16
ATTN_TOL = {"bf16": 2e-3, "f32": 1e-5}


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def make_ctx(units, g, max_len, max_clusters, max_budget, dtype, iters=10, m=320, c_plus=4, ratio=80):
    return ckv.Context(units=units, g=g, max_len=max_len, max_clusters=max_clusters,
                       max_budget=max_budget, kv_dtype=dtype, iters=iters, m=m, c_plus=c_plus,
                       ratio=ratio)


def check_assignment(keys: np.ndarray, mu32: np.ndarray, labels_gpu: np.ndarray, operand: str):
    """Compare GPU labels with the oracle's arg-max for the same fp32 centroids.
    Returns (n_rows, n_near_tie_rows)."""
    mu_hat, amb = ck.normalize_centroids(mu32.astype(np.float64), operand)
    cos = ck.cosine_to_centroids(keys, mu_hat)
    lab_o = ck.assign(keys, mu_hat)
    eps = EPS_BF16 if operand == "bf16" else EPS_F32
    ak = np.abs(keys)
    nrm = np.sqrt(np.sum(keys * keys, axis=1, keepdims=True))
    nrm[nrm == 0] = 1.0
    err = (eps * (ak @ np.abs(mu_hat).T) + ak @ amb.T) / nrm
    rows = np.arange(len(keys))
    top = cos[rows, lab_o]
    band = err + err[rows, lab_o][:, None]
    within = (top[:, None] - cos) <= band          # labels the GPU may legitimately pick
    near = within.sum(axis=1) > 1
    exact_ok = labels_gpu[~near] == lab_o[~near]
    assert exact_ok.all(), (
        f"{(~exact_ok).sum()} rows differ outside the tie band; first: "
        f"{np.flatnonzero(~near)[~exact_ok][:5]}")
    ok_near = within[rows[near], labels_gpu[near]]
    assert ok_near.all(), "a near-tie row took a label outside the band"
    return len(keys), int(near.sum())


def check_centroids(mu_gpu: np.ndarray, mu_ref: np.ndarray, rel=1e-5):
    scale = np.maximum(np.abs(mu_ref).max(axis=-1, keepdims=True), 1e-30)
    worst = (np.abs(mu_gpu - mu_ref) / scale).max()
    assert worst <= rel, f"centroid relative error {worst:.3e} > {rel}"
    return float(worst)


def score_tol(q: np.ndarray, mu: np.ndarray, dtype: str) -> np.ndarray:
    """Per-cluster bound |score_gpu - score_exact| for q [g, d], mu [C, d]."""
    eps = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -16
    return eps * (np.abs(mu) @ np.abs(q).sum(axis=0)) + 1e-30


def upload_state(ctx: ckv.Context, states: list[dict], clustered_end: int, device="cuda"):
    """Import per-unit oracle cluster state (mu, sizes, offsets, perm) into ctx."""
    C = len(states[0]["sizes"])
    mu = torch.tensor(np.stack([s["mu"] for s in states]), dtype=torch.float32, device=device)
    sizes = torch.tensor(np.stack([s["sizes"] for s in states]), dtype=torch.int32, device=device)
    offs = torch.tensor(np.stack([s["offsets"] for s in states]), dtype=torch.int32, device=device)
    perm = torch.tensor(np.stack([s["perm"] for s in states]), dtype=torch.int32, device=device)
    ctx.import_clusters(C, clustered_end, mu.contiguous(), sizes.contiguous(), offs.contiguous(),
                        perm.contiguous())
    torch.cuda.synchronize()
    return mu


def export_state(ctx: ckv.Context, units: int, d: int = 128, dtype: str = "bf16"):
    inf = ctx.info()
    C, np_ = inf.n_clusters, inf.clustered_end - 16
    mu = torch.empty(units, C, d, dtype=torch.float32, device="cuda")
    mh = torch.empty(units, C, d, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                     device="cuda")
    sizes = torch.empty(units, C, dtype=torch.int32, device="cuda")
    offs = torch.empty(units, C + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(units, max(np_, 1), dtype=torch.int32, device="cuda")
    ctx.export_clusters(mu, mh, sizes, offs, perm)
    torch.cuda.synchronize()
    return dict(mu=mu.cpu().numpy().astype(np.float64), mu_hat=mh.float().cpu().numpy(),
                sizes=sizes.cpu().numpy(), offsets=offs.cpu().numpy(),
                perm=perm.cpu().numpy()[:, :np_])


def host_mapped(t: torch.Tensor) -> bool:
    """True when the pinned host tensor t is addressable by kernels at its host
    address (unified addressing); checked with cudaHostGetDevicePointer."""
    import ctypes
    path = None
    for line in open("/proc/self/maps"):
        if "libcudart" in line:
            path = line.split()[-1]
            break
    rt = ctypes.CDLL(path or "libcudart.so")
    rt.cudaHostGetDevicePointer.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p, ctypes.c_uint]
    rt.cudaHostGetDevicePointer.restype = ctypes.c_int
    d = ctypes.c_void_p()
    return rt.cudaHostGetDevicePointer(ctypes.byref(d), ctypes.c_void_p(t.data_ptr()), 0) == 0 and \
        d.value == t.data_ptr()
