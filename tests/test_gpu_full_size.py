"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark uses (every unit of the workload in one call): prefill clustering of
all units, then a lockstep assignment and update, scoring, selection and
attention.  Invariants are checked on every unit (on the device); the oracle
checks sampled units one by one.

  layer_32k    8 units x 32k keys, C = 409, B = 1024
  decode_32k   256 units x 32k keys, C = 409 (+4 per 320 steps), B = 1024
  batch16_32k  4096 units x 32k keys, C = 409, B = 2048 (68.7 GB of K/V)
  long_128k    1024 units x 128k keys, C = 1638, B = 2048 (68.7 GB of K/V)
"""
import numpy as np
import pytest
import torch

import oracle.clusterkv as ck
from parity import ATTN_TOL, check_assignment, check_centroids, score_tol, to64
from recallable_kv_cache_gb300 import ckv, synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLES = {
    "layer_32k": [0, 5],
    "decode_32k": [0, 137, 255],
    "batch16_32k": [0, 2049, 4095],
    "long_128k": [0, 700],
}


@pytest.fixture(scope="module", params=list(SAMPLES))
def full(request):
    name = request.param
    w = synth.WORKLOADS[name]
    torch.cuda.empty_cache()
    K, V = synth.make_kv(w, device="cuda")
    Q = synth.make_queries(w, 2, device="cuda")
    ctx = ckv.Context(units=w.units, g=w.g, max_len=w.max_len, max_clusters=w.max_clusters,
                      max_budget=w.B, iters=w.iters, m=w.m, c_plus=w.c_plus)
    ctx.cluster_prefill(K, w.L, w.C)
    torch.cuda.synchronize()
    assert ctx.device_error() == 0
    d = dict(name=name, w=w, K=K, V=V, Q=Q, ctx=ctx, samples=SAMPLES[name])
    yield d
    ctx.close()
    d.clear()
    del K, V, Q
    torch.cuda.empty_cache()


def export_device(ctx, w):
    """Cluster state of every unit, left on the device."""
    inf = ctx.info()
    C, n = inf.n_clusters, inf.clustered_end - w.sinks
    st = dict(mu=torch.empty(w.units, C, w.d, dtype=torch.float32, device="cuda"),
              mu_hat=torch.empty(w.units, C, w.d, dtype=torch.bfloat16, device="cuda"),
              sizes=torch.empty(w.units, C, dtype=torch.int32, device="cuda"),
              offsets=torch.empty(w.units, C + 1, dtype=torch.int32, device="cuda"),
              perm=torch.empty(w.units, n, dtype=torch.int32, device="cuda"))
    ctx.export_clusters(st["mu"], st["mu_hat"], st["sizes"], st["offsets"], st["perm"])
    torch.cuda.synchronize()
    return st


def unit_state(st, u):
    return {k: (v[u].double() if k in ("mu", "mu_hat") else v[u]).cpu().numpy() for k, v in st.items()}


def check_csr_all_units(st, first_token, n):
    """Every unit: sizes sum to n, offsets are their exclusive scan, perm is a
    permutation of [first_token, first_token + n) ascending inside each cluster."""
    sizes, offs, perm = st["sizes"].long(), st["offsets"].long(), st["perm"].long()
    assert bool((sizes.sum(1) == n).all())
    assert bool((offs[:, 0] == 0).all())
    assert torch.equal(offs[:, 1:] - offs[:, :-1], sizes)
    srt = torch.sort(perm, dim=1).values
    want = torch.arange(first_token, first_token + n, device=perm.device).expand_as(srt)
    assert torch.equal(srt, want)
    starts = torch.zeros_like(perm, dtype=torch.bool)
    starts.scatter_(1, offs[:, :-1].clamp(max=n - 1), True)
    rising = perm[:, 1:] > perm[:, :-1]
    assert bool((rising | starts[:, 1:]).all())


def test_prefill_csr_every_unit(full):
    w, ctx = full["w"], full["ctx"]
    st = export_device(ctx, w)
    assert st["sizes"].shape[1] == w.C
    check_csr_all_units(st, w.sinks, w.L - w.sinks)
    # no centroid is lost: non-empty clusters have finite, non-zero centroids
    nz = st["sizes"] > 0
    assert bool(torch.isfinite(st["mu"]).all())
    assert bool((st["mu"].abs().sum(-1)[nz] > 0).all())


def test_assign_and_update_lockstep_sampled(full):
    """One more assignment with the prefill's final centroids (the same kernel
    and grid as inside the prefill), then one update from those labels."""
    w, ctx, K = full["w"], full["ctx"], full["K"]
    n = w.L - w.sinks
    before = export_device(ctx, w)
    labels = torch.empty(w.units, n, dtype=torch.int32, device="cuda")
    ctx.kmeans_assign(K, w.L, labels)
    ctx.kmeans_update(K, w.L, labels)
    after = export_device(ctx, w)
    assert ctx.device_error() == 0
    check_csr_all_units(after, w.sinks, n)
    lab = labels.cpu().numpy()
    for u in full["samples"]:
        keys = to64(K[u, w.sinks:w.L])
        mu_in = unit_state(before, u)["mu"]
        rows, near = check_assignment(keys, mu_in, lab[u], "bf16")
        assert near <= max(2, rows // 100), f"unit {u}: {near} near-tie rows of {rows}"
        # update, given the GPU labels: CSR bit-exact, centroids within 1e-5
        sizes, offsets, perm = ck.build_csr(lab[u], w.C, w.sinks)
        got = unit_state(after, u)
        assert np.array_equal(got["sizes"], sizes)
        assert np.array_equal(got["offsets"], offsets)
        assert np.array_equal(got["perm"], perm)
        check_centroids(got["mu"], ck.update(keys, lab[u], mu_in))


def test_decode_step_sampled(full):
    """Scoring, selection (fused and given scores) and attention for every unit
    at once; the oracle checks sampled units given the GPU's upstream values."""
    w, ctx, K, V = full["w"], full["ctx"], full["K"], full["V"]
    st = export_device(ctx, w)
    C = st["sizes"].shape[1]
    pend = min(57, w.decode_steps)  # pending tokens attended besides the selection
    cur_len = w.L + pend
    for qi in range(2):
        q = full["Q"][qi].contiguous()
        sc = torch.empty(w.units, C, dtype=torch.float32, device="cuda")
        ctx.score(q, sc)
        idx = torch.full((w.units, w.B), -1, dtype=torch.int32, device="cuda")
        cnt = torch.empty(w.units, dtype=torch.int32, device="cuda")
        ctx.select(q, w.B, idx, cnt)
        idx2, cnt2 = torch.full_like(idx, -1), torch.empty_like(cnt)
        ctx.select_scored(sc, w.B, idx2, cnt2)
        assert torch.equal(cnt, cnt2) and torch.equal(idx, idx2)
        assert bool((cnt == min(w.B, w.L - w.sinks)).all())
        out = torch.empty(w.units, w.g, w.d, dtype=torch.float32, device="cuda")
        ctx.sparse_decode_attn(q, K, V, idx, cnt, w.B, cur_len, out)
        # the whole step in one call: same selection, same output
        idx3, cnt3 = torch.full_like(idx, -1), torch.empty_like(cnt)
        out3 = torch.empty_like(out)
        ctx.decode_step(q, K, V, w.B, cur_len, idx3, cnt3, out3)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
        assert torch.equal(cnt, cnt3) and torch.equal(idx, idx3)
        assert (out - out3).abs().max().item() <= 1e-5
        scores, idx_h, cnt_h, out_h = sc.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy(), to64(out)
        for u in full["samples"]:
            s = unit_state(st, u)
            qu = to64(q[u])
            # scores within the bound of the bf16 centroid copy
            want = ck.score(qu, s["mu"])
            assert (np.abs(scores[u] - want) <= score_tol(qu, s["mu"], "bf16")).all()
            # selection given identical scores: bit-exact
            sel, c = ck.select(scores[u].astype(np.float64), s["sizes"], s["offsets"], s["perm"], w.B)
            assert cnt_h[u] == c
            assert np.array_equal(idx_h[u, :c], sel)
            # attention given identical idx
            Ku, Vu = to64(K[u, :cur_len]), to64(V[u, :cur_len])
            toks = ck.attention_tokens(w.sinks, w.L, cur_len, idx_h[u, :c])
            err = np.abs(out_h[u] - ck.sparse_attention(qu, Ku, Vu, toks)).max()
            assert err <= ATTN_TOL["bf16"], f"unit {u}: attention error {err}"


def test_incremental_full_size(full):
    """Workloads with incremental clustering: the 320 new tokens of every unit
    clustered into 4 clusters appended after the prefill clusters, in the
    benchmark's launch configuration (every unit in one call).  Run for
    k = 1 .. 10 Lloyd iterations from the same prefill state; on every unit,
    every iteration is checked in lock step against the oracle's step from
    the GPU's state after k - 1 iterations (iteration 1 from the seeds: keys at
    stride 80 on both sides)."""
    w, ctx, K = full["w"], full["ctx"], full["K"]
    if w.n_incremental == 0:
        pytest.skip("no incremental clustering in this workload (max_len leaves no room for a block)")
    inf = ctx.info()
    C0, end0 = inf.n_clusters, inf.clustered_end
    pre = export_device(ctx, w)
    keys = K[:, end0:end0 + w.m].double().cpu().numpy()          # [units, m, d]
    prev = keys[:, ::w.m // w.c_plus][:, :w.c_plus].astype(np.float32).astype(np.float64)
    for k in range(1, w.iters + 1):
        c2 = ckv.Context(units=w.units, g=w.g, max_len=w.max_len, max_clusters=w.max_clusters,
                         max_budget=w.B, iters=k, m=w.m, c_plus=w.c_plus)
        c2.import_clusters(C0, end0, pre["mu"], pre["sizes"], pre["offsets"], pre["perm"])
        c2.cluster_incremental(K, end0)
        st = export_device(c2, w)
        assert c2.device_error() == 0
        c2.close()
        assert st["sizes"].shape[1] == C0 + w.c_plus
        check_csr_all_units(st, w.sinks, end0 + w.m - w.sinks)
        assert torch.equal(st["sizes"][:, :C0], pre["sizes"])
        sizes = st["sizes"][:, C0:].cpu().numpy()
        offs = st["offsets"][:, C0:].cpu().numpy()
        seg = st["perm"][:, end0 - w.sinks:].cpu().numpy()
        mu = st["mu"][:, C0:].double().cpu().numpy()
        for u in range(w.units):
            lab = np.empty(w.m, dtype=np.int64)
            for j in range(w.c_plus):
                lab[seg[u, offs[u, j] - offs[u, 0]:offs[u, j + 1] - offs[u, 0]] - end0] = j
            check_assignment(keys[u], prev[u], lab, "bf16")
            wsz, woff, wperm = ck.build_csr(lab, w.c_plus, end0)
            assert np.array_equal(sizes[u], wsz) and np.array_equal(offs[u] - offs[u, 0], woff)
            assert offs[u, 0] == end0 - w.sinks
            assert np.array_equal(seg[u], wperm)
            check_centroids(mu[u], ck.update(keys[u], lab, prev[u]))
        prev = mu
