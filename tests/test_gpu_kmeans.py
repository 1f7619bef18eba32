"""GPU parity of the clustering path (seeding, tcgen05 assignment, the
deterministic update and CSR build, incremental clustering) against the CPU
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle.clusterkv as ck
from parity import (check_assignment, check_centroids, export_state, make_ctx, to64)
from recallable_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


def workload(name, **kw):
    base = synth.WORKLOADS[name]
    return synth.scaled(base, **kw)


def operand(w):
    return "bf16" if w.dtype == "bf16" else "f64"


# (workload, units, L, C): ragged token tails (n % 128 != 0) and centroid
# counts that need 1, 2 and 3 TMEM column chunks (C <= 256, <= 512, > 512),
# and counts above 640 that the kernel splits into passes over the keys
# (700: two passes of 352 rows; 1638, the 128k workload's C: four of 416)
ASSIGN_CASES = [
    ("layer_32k", 2, 16 + 1000, 13),
    ("layer_32k", 2, 16 + 3000, 300),
    ("layer_32k", 1, 16 + 2100, 520),
    ("layer_32k", 3, 16 + 129, 1),
    ("tiny_2k", 1, 2048, 25),
    ("tiny_2k", 2, 16 + 700, 41),
    ("layer_32k", 2, 16 + 2600, 700),
    ("long_128k", 1, 16 + 4000, 1638),
]


@pytest.mark.parametrize("wname,U,L,C", ASSIGN_CASES)
def test_assign_lockstep(wname, U, L, C):
    w = workload(wname, units=U, L=L, decode_steps=0, C=C, n_centres=max(C, 2))
    K, _ = synth.make_kv(w)
    if U > 1:
        K[1, 40:45] = 0  # zero-norm keys join cluster 0
    ctx = make_ctx(U, w.g, w.max_len, C, 64, w.dtype, iters=3)
    Kd = K.cuda().contiguous()
    n = L - 16
    labels = torch.empty(U, n, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(C)
    # iteration-0 centroids (seeds) and centroids after two oracle iterations
    for trial in range(2):
        mus = []
        for u in range(U):
            keys = to64(K[u, 16:L])
            if trial == 0:
                mu = ck.seed_centroids(keys, C)
            else:
                mu = ck.kmeans(keys, C, 2, operand(w))["mu"]
            mus.append(mu.astype(np.float32))
        mu32 = np.stack(mus)
        mu32[:, -1] *= rng.uniform(0.5, 2.0)   # centroid norms do not matter to the cosine
        ctx.import_clusters(C, 0, torch.from_numpy(mu32).cuda())
        ctx.kmeans_assign(Kd, L, labels)
        got = labels.cpu().numpy()
        for u in range(U):
            rows, near = check_assignment(to64(K[u, 16:L]), mu32[u].astype(np.float64), got[u], operand(w))
            assert near <= max(2, rows // 100), f"{near} near-tie rows of {rows}"
        if U > 1:
            assert (got[1, 40 - 16:45 - 16] == 0).all()
    ctx.close()


@pytest.mark.parametrize("C,dups", [(400, [(5, 300)]), (700, [(10, 600), (3, 200), (400, 690)])])
def test_assign_duplicate_centroids_tie_to_lower(C, dups):
    """Two centroids with the same direction give bit-identical dots, so every
    key nearest to them must take the lower index, whether the copies sit in
    one TMEM chunk, two chunks, or two passes over the keys."""
    w = workload("layer_32k", units=2, L=16 + 3000, decode_steps=0, C=C, n_centres=C)
    K, _ = synth.make_kv(w)
    n = w.L - 16
    ctx = make_ctx(2, w.g, w.max_len, C, 64, w.dtype, iters=1)
    mu32 = np.stack([ck.seed_centroids(to64(K[u, 16:w.L]), C) for u in range(2)]).astype(np.float32)
    for lo, hi in dups:
        mu32[:, hi] = 2.0 * mu32[:, lo]   # same direction, other norm
    ctx.import_clusters(C, 0, torch.from_numpy(mu32).cuda())
    labels = torch.empty(2, n, dtype=torch.int32, device="cuda")
    ctx.kmeans_assign(K.cuda().contiguous(), w.L, labels)
    got = labels.cpu().numpy()
    ctx.close()
    for u in range(2):
        mu_hat, _ = ck.normalize_centroids(mu32[u].astype(np.float64), "bf16")
        lab_o = ck.assign(to64(K[u, 16:w.L]), mu_hat)
        check_assignment(to64(K[u, 16:w.L]), mu32[u].astype(np.float64), got[u], "bf16")
        for lo, hi in dups:
            assert np.array_equal(mu_hat[lo], mu_hat[hi])
            assert (lab_o == lo).any(), "the duplicated centroid should attract keys"
            assert not (got[u] == hi).any(), f"a key took the higher duplicate {hi}"


@pytest.mark.parametrize("wname,U,L,C", ASSIGN_CASES[:5])
def test_update_lockstep(wname, U, L, C):
    w = workload(wname, units=U, L=L, decode_steps=0, C=C, n_centres=max(C, 2))
    K, _ = synth.make_kv(w)
    ctx = make_ctx(U, w.g, w.max_len, C, 64, w.dtype, iters=3)
    Kd = K.cuda().contiguous()
    n = L - 16
    olds, labs, wants = [], [], []
    for u in range(U):
        keys = to64(K[u, 16:L])
        r = ck.kmeans(keys, C, 2, operand(w))
        old = r["mu"].astype(np.float32).astype(np.float64)
        lab = ck.assign(keys, ck.normalize_centroids(old, operand(w))[0])
        olds.append(old)
        labs.append(lab)
        wants.append((ck.update(keys, lab, old), ck.build_csr(lab, C, 16)))
    ctx.import_clusters(C, 0, torch.tensor(np.stack(olds), dtype=torch.float32).cuda())
    ctx.kmeans_update(Kd, L, torch.tensor(np.stack(labs), dtype=torch.int32).cuda())
    st = export_state(ctx, U, dtype=w.dtype)
    for u in range(U):
        mu_w, (sz, off, perm) = wants[u]
        assert np.array_equal(st["sizes"][u], sz)
        assert np.array_equal(st["offsets"][u], off)
        assert np.array_equal(st["perm"][u], perm)
        check_centroids(st["mu"][u], mu_w)
        # operand copy: mu_hat is bf16(mu / ||mu||) up to the ambiguous roundings
        if w.dtype == "bf16":
            mh, amb = ck.normalize_centroids(st["mu"][u], "bf16")
            diff = np.abs(st["mu_hat"][u] - mh)
            assert (diff <= amb + 0.0).all()
    ctx.close()


def test_update_empty_cluster_keeps_centroid():
    w = workload("layer_32k", units=1, L=16 + 500, decode_steps=0, C=6, n_centres=6)
    K, _ = synth.make_kv(w)
    ctx = make_ctx(1, 4, w.max_len, 6, 64, "bf16")
    keys = to64(K[0, 16:w.L])
    rng = np.random.default_rng(3)
    old = rng.standard_normal((6, 128)).astype(np.float32)
    lab = rng.integers(0, 4, size=500).astype(np.int32)   # clusters 4, 5 empty
    ctx.import_clusters(6, 0, torch.from_numpy(old[None]).cuda())
    ctx.kmeans_update(K.cuda(), w.L, torch.from_numpy(lab[None]).cuda())
    st = export_state(ctx, 1)
    assert list(st["sizes"][0][4:]) == [0, 0]
    assert np.array_equal(st["mu"][0][4:], old[4:].astype(np.float64))
    check_centroids(st["mu"][0], ck.update(keys, lab, old.astype(np.float64)))
    ctx.close()


def labels_from_csr(sizes, offsets, perm, first_token, n):
    """The label of every token of a cluster segment [first_token, first_token
    + n), recovered from its CSR (and the CSR's invariants checked)."""
    C = len(sizes)
    assert sizes.sum() == n
    assert np.array_equal(offsets[1:] - offsets[:-1], sizes)
    assert np.array_equal(np.sort(perm), np.arange(first_token, first_token + n))
    lab = np.empty(n, dtype=np.int64)
    for c in range(C):
        seg = perm[offsets[c] - offsets[0]:offsets[c + 1] - offsets[0]]
        assert np.all(np.diff(seg) > 0)
        lab[seg - first_token] = c
    return lab


def _lockstep_chain(w, iters, units):
    """The GPU prefill run for k = 1 .. iters Lloyd iterations (it is
    deterministic, so the run of k iterations passes through the states of
    the run of k - 1).  Every iteration k of every unit is checked against
    the oracle's step applied to the GPU's own state after k - 1 iterations:
    the labels (recovered from the CSR) by the assignment rule, the CSR
    bit-exact given those labels, the centroids within 1e-5 of the means.
    Iteration 1 starts from the seeds, which both sides take from the keys.
    While the GPU labels equal those of the oracle's own free-running
    trajectory, the centroids must also agree with that trajectory; returns
    the number of (unit, iteration) pairs on it and the near-tie rows seen."""
    K, _ = synth.make_kv(w)
    Kd = K.cuda().contiguous()
    op = operand(w)
    n = w.L - 16
    keys = [to64(K[u, 16:w.L]) for u in range(units)]
    prev = [ck.seed_centroids(keys[u], w.C).astype(np.float32).astype(np.float64) for u in range(units)]
    traj = [ck.kmeans(keys[u], w.C, iters, op, trace=True)["trace"] for u in range(units)]
    on_traj = [True] * units
    exact, near_rows = 0, 0
    for k in range(1, iters + 1):
        ctx = make_ctx(units, w.g, w.max_len, w.C, 64, w.dtype, iters=k)
        ctx.cluster_prefill(Kd, w.L, w.C)
        st = export_state(ctx, units, dtype=w.dtype)
        ctx.close()
        for u in range(units):
            lab = labels_from_csr(st["sizes"][u], st["offsets"][u], st["perm"][u], 16, n)
            _, near = check_assignment(keys[u], prev[u], lab, op)
            near_rows += near
            sizes, offs, perm = ck.build_csr(lab, w.C, 16)
            assert np.array_equal(st["sizes"][u], sizes) and np.array_equal(st["offsets"][u], offs)
            assert np.array_equal(st["perm"][u], perm)
            check_centroids(st["mu"][u], ck.update(keys[u], lab, prev[u]))
            if on_traj[u] and np.array_equal(lab, traj[u][k - 1]["labels"]):
                check_centroids(st["mu"][u], traj[u][k - 1]["mu_out"])
                exact += 1
            else:
                on_traj[u] = False
            prev[u] = st["mu"][u]
    return exact, near_rows


def test_prefill_tiny_fp32_full_config():
    """The tiny single-head workload at its full size: 2048 fp32 keys, C = 25,
    10 iterations, seeds at stride 80."""
    w = synth.WORKLOADS["tiny_2k"]
    exact, _ = _lockstep_chain(w, 10, 1)
    assert exact >= 1


def test_prefill_bf16_free_running():
    w = workload("layer_32k", units=2, L=16 + 4000, decode_steps=0, C=50, n_centres=50)
    exact, _ = _lockstep_chain(w, 10, 2)
    assert exact >= 1


def test_prefill_is_deterministic():
    w = workload("layer_32k", units=2, L=16 + 5000, decode_steps=0, C=62, n_centres=62)
    K, _ = synth.make_kv(w)
    Kd = K.cuda().contiguous()
    outs = []
    for _ in range(2):
        ctx = make_ctx(2, 4, w.max_len, 62, 64, "bf16")
        ctx.cluster_prefill(Kd, w.L, 62)
        outs.append(export_state(ctx, 2))
        ctx.close()
    for k in ("mu", "mu_hat", "sizes", "offsets", "perm"):
        assert np.array_equal(outs[0][k], outs[1][k]), k


def test_incremental():
    """Prefill, then two incremental clusterings of 320 tokens into 4
    clusters each, appended after the prefill clusters; run for k = 1 .. 10
    Lloyd iterations, every iteration of every block checked in lock step
    against the oracle's step from the GPU's state after k - 1 iterations
    (iteration 1 from the seeds, keys at stride 80 on both sides)."""
    w = workload("layer_32k", units=2, L=16 + 800, decode_steps=700, C=10, n_centres=10)
    K, _ = synth.make_kv(w)
    Kd = K.cuda().contiguous()
    blocks = [(u, r) for u in range(2) for r in range(2)]
    keys = {b: to64(K[b[0], w.L + 320 * b[1]:w.L + 320 * (b[1] + 1)]) for b in blocks}
    prev = {b: ck.seed_centroids(keys[b], 4).astype(np.float32).astype(np.float64) for b in blocks}
    traj = {b: ck.kmeans(keys[b], 4, 10, "bf16", trace=True)["trace"] for b in blocks}
    on_traj = {b: True for b in blocks}
    exact = 0
    base = None
    for k in range(1, 11):
        ctx = make_ctx(2, 4, w.max_len, 10 + 8, 64, "bf16", iters=k)
        ctx.cluster_prefill(Kd, w.L, 10)
        pre = export_state(ctx, 2)
        ctx.cluster_incremental(Kd, w.L, 320, 4)
        ctx.cluster_incremental(Kd, w.L + 320, 320, 4)
        inf = ctx.info()
        assert inf.n_clusters == 18 and inf.clustered_end == w.L + 640
        st = export_state(ctx, 2)
        assert ctx.device_error() == 0
        ctx.close()
        for u in range(2):
            # the prefill part is unchanged by the appends
            assert np.array_equal(st["sizes"][u][:10], pre["sizes"][u])
            assert np.array_equal(st["perm"][u][:w.L - 16], pre["perm"][u])
        for (u, r) in blocks:
            b = (u, r)
            start = w.L + 320 * r
            cs = slice(10 + 4 * r, 14 + 4 * r)
            seg_lo = st["offsets"][u][10 + 4 * r]
            assert seg_lo == w.L - 16 + 320 * r
            sizes, offs = st["sizes"][u][cs], st["offsets"][u][10 + 4 * r:15 + 4 * r]
            perm = st["perm"][u][seg_lo:seg_lo + 320]
            lab = labels_from_csr(sizes, offs, perm, start, 320)
            check_assignment(keys[b], prev[b], lab, "bf16")
            wsz, woff, wperm = ck.build_csr(lab, 4, start)
            assert np.array_equal(sizes, wsz) and np.array_equal(offs - seg_lo, woff)
            assert np.array_equal(perm, wperm)
            check_centroids(st["mu"][u][cs], ck.update(keys[b], lab, prev[b]))
            if on_traj[b] and np.array_equal(lab, traj[b][k - 1]["labels"]):
                check_centroids(st["mu"][u][cs], traj[b][k - 1]["mu_out"])
                exact += 1
            else:
                on_traj[b] = False
            prev[b] = st["mu"][u][cs]
    assert exact >= 1


def test_incremental_begin_commit():
    """The split incremental clustering: while it is pending the decode calls
    see the previous clusters (its tokens are attended as pending tokens);
    after the commit the state is bit-identical to ckv_cluster_incremental's."""
    from parity import ATTN_TOL
    from recallable_kv_cache_gb300.ckv import CKVError
    w = workload("layer_32k", units=2, L=16 + 800, decode_steps=700, C=10, n_centres=10, B=128)
    K, V = synth.make_kv(w)
    Q = synth.make_queries(w, 1)
    Kd, Vd = K.cuda().contiguous(), V.cuda().contiguous()
    a = make_ctx(2, 4, w.max_len, 18, 128, "bf16")
    b = make_ctx(2, 4, w.max_len, 18, 128, "bf16")
    a.cluster_prefill(Kd, w.L, 10)
    b.cluster_prefill(Kd, w.L, 10)
    before = export_state(b, 2)
    a.cluster_incremental(Kd, w.L, 320, 4)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    ev.record(main)
    side.wait_event(ev)
    b.cluster_incremental_begin(Kd, w.L, 320, 4, stream=side)
    with pytest.raises(CKVError):
        b.cluster_incremental_begin(Kd, w.L, 320, 4, stream=side)
    with pytest.raises(CKVError):
        b.cluster_incremental(Kd, w.L, 320, 4)
    inf = b.info()
    assert inf.n_clusters == 10 and inf.clustered_end == w.L
    # decode while pending: previous clusters, 330 pending tokens
    q = Q[0].cuda().contiguous()
    idx = torch.empty(2, 128, dtype=torch.int32, device="cuda")
    cnt = torch.empty(2, dtype=torch.int32, device="cuda")
    out = torch.empty(2, 4, 128, dtype=torch.float32, device="cuda")
    cur_len = w.L + 330
    b.decode_step(q, Kd, Vd, 128, cur_len, idx, cnt, out)
    torch.cuda.synchronize()
    got, ih, ch = to64(out), idx.cpu().numpy(), cnt.cpu().numpy()
    for u in range(2):
        sel, c = ck.select(ck.score(to64(Q[0][u]), before["mu"][u]), before["sizes"][u], before["offsets"][u],
                           before["perm"][u], 128)
        assert ch[u] == c
        toks = ck.attention_tokens(16, w.L, cur_len, ih[u, :c])
        want = ck.sparse_attention(to64(Q[0][u]), to64(K[u]), to64(V[u]), toks)
        assert np.abs(got[u] - want).max() <= ATTN_TOL["bf16"]
    b.cluster_incremental_commit(stream=main)
    with pytest.raises(CKVError):
        b.cluster_incremental_commit(stream=main)
    inf = b.info()
    assert inf.n_clusters == 14 and inf.clustered_end == w.L + 320
    sa, sb = export_state(a, 2), export_state(b, 2)
    for k in ("mu", "mu_hat", "sizes", "offsets", "perm"):
        assert np.array_equal(sa[k], sb[k]), k
    a.close()
    b.close()
