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


def _free_running(w, iters, units):
    """Run the GPU prefill and the oracle K-means on the same keys.  When the
    oracle's trajectory has no near-tie row in any iteration, the GPU must
    reproduce it exactly (labels, CSR) with centroids within 1e-5."""
    K, _ = synth.make_kv(w)
    ctx = make_ctx(units, w.g, w.max_len, w.C, 64, w.dtype, iters=iters)
    ctx.cluster_prefill(K.cuda().contiguous(), w.L, w.C)
    st = export_state(ctx, units, dtype=w.dtype)
    ctx.close()
    exact_units = 0
    for u in range(units):
        keys = to64(K[u, 16:w.L])
        r = ck.cluster_prefill(to64(K[u]), w.L, w.C, iters=iters, operand=operand(w), trace=True)
        near = 0
        for stp in r["trace"]:
            mu32 = stp["mu_in"].astype(np.float32).astype(np.float64)
            lab = ck.assign(keys, ck.normalize_centroids(mu32, operand(w))[0])
            _, nr = check_assignment(keys, mu32, lab, operand(w))
            near += nr
        # invariants that hold whatever the trajectory
        assert st["sizes"][u].sum() == w.L - 16
        assert np.array_equal(np.sort(st["perm"][u]), np.arange(16, w.L))
        lab_gpu = np.empty(w.L - 16, dtype=np.int64)
        for c in range(w.C):
            seg = st["perm"][u][st["offsets"][u][c]:st["offsets"][u][c + 1]]
            assert np.all(np.diff(seg) > 0)
            lab_gpu[seg - 16] = c
        if near == 0:
            assert np.array_equal(st["sizes"][u], r["sizes"])
            assert np.array_equal(st["offsets"][u], r["offsets"])
            assert np.array_equal(st["perm"][u], r["perm"])
            check_centroids(st["mu"][u], r["mu"])
            exact_units += 1
        # the GPU centroids are the means of the GPU clusters
        check_centroids(st["mu"][u][st["sizes"][u] > 0],
                        ck.update(keys, lab_gpu, st["mu"][u])[st["sizes"][u] > 0])
    return exact_units


def test_prefill_tiny_fp32_full_config():
    """The tiny single-head workload at its full size: 2048 fp32 keys, C = 25,
    10 iterations, seeds at stride 80."""
    w = synth.WORKLOADS["tiny_2k"]
    _free_running(w, 10, 1)


def test_prefill_bf16_free_running():
    w = workload("layer_32k", units=2, L=16 + 4000, decode_steps=0, C=50, n_centres=50)
    _free_running(w, 10, 2)


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


@pytest.mark.parametrize("iters", [1, 10])
def test_incremental(iters):
    """Prefill, then two incremental clusterings of 320 tokens into 4
    clusters each, appended after the prefill clusters."""
    w = workload("layer_32k", units=2, L=16 + 800, decode_steps=700, C=10, n_centres=10)
    K, _ = synth.make_kv(w)
    Kd = K.cuda().contiguous()
    ctx = make_ctx(2, 4, w.max_len, 10 + 8, 64, "bf16", iters=iters)
    ctx.cluster_prefill(Kd, w.L, 10)
    base = export_state(ctx, 2)
    ctx.cluster_incremental(Kd, w.L, 320, 4)
    ctx.cluster_incremental(Kd, w.L + 320, 320, 4)
    inf = ctx.info()
    assert inf.n_clusters == 18 and inf.clustered_end == w.L + 640
    st = export_state(ctx, 2)
    ctx.close()
    for u in range(2):
        # prefill part unchanged
        assert np.array_equal(st["sizes"][u][:10], base["sizes"][u])
        assert np.array_equal(st["perm"][u][: w.L - 16], base["perm"][u])
        for r in range(2):
            start = w.L + 320 * r
            inc = ck.cluster_incremental(to64(K[u]), start, 320, 4, iters=iters, operand="bf16", trace=True)
            keys = to64(K[u, start:start + 320])
            near = sum(check_assignment(keys, s["mu_in"].astype(np.float32).astype(np.float64),
                                        ck.assign(keys, ck.normalize_centroids(
                                            s["mu_in"].astype(np.float32).astype(np.float64), "bf16")[0]),
                                        "bf16")[1] for s in inc["trace"])
            cs = slice(10 + 4 * r, 14 + 4 * r)
            seg_lo = st["offsets"][u][10 + 4 * r]
            assert seg_lo == w.L - 16 + 320 * r
            got_perm = st["perm"][u][seg_lo: seg_lo + 320]
            assert np.array_equal(np.sort(got_perm), np.arange(start, start + 320))
            if near == 0:
                assert np.array_equal(st["sizes"][u][cs], inc["sizes"])
                assert np.array_equal(st["offsets"][u][cs] - seg_lo, inc["offsets"][:4])
                assert np.array_equal(got_perm, inc["perm"])
                check_centroids(st["mu"][u][cs], inc["mu"])


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
