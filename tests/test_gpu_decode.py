"""GPU parity of the decode step (scoring, selection, sparse attention) against
the CPU oracle, through the C ABI.  Each part gets the oracle's own upstream
result as input so that errors do not cascade."""
import numpy as np
import pytest
import torch

import oracle.clusterkv as ck
from parity import (ATTN_TOL, check_assignment, make_ctx, score_tol, to64, upload_state)
from recallable_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, units, L, C, B, pending)
    "bf16_g4": ("layer_32k", 3, 16 + 1000, 13, 200, 37),
    "f32_g1": ("tiny_2k", 1, 2048, 25, 256, 5),
    "bf16_g4_c300": ("layer_32k", 2, 16 + 6000, 300, 1024, 320),
}


def build_case(name, seed_shift=0):
    wname, U, L, C, B, pend = CASES[name]
    w = synth.scaled(synth.WORKLOADS[wname], units=U, L=L, decode_steps=pend + 8, C=C, B=B,
                     n_centres=C, seed=synth.WORKLOADS[wname].seed + seed_shift)
    K, V = synth.make_kv(w)
    Q = synth.make_queries(w, 3)
    states = [ck.cluster_prefill(to64(K[u]), L, C, iters=3, operand="bf16" if w.dtype == "bf16" else "f64")
              for u in range(U)]
    for s in states:  # the GPU keeps fp32 centroids: the oracle uses the same values
        s["mu"] = s["mu"].astype(np.float32).astype(np.float64)
    return w, K, V, Q, states


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    torch.cuda.init()
    w, K, V, Q, states = build_case(request.param)
    ctx = make_ctx(w.units, w.g, w.max_len, w.C + 8, max(w.B, 1024), w.dtype)
    upload_state(ctx, states, w.L)
    Kd, Vd = K.cuda().contiguous(), V.cuda().contiguous()
    yield dict(w=w, K=K, V=V, Q=Q, states=states, ctx=ctx, Kd=Kd, Vd=Vd, name=request.param)
    ctx.close()


def test_score_parity(case):
    w, ctx = case["w"], case["ctx"]
    for qi in range(case["Q"].shape[0]):
        q = case["Q"][qi]
        sc = torch.empty(w.units, w.C, dtype=torch.float32, device="cuda")
        ctx.score(q.cuda().contiguous(), sc)
        got = to64(sc)
        for u in range(w.units):
            want = ck.score(to64(q[u]), case["states"][u]["mu"])
            tol = score_tol(to64(q[u]), case["states"][u]["mu"], w.dtype)
            assert (np.abs(got[u] - want) <= tol).all(), np.abs(got[u] - want).max()


@pytest.mark.parametrize("B", [0, 1, 57, 200, 10 ** 9])
def test_select_given_scores_bit_exact(case, B):
    w, ctx = case["w"], case["ctx"]
    B = min(B, 1024)
    q = case["Q"][0]
    sc = np.stack([ck.score(to64(q[u]), case["states"][u]["mu"]) for u in range(w.units)]).astype(np.float32)
    idx = torch.full((w.units, max(B, 1)), -7, dtype=torch.int32, device="cuda")
    cnt = torch.empty(w.units, dtype=torch.int32, device="cuda")
    ctx.select_scored(torch.from_numpy(sc).cuda(), B, idx, cnt)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for u in range(w.units):
        st = case["states"][u]
        want, wc = ck.select(sc[u].astype(np.float64), st["sizes"], st["offsets"], st["perm"], B)
        assert cnt[u] == wc == min(B, w.L - 16)
        assert np.array_equal(idx[u, :wc], want)
        assert (idx[u, wc:] == -7).all()  # entries past count untouched


def test_select_equals_score_then_select(case):
    """ckv_select (scoring into the context's scratch, then selection) against
    the two public calls ckv_score + ckv_select_scored."""
    w, ctx = case["w"], case["ctx"]
    q = case["Q"][1].cuda().contiguous()
    sc = torch.empty(w.units, w.C, dtype=torch.float32, device="cuda")
    ctx.score(q, sc)
    i1 = torch.empty(w.units, w.B, dtype=torch.int32, device="cuda")
    c1 = torch.empty(w.units, dtype=torch.int32, device="cuda")
    i2, c2 = torch.empty_like(i1), torch.empty_like(c1)
    ctx.select_scored(sc, w.B, i1, c1)
    ctx.select(q, w.B, i2, c2)
    assert torch.equal(c1, c2) and torch.equal(i1, i2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("g", [1, 2, 8])
def test_select_scores_its_units_for_every_group_size(dtype, g):
    """Up to 1024 clusters each selection CTA scores its own unit (one kernel
    instance per key dtype and group size): ckv_select equals ckv_score +
    ckv_select_scored bit for bit, and the selection from those scores equals
    the oracle's; random cluster layouts (empty clusters included)."""
    torch.cuda.init()
    U, C, n, d = 3, 45, 600, 128
    L = 16 + n
    rng = np.random.default_rng(77 + g + (0 if dtype == "bf16" else 100))
    ctx = make_ctx(U, g, L + 8, C, 1024, dtype)
    states = []
    for u in range(U):
        labels = rng.integers(0, C, size=n)
        labels[labels % 7 == 3] = 0  # some clusters stay empty
        sizes, offsets, perm = ck.build_csr(labels, C, 16)
        mu = rng.standard_normal((C, d)).astype(np.float32).astype(np.float64)
        states.append(dict(mu=mu, sizes=sizes, offsets=offsets, perm=perm))
    upload_state(ctx, states, L)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.from_numpy(rng.standard_normal((U, g, d))).to(tdt).cuda().contiguous()
    sc = torch.empty(U, C, dtype=torch.float32, device="cuda")
    ctx.score(q, sc)
    for B in (1, 100, 599, 1024):
        i1 = torch.full((U, B), -2, dtype=torch.int32, device="cuda")
        c1 = torch.empty(U, dtype=torch.int32, device="cuda")
        i2, c2 = torch.full_like(i1, -2), torch.empty_like(c1)
        ctx.select_scored(sc, B, i1, c1)
        ctx.select(q, B, i2, c2)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
        assert torch.equal(c1, c2) and torch.equal(i1, i2)
        got_i, got_c, s64 = i2.cpu().numpy(), c2.cpu().numpy(), to64(sc)
        for u in range(U):
            st = states[u]
            want, wc = ck.select(s64[u], st["sizes"], st["offsets"], st["perm"], B)
            assert got_c[u] == wc and np.array_equal(got_i[u, :wc], want)
    ctx.close()


@pytest.mark.parametrize("pending", [0, 1, "case"])
def test_attention_given_idx(case, pending):
    w, ctx = case["w"], case["ctx"]
    pend = CASES[case["name"]][5] if pending == "case" else pending
    cur_len = w.L + pend
    for qi in range(2):
        q = case["Q"][qi]
        sc = np.stack([ck.score(to64(q[u]), case["states"][u]["mu"]) for u in range(w.units)])
        idx = np.zeros((w.units, w.B), dtype=np.int32)
        cnt = np.zeros(w.units, dtype=np.int32)
        for u in range(w.units):
            st = case["states"][u]
            sel, c = ck.select(sc[u], st["sizes"], st["offsets"], st["perm"], w.B)
            idx[u, :c], cnt[u] = sel, c
        out = torch.empty(w.units, w.g, 128, dtype=torch.float32, device="cuda")
        ctx.sparse_decode_attn(q.cuda().contiguous(), case["Kd"], case["Vd"], torch.from_numpy(idx).cuda(),
                               torch.from_numpy(cnt).cuda(), w.B, cur_len, out)
        got = to64(out)
        for u in range(w.units):
            toks = ck.attention_tokens(16, w.L, cur_len, idx[u, :cnt[u]])
            want = ck.sparse_attention(to64(q[u]), to64(case["K"][u]), to64(case["V"][u]), toks)
            err = np.abs(got[u] - want).max()
            assert err <= ATTN_TOL[w.dtype], err
        assert ctx.device_error() == 0


def test_budget_covering_everything_is_full_attention(case):
    """B >= clustered tokens: the sparse set is every token (sinks, clustered,
    pending), so the result equals full attention."""
    w, ctx = case["w"], case["ctx"]
    B = 1024
    if w.L - 16 > B:
        pytest.skip("more clustered tokens than the largest budget of this case")
    q = case["Q"][2].cuda().contiguous()
    idx = torch.empty(w.units, B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(w.units, dtype=torch.int32, device="cuda")
    ctx.select(q, B, idx, cnt)
    cur_len = w.L + 3
    out = torch.empty(w.units, w.g, 128, dtype=torch.float32, device="cuda")
    ctx.sparse_decode_attn(q, case["Kd"], case["Vd"], idx, cnt, B, cur_len, out)
    got = to64(out)
    for u in range(w.units):
        want = ck.full_attention(to64(case["Q"][2][u]), to64(case["K"][u]), to64(case["V"][u]), cur_len)
        assert np.abs(got[u] - want).max() <= ATTN_TOL[w.dtype]


def test_bad_index_is_reported_not_faulted(case):
    w, ctx = case["w"], case["ctx"]
    q = case["Q"][0].cuda().contiguous()
    idx = torch.randint(16, w.L, (w.units, w.B), dtype=torch.int32, device="cuda")
    idx[:, 3] = w.max_len + 1000  # outside [0, cur_len)
    idx[:, 4] = -5
    cnt = torch.full((w.units,), w.B, dtype=torch.int32, device="cuda")
    out = torch.empty(w.units, w.g, 128, dtype=torch.float32, device="cuda")
    assert ctx.device_error() == 0
    ctx.sparse_decode_attn(q, case["Kd"], case["Vd"], idx, cnt, w.B, w.L, out)
    assert ctx.device_error() == 2  # CKV_DEV_BAD_INDEX
    assert torch.isfinite(out).all()
    # the skipped rows are excluded from the softmax
    toks_ok = idx.cpu().numpy()
    for u in range(w.units):
        keep = toks_ok[u][(toks_ok[u] >= 0) & (toks_ok[u] < w.L)]
        want = ck.sparse_attention(to64(case["Q"][0][u]), to64(case["K"][u]), to64(case["V"][u]),
                                   ck.attention_tokens(16, w.L, w.L, keep))
        assert np.abs(to64(out)[u] - want).max() <= ATTN_TOL[w.dtype]


def test_select_ties_and_empty_clusters():
    """Hand-made CSR with empty clusters and tied scores (including -0.0):
    ranks by (score desc, index asc), skips empty clusters, trims the last."""
    torch.cuda.init()
    U, d, C, L = 2, 128, 7, 16 + 20
    ctx = make_ctx(U, 1, L + 8, C, 64, "f32")
    rng = np.random.default_rng(0)
    sizes = np.array([3, 0, 5, 2, 0, 6, 4], dtype=np.int32)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    perm = (16 + rng.permutation(20)).astype(np.int32)
    st = dict(mu=rng.standard_normal((C, d)), sizes=sizes, offsets=offsets, perm=perm)
    upload_state(ctx, [st, st], L)
    scores = np.array([[1.0, 5.0, 1.0, -0.0, 9.0, 0.0, 1.0],
                       [-1.0, -1.0, -2.0, -1.0, -3.0, -1.0, -1.0]], dtype=np.float32)
    for B in (0, 1, 3, 4, 9, 13, 20, 64):
        idx = torch.full((U, max(B, 1)), -1, dtype=torch.int32, device="cuda")  # [units][B]
        cnt = torch.empty(U, dtype=torch.int32, device="cuda")
        ctx.select_scored(torch.from_numpy(scores).cuda(), B, idx, cnt)
        for u in range(U):
            want, wc = ck.select(scores[u].astype(np.float64), sizes, offsets, perm, B)
            assert cnt[u].item() == wc
            assert np.array_equal(idx[u, :wc].cpu().numpy(), want)
    ctx.close()


@pytest.mark.parametrize("C", [129, 1500, 3000, 6000])
def test_select_large_cluster_counts(C):
    """Random CSR with many clusters (the sort then holds 1, 2 or 4 keys per
    thread), tied scores, empty clusters: selection from given scores against
    the oracle, and the fused path against scoring followed by selection."""
    torch.cuda.init()
    U, d = 2, 128
    rng = np.random.default_rng(C)
    n = 6 * C
    L = 16 + n
    ctx = make_ctx(U, 4, L + 8, C, 2048, "bf16")
    states = []
    for u in range(U):
        labels = rng.integers(0, C, size=n)
        labels[labels % 7 == 3] = 0          # some clusters stay empty, one gets big
        sizes, offsets, perm = ck.build_csr(labels, C, 16)
        mu = rng.standard_normal((C, d)).astype(np.float32).astype(np.float64)
        states.append(dict(mu=mu, sizes=sizes, offsets=offsets, perm=perm))
    upload_state(ctx, states, L)
    scores = rng.integers(-20, 20, size=(U, C)).astype(np.float32)   # many ties
    for B in (1, 700, 2048):
        idx = torch.full((U, B), -1, dtype=torch.int32, device="cuda")
        cnt = torch.empty(U, dtype=torch.int32, device="cuda")
        ctx.select_scored(torch.from_numpy(scores).cuda(), B, idx, cnt)
        for u in range(U):
            st = states[u]
            want, wc = ck.select(scores[u].astype(np.float64), st["sizes"], st["offsets"], st["perm"], B)
            assert cnt[u].item() == wc
            assert np.array_equal(idx[u, :wc].cpu().numpy(), want)
    # ckv_select: its scores must rank like the GPU's own scores
    q = torch.from_numpy(rng.standard_normal((U, 4, d))).to(torch.bfloat16).cuda()
    sc = torch.empty(U, C, dtype=torch.float32, device="cuda")
    ctx.score(q, sc)
    i1 = torch.empty(U, 2048, dtype=torch.int32, device="cuda")
    c1 = torch.empty(U, dtype=torch.int32, device="cuda")
    i2, c2 = torch.empty_like(i1), torch.empty_like(c1)
    ctx.select_scored(sc, 2048, i1, c1)
    ctx.select(q, 2048, i2, c2)
    # ckv_select scores with the same kernel as ckv_score: identical selection
    assert torch.equal(c1, c2)
    for u in range(U):
        assert torch.equal(i1[u, :c1[u]], i2[u, :c2[u]])
    ctx.close()


def test_l2_persistence_changes_no_result(case):
    """With the centroid copy and perm held in a persisting L2 set-aside
    (ckv_set_l2_persistence) the selection and the attention give exactly
    the results they give without it; turning it on twice and off again is
    accepted."""
    w, ctx = case["w"], case["ctx"]
    pend = CASES[case["name"]][5]
    q = case["Q"][0].cuda().contiguous()
    cur_len = w.L + pend

    def run():
        i = torch.full((w.units, w.B), -3, dtype=torch.int32, device="cuda")
        c = torch.empty(w.units, dtype=torch.int32, device="cuda")
        o = torch.empty(w.units, w.g, 128, dtype=torch.float32, device="cuda")
        ctx.decode_step(q, case["Kd"], case["Vd"], w.B, cur_len, i, c, o)
        torch.cuda.synchronize()
        return i, c, o

    i0, c0, o0 = run()
    try:
        ctx.set_l2_persistence(-1)
        ctx.set_l2_persistence(1 << 20)
        i1, c1, o1 = run()
        ctx.set_l2_persistence(-1)
        i2, c2, o2 = run()
    finally:
        ctx.set_l2_persistence(0)
    i3, c3, o3 = run()
    assert ctx.device_error() == 0
    for i, c, o in ((i1, c1, o1), (i2, c2, o2), (i3, c3, o3)):
        assert torch.equal(c, c0) and torch.equal(i, i0) and torch.equal(o, o0)


def test_decode_step_equals_select_then_attention(case):
    """ckv_decode_step (selection then attention in one call) gives the idx /
    count of ckv_select and the output of ckv_sparse_decode_attn; three steps
    in a row."""
    w, ctx = case["w"], case["ctx"]
    pend = CASES[case["name"]][5]
    for qi in range(3):
        q = case["Q"][qi].cuda().contiguous()
        cur_len = w.L + (pend if qi != 1 else 0)
        i1 = torch.full((w.units, w.B), -3, dtype=torch.int32, device="cuda")
        c1 = torch.empty(w.units, dtype=torch.int32, device="cuda")
        o1 = torch.empty(w.units, w.g, 128, dtype=torch.float32, device="cuda")
        ctx.select(q, w.B, i1, c1)
        ctx.sparse_decode_attn(q, case["Kd"], case["Vd"], i1, c1, w.B, cur_len, o1)
        i2, c2, o2 = torch.full_like(i1, -3), torch.empty_like(c1), torch.empty_like(o1)
        ctx.decode_step(q, case["Kd"], case["Vd"], w.B, cur_len, i2, c2, o2)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
        assert torch.equal(c1, c2) and torch.equal(i1, i2)
        assert (o1 - o2).abs().max().item() <= 1e-5
        got = to64(o2)
        idx, cnt = i2.cpu().numpy(), c2.cpu().numpy()
        for u in range(w.units):
            toks = ck.attention_tokens(16, w.L, cur_len, idx[u, :cnt[u]])
            want = ck.sparse_attention(to64(case["Q"][qi][u]), to64(case["K"][u]), to64(case["V"][u]), toks)
            assert np.abs(got[u] - want).max() <= ATTN_TOL[w.dtype]


@pytest.mark.parametrize("C", [13, 129, 409, 1000])
def test_decode_step_selection_edge_cases(C):
    """ckv_decode_step's selection equals ckv_select's, and both the oracle's
    given the GPU's own scores: random cluster layouts with empty clusters,
    duplicated centroids (tied scores), a zero query (every score tied: rank
    by cluster index), budgets 0, 1, ragged, at and above the clustered
    tokens; the step's attention over that selection against the oracle."""
    torch.cuda.init()
    U, g, d, pend = 3, 4, 128, 21
    rng = np.random.default_rng(1000 + C)
    n = 7 * C + 5
    L = 16 + n
    max_len = L + 64
    ctx = make_ctx(U, g, max_len, C, n + 50, "bf16")
    states = []
    for u in range(U):
        labels = rng.integers(0, C, size=n)
        labels[labels % 5 == 2] = C - 1          # some clusters stay empty, one grows
        sizes, offsets, perm = ck.build_csr(labels, C, 16)
        mu = rng.standard_normal((C, d))
        mu[1::4] = mu[0]                         # duplicated rows: tied scores
        mu = torch.from_numpy(mu).to(torch.bfloat16).double().numpy()   # exact in the bf16 copy
        states.append(dict(mu=mu, sizes=sizes, offsets=offsets, perm=perm))
    upload_state(ctx, states, L)
    K = torch.from_numpy(rng.standard_normal((U, max_len, d))).to(torch.bfloat16)
    V = torch.from_numpy(rng.standard_normal((U, max_len, d))).to(torch.bfloat16)
    Kd, Vd = K.cuda().contiguous(), V.cuda().contiguous()
    cur_len = L + pend
    qs = [torch.from_numpy(rng.standard_normal((U, g, d))).to(torch.bfloat16), torch.zeros(U, g, d, dtype=torch.bfloat16)]
    for q in qs:
        qd = q.cuda().contiguous()
        sc = torch.empty(U, C, dtype=torch.float32, device="cuda")
        ctx.score(qd, sc)
        for B in sorted({b for b in (0, 1, 57, 700, n, n + 50) if b <= n + 50}):
            i1 = torch.full((U, max(B, 1)), -5, dtype=torch.int32, device="cuda")
            c1 = torch.empty(U, dtype=torch.int32, device="cuda")
            o1 = torch.empty(U, g, d, dtype=torch.float32, device="cuda")
            ctx.decode_step(qd, Kd, Vd, B, cur_len, i1, c1, o1)
            i2, c2 = torch.full_like(i1, -5), torch.empty_like(c1)
            ctx.select(qd, B, i2, c2)
            torch.cuda.synchronize()
            assert ctx.device_error() == 0
            assert torch.equal(c1, c2) and torch.equal(i1, i2)
            scores, idx, cnt, out = sc.cpu().numpy(), i1.cpu().numpy(), c1.cpu().numpy(), to64(o1)
            for u in range(U):
                st = states[u]
                want, wc = ck.select(scores[u].astype(np.float64), st["sizes"], st["offsets"], st["perm"], B)
                assert cnt[u] == wc == min(B, n)
                assert np.array_equal(idx[u, :wc], want)
                assert (idx[u, wc:] == -5).all()
                toks = ck.attention_tokens(16, L, cur_len, idx[u, :wc])
                ref = ck.sparse_attention(to64(q[u]), to64(K[u]), to64(V[u]), toks)
                assert np.abs(out[u] - ref).max() <= ATTN_TOL["bf16"]
    ctx.close()
