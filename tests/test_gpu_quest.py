"""GPU parity of the page-granular comparator (Quest) against its CPU oracle,
through the C ABI: page bounds bit-exact (maxima and minima of key values are
key values), page weights within fp32 summation error, page selection given
identical weights bit-exact, attention over the selected pages within the
attention tolerance."""
import numpy as np
import pytest
import torch

import oracle.clusterkv as ck
import oracle.quest as qo
from parity import ATTN_TOL, make_ctx, to64
from recallable_kv_cache_gb300 import ckv, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,L", [("bf16", 16 + 1000), ("f32", 2048), ("bf16", 16 + 4096)])
def test_quest_pages_scores_select_attend(dtype, L):
    base = synth.WORKLOADS["layer_32k" if dtype == "bf16" else "tiny_2k"]
    U = 3 if dtype == "bf16" else 1
    w = synth.scaled(base, units=U, L=L, decode_steps=8, C=max(1, (L - 16) // 80), n_centres=50, B=256)
    K, V = synth.make_kv(w)
    Q = synth.make_queries(w, 2)
    Kd, Vd = K.cuda().contiguous(), V.cuda().contiguous()
    n = L - 16
    P = (n + 15) // 16
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    pmax = torch.empty(U, P, 128, dtype=tdt, device="cuda")
    pmin = torch.empty_like(pmax)
    ckv.quest_pages(Kd, L, pmax, pmin)
    scores = torch.empty(U, P, dtype=torch.float32, device="cuda")
    # pages as clusters: sizes 16 (last short), offsets, identity permutation
    sizes, offsets, perm = qo.page_csr(n, 16, 16)
    ctx = make_ctx(U, w.g, w.max_len, P, 256, dtype)
    ctx.import_clusters(P, L, torch.zeros(U, P, 128, device="cuda"),
                        torch.from_numpy(np.tile(sizes, (U, 1))).cuda(),
                        torch.from_numpy(np.tile(offsets, (U, 1))).cuda(),
                        torch.from_numpy(np.tile(perm, (U, 1))).cuda())
    for u in range(U):
        kmax, kmin = qo.page_bounds(to64(K[u, 16:L]))
        assert np.array_equal(to64(pmax[u]), kmax) and np.array_equal(to64(pmin[u]), kmin)
    for qi in range(2):
        q = Q[qi].cuda().contiguous()
        ckv.quest_score(q, pmax, pmin, scores)
        idx = torch.empty(U, 256, dtype=torch.int32, device="cuda")
        cnt = torch.empty(U, dtype=torch.int32, device="cuda")
        ctx.select_scored(scores, 256, idx, cnt)
        out = torch.empty(U, w.g, 128, dtype=torch.float32, device="cuda")
        cur_len = L + 5
        ctx.sparse_decode_attn(q, Kd, Vd, idx, cnt, 256, cur_len, out)
        torch.cuda.synchronize()
        assert ctx.device_error() == 0
        sc, ih, ch, oh = scores.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy(), to64(out)
        for u in range(U):
            qu = to64(Q[qi][u])
            kmax, kmin = qo.page_bounds(to64(K[u, 16:L]))
            want = qo.page_scores(qu, kmax, kmin)
            terms = sum(np.abs(np.maximum(kmax * qh, kmin * qh)).sum(axis=1) for qh in np.atleast_2d(qu))
            assert (np.abs(sc[u] - want) <= 2.0 ** -16 * terms + 1e-30).all()
            sel, c = qo.select_pages(sc[u].astype(np.float64), n, 256, 16, 16)
            assert ch[u] == c and np.array_equal(ih[u, :c], sel)
            toks = ck.attention_tokens(16, L, cur_len, sel)
            err = np.abs(oh[u] - ck.sparse_attention(qu, to64(K[u]), to64(V[u]), toks)).max()
            assert err <= ATTN_TOL[dtype], err
    ctx.close()
