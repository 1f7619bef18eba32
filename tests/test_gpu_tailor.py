"""GPU parity of the channel pre-score (ckv_centroid_channels,
ckv_channel_prescore) against its CPU oracle: the channel-major copy and the
per-channel maxima bit-exact, the critical channels bit-exact (the ranking is
taken in fp32 on both sides), the scores within fp32 summation error."""
import numpy as np
import pytest
import torch

import oracle.tailor as to
from parity import make_ctx, to64
from recallable_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,U,g,C", [("bf16", 5, 4, 409), ("f32", 2, 1, 25), ("bf16", 3, 4, 1000)])
def test_prescore_parity(dtype, U, g, C):
    torch.cuda.init()
    rng = np.random.default_rng(C + U)
    d = 128
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    mu32 = rng.standard_normal((U, C, d)).astype(np.float32)
    mu32[:, :, 7] *= 20.0                       # an outlier channel, as in real keys
    ctx = make_ctx(U, g, 4096, C + 3, 64, dtype)
    ctx.import_clusters(C, 0, torch.from_numpy(mu32).cuda())
    mu_s = to64(torch.from_numpy(mu32).to(tdt))  # the scoring operand the context keeps
    muT = torch.empty(U, d, C + 3, dtype=tdt, device="cuda")
    chmax = torch.empty(U, d, dtype=torch.float32, device="cuda")
    ctx.centroid_channels(muT, chmax)
    q = torch.from_numpy(rng.standard_normal((U, g, d)).astype(np.float32)).to(tdt).cuda()
    mt, cm = to64(muT), chmax.cpu().numpy().astype(np.float64)
    for u in range(U):
        assert np.array_equal(mt[u, :, :C], mu_s[u].T)
        assert np.array_equal(cm[u], to.channel_max(mu_s[u]))
    for r in (1, 8, 12, 32):
        scores = torch.empty(U, C, dtype=torch.float32, device="cuda")
        chans = torch.empty(U, r, dtype=torch.int32, device="cuda")
        ctx.channel_prescore(q, muT, chmax, r, scores, chans)
        torch.cuda.synchronize()
        sc, ch = scores.cpu().numpy().astype(np.float64), chans.cpu().numpy()
        for u in range(U):
            qu = to64(q[u])
            want, wch = to.prescore(qu, mu_s[u], r)
            assert np.array_equal(ch[u], wch), (r, u)
            qs = to.head_sum_f32(qu).astype(np.float64)
            terms = np.abs(mu_s[u][:, wch] * qs[wch]).sum(axis=1)
            assert (np.abs(sc[u] - want) <= (r + 1) * 2.0 ** -24 * terms + 1e-30).all(), (r, u)
    ctx.close()


def test_prescore_selects_with_select_scored():
    """The pre-scores feed the cluster selection like exact scores do."""
    torch.cuda.init()
    w = synth.scaled(synth.WORKLOADS["layer_32k"], units=2, L=16 + 2000, decode_steps=4, C=25, n_centres=25, B=128)
    K, _ = synth.make_kv(w)
    ctx = make_ctx(w.units, w.g, w.max_len, w.C, 128, w.dtype)
    ctx.cluster_prefill(K.cuda().contiguous(), w.L, w.C)
    muT = torch.empty(w.units, 128, w.C, dtype=torch.bfloat16, device="cuda")
    chmax = torch.empty(w.units, 128, dtype=torch.float32, device="cuda")
    ctx.centroid_channels(muT, chmax)
    q = synth.make_queries(w, 1)[0].cuda().contiguous()
    scores = torch.empty(w.units, w.C, dtype=torch.float32, device="cuda")
    ctx.channel_prescore(q, muT, chmax, 8, scores)
    idx = torch.empty(w.units, 128, dtype=torch.int32, device="cuda")
    cnt = torch.empty(w.units, dtype=torch.int32, device="cuda")
    ctx.select_scored(scores, 128, idx, cnt)
    torch.cuda.synchronize()
    assert ctx.device_error() == 0
    assert (cnt.cpu().numpy() == 128).all()
    for u in range(w.units):
        ids = idx[u].cpu().numpy()
        assert len(set(ids.tolist())) == 128 and ids.min() >= 16 and ids.max() < w.L
    ctx.close()
