"""Failure detection without a GPU fault: every wait inside the kernels is
bounded, and a wait that runs out records CKV_DEV_TIMEOUT, lets the kernel
finish the copies and tensor-core work it started, and returns.  Each test
makes one wait run out on purpose (ckv_set_wait_limit with stall = 1: the
kernel first waits on a barrier or flag that nothing ever completes, with a
limit of about a millisecond), checks the status read back through
ckv_get_device_error, then runs the same call normally on the same context
and checks it against the oracle."""
import numpy as np
import pytest
import torch

import oracle.clusterkv as ck
from parity import ATTN_TOL, check_assignment, make_ctx, to64, upload_state
from recallable_kv_cache_gb300 import ckv, synth

pytestmark = pytest.mark.gpu

SHORT = 2_000_000    # SM cycles: about 1 ms
TIMEOUT = 1          # CKV_DEV_TIMEOUT


def test_assignment_wait_runs_out_then_recovers():
    """The tensor-core assignment: its MMA issuer gives up while the key tiles
    it was waiting for are still landing; the producer and issuer drain, TMEM
    is released, and the next assignment on the context is correct."""
    torch.cuda.init()
    w = synth.scaled(synth.WORKLOADS["layer_32k"], units=2, L=16 + 3000, decode_steps=0, C=300, n_centres=300)
    K, _ = synth.make_kv(w)
    Kd = K.cuda().contiguous()
    ctx = make_ctx(2, 4, w.max_len, 300, 64, "bf16", iters=1)
    mu32 = np.stack([ck.seed_centroids(to64(K[u, 16:w.L]), 300) for u in range(2)]).astype(np.float32)
    ctx.import_clusters(300, 0, torch.from_numpy(mu32).cuda())
    labels = torch.full((2, w.L - 16), -1, dtype=torch.int32, device="cuda")
    ctx.set_wait_limit(SHORT, stall=True)
    ctx.kmeans_assign(Kd, w.L, labels)
    assert ctx.device_error() == TIMEOUT
    ctx.set_wait_limit()  # default limit, no stall
    ctx.kmeans_assign(Kd, w.L, labels)
    assert ctx.device_error() == 0
    got = labels.cpu().numpy()
    for u in range(2):
        check_assignment(to64(K[u, 16:w.L]), mu32[u].astype(np.float64), got[u], "bf16")
    ctx.close()


def _decode_case(dtype, g):
    base = synth.WORKLOADS["layer_32k" if dtype == "bf16" else "tiny_2k"]
    w = synth.scaled(base, units=3, g=g, L=16 + 900, decode_steps=40, C=12, n_centres=12, B=128)
    K, V = synth.make_kv(w)
    q = synth.make_queries(w, 1)[0]
    states = [ck.cluster_prefill(to64(K[u]), w.L, w.C, iters=2) for u in range(w.units)]
    for s in states:
        s["mu"] = s["mu"].astype(np.float32).astype(np.float64)
    ctx = make_ctx(w.units, g, w.max_len, w.C, w.B, w.dtype)
    upload_state(ctx, states, w.L)
    return w, K, V, q, states, ctx


def _check_attention(w, K, V, q, states, idx, cnt, out, cur_len):
    for u in range(w.units):
        st = states[u]
        want_idx, c = ck.select(ck.score(to64(q[u]), st["mu"]), st["sizes"], st["offsets"], st["perm"], w.B)
        assert cnt[u] == c
        toks = ck.attention_tokens(16, w.L, cur_len, idx[u, :c])
        ref = ck.sparse_attention(to64(q[u]), to64(K[u]), to64(V[u]), toks)
        assert np.abs(out[u] - ref).max() <= ATTN_TOL[w.dtype]


def test_fp32_attention_wait_runs_out_then_recovers():
    """The fp32 attention: a consumer warp gives up, the producer stops and
    waits for its copies in flight; the next call is correct."""
    torch.cuda.init()
    w, K, V, q, states, ctx = _decode_case("f32", 4)
    qd, Kd, Vd = q.cuda().contiguous(), K.cuda().contiguous(), V.cuda().contiguous()
    idx = torch.empty(w.units, w.B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(w.units, dtype=torch.int32, device="cuda")
    out = torch.empty(w.units, w.g, 128, dtype=torch.float32, device="cuda")
    cur_len = w.L + 9
    ctx.select(qd, w.B, idx, cnt)
    ctx.set_wait_limit(SHORT, stall=True)
    ctx.sparse_decode_attn(qd, Kd, Vd, idx, cnt, w.B, cur_len, out)
    assert ctx.device_error() == TIMEOUT
    ctx.set_wait_limit()
    ctx.sparse_decode_attn(qd, Kd, Vd, idx, cnt, w.B, cur_len, out)
    assert ctx.device_error() == 0
    _check_attention(w, K, V, q, states, idx.cpu().numpy(), cnt.cpu().numpy(), to64(out), cur_len)
    ctx.close()
