"""The allocation-free attention entry point (for callers that may not call
cudaMalloc: code inside CUDA graph capture, or under an engine that owns all
device memory) gives the same output as the context-based entry point, on two
calls in a row that reuse its fixed scratch array.  Kept in a file that pytest
collects last so a failure here never hides the other tests."""
import numpy as np
import pytest
import torch

import oracle.clusterkv as ck
from parity import ATTN_TOL, make_ctx, to64, upload_state
from recallable_kv_cache_gb300 import ckv, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,g", [("bf16", 4), ("f32", 1), ("f32", 8)])
def test_noalloc_matches_context_entry_point_twice(dtype, g):
    """bf16 K/V (tensor-core kernel, 16-row work items) and fp32 K/V with one and
    eight query heads per KV head (the fp32 kernel's work items hold 64 and 32
    rows, which sets the split count the scratch must hold)."""
    torch.cuda.init()
    base = synth.WORKLOADS["layer_32k" if dtype == "bf16" else "tiny_2k"]
    w = synth.scaled(base, units=3, g=g, L=16 + 1200, decode_steps=60, C=15, n_centres=15, B=256)
    K, V = synth.make_kv(w)
    Q = synth.make_queries(w, 2)
    states = [ck.cluster_prefill(to64(K[u]), w.L, w.C, iters=2) for u in range(w.units)]
    ctx = make_ctx(w.units, w.g, w.max_len, w.C, w.B, w.dtype)
    upload_state(ctx, states, w.L)
    Kd, Vd = K.cuda().contiguous(), V.cuda().contiguous()
    idx = torch.empty(w.units, w.B, dtype=torch.int32, device="cuda")
    cnt = torch.empty(w.units, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, (qi, pend) in enumerate([(0, 7), (1, 41)]):
        q = Q[qi].cuda().contiguous()
        ctx.select(q, w.B, idx, cnt)
        cur = w.L + pend
        want = torch.empty(w.units, w.g, 128, dtype=torch.float32, device="cuda")
        got = torch.full_like(want, float("nan"))
        ctx.sparse_decode_attn(q, Kd, Vd, idx, cnt, w.B, cur, want)
        ckv.sparse_decode_attn_noalloc(q, Kd, Vd, idx, cnt, w.units, w.g, w.max_len, 16, w.L, cur, w.B,
                                       got, dev_err=err)
        torch.cuda.synchronize()
        diff = (got - want).abs().max().item()
        assert diff <= ATTN_TOL[w.dtype], (call, diff)
        assert int(err.item()) == 0
    ctx.close()


def test_noalloc_rejects_oversized_call():
    torch.cuda.init()
    q = torch.zeros(4096, 4, 128, dtype=torch.bfloat16, device="cuda")
    K = torch.zeros(4096, 64, 128, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(4096, 2048, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(4096, dtype=torch.int32, device="cuda")
    out = torch.empty(4096, 4, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(ckv.CKVError, match="CAPACITY"):
        ckv.sparse_decode_attn_noalloc(q, K, K, idx, cnt, 4096, 4, 64, 16, 32, 40, 2048, out)
