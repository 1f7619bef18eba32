"""GPU parity of the reuse measurement (ckv_selection_overlap) against the CPU
oracle on seeded synthetic selections: R = 0, 1, 2, 3, counts below, at and
above the budget (clamped), ids outside [0, max_len) (ignored), empty units."""
import numpy as np
import pytest
import torch

import oracle.reuse as ro
from recallable_kv_cache_gb300 import ckv

pytestmark = pytest.mark.gpu


def _sets(rng, U, B, max_len, shared=None):
    idx = np.full((U, B), -7, dtype=np.int32)
    cnt = rng.integers(0, B + 1, size=U).astype(np.int32)
    for u in range(U):
        pool = shared[u] if shared is not None else None
        if pool is not None and rng.random() < 0.7:
            pick = rng.choice(pool, size=min(cnt[u], len(pool)), replace=False)
            rest = rng.choice(max_len, size=cnt[u] - len(pick), replace=False)
            idx[u, :cnt[u]] = np.concatenate([pick, rest])
        else:
            idx[u, :cnt[u]] = rng.choice(max_len, size=cnt[u], replace=False)
    return idx, cnt


@pytest.mark.parametrize("R", [0, 1, 2, 3])
def test_overlap_parity(R):
    torch.cuda.init()
    rng = np.random.default_rng(40 + R)
    U, B, max_len = 37, 300, 5000
    pools = [rng.choice(max_len, size=200, replace=False) for _ in range(U)]
    prev = [_sets(rng, U, B, max_len, pools) for _ in range(R)]
    cur_i, cur_c = _sets(rng, U, B, max_len, pools)
    cur_c[0] = B + 50       # clamped to B (the tail holds -7: ignored)
    cur_c[1] = -3           # clamped to 0
    cur_i[2, :5] = [max_len, max_len + 9, -1, 3, 3]   # out of range ids are ignored
    if R:
        prev[0][1][3] = 10 ** 6   # a previous count above B is clamped too
    dev = lambda a: torch.from_numpy(a).cuda()
    prev_d = [(dev(i), dev(c)) for i, c in prev]
    hits = torch.full((U,), -1, dtype=torch.int32, device="cuda")
    ckv.selection_overlap(prev_d, dev(cur_i), dev(cur_c), hits, max_len)
    got = hits.cpu().numpy()
    clamp = lambda c: int(min(max(c, 0), B))
    for u in range(U):
        ps = [[t for t in i[u, :clamp(c[u])] if 0 <= t < max_len] for i, c in prev]
        cur = [t for t in cur_i[u, :clamp(cur_c[u])] if 0 <= t < max_len]
        assert got[u] == ro.selection_hits(ps, cur), u


def test_overlap_rejects_bad_arguments():
    torch.cuda.init()
    z = torch.zeros(4, 8, dtype=torch.int32, device="cuda")
    c = torch.zeros(4, dtype=torch.int32, device="cuda")
    h = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(ckv.CKVError):
        ckv.selection_overlap([(z, c)] * 9, z, c, h, 100)            # R > 8
    with pytest.raises(ckv.CKVError):
        ckv.selection_overlap([(z, c)], z, c, h, 2_000_000)           # bitmap too large
