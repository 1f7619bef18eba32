"""ckv_append_kv: the new K/V row of every unit lands in row pos of the caches,
from device memory and from pinned host memory the device maps; other rows
are untouched; bad arguments are rejected before any launch."""
import pytest
import torch

from parity import host_mapped
from recallable_kv_cache_gb300 import ckv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_append_rows(dtype, where):
    torch.cuda.init()
    g = torch.Generator().manual_seed(5)
    U, max_len, d = 37, 300, 128
    K0 = torch.randn(U, max_len, d, generator=g).to(dtype)
    V0 = torch.randn(U, max_len, d, generator=g).to(dtype)
    K, V = K0.cuda(), V0.cuda()
    kn = torch.randn(U, d, generator=g).to(dtype)
    vn = torch.randn(U, d, generator=g).to(dtype)
    if where == "device":
        ks, vs = kn.cuda(), vn.cuda()
    else:
        ks, vs = kn.pin_memory(), vn.pin_memory()
        if not (host_mapped(ks) and host_mapped(vs)):
            pytest.skip("pinned host memory is not addressable at its host address here")
    for pos in (0, 17, max_len - 1):
        ckv.append_kv(ks, vs, K, V, pos)
        K0[:, pos] = kn
        V0[:, pos] = vn
    torch.cuda.synchronize()
    assert torch.equal(K.cpu(), K0) and torch.equal(V.cpu(), V0)


@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_append_block_of_rows(where):
    """n rows per unit from a source with a longer row stride (a prompt's block)."""
    torch.cuda.init()
    g = torch.Generator().manual_seed(6)
    U, max_len, d, src_len, n, pos = 9, 200, 128, 40, 25, 100
    K0 = torch.randn(U, max_len, d, generator=g).to(torch.bfloat16)
    V0 = torch.randn(U, max_len, d, generator=g).to(torch.bfloat16)
    K, V = K0.cuda(), V0.cuda()
    ks = torch.randn(U, src_len, d, generator=g).to(torch.bfloat16)
    vs = torch.randn(U, src_len, d, generator=g).to(torch.bfloat16)
    if where == "device":
        ksd, vsd = ks.cuda(), vs.cuda()
    else:
        ksd, vsd = ks.pin_memory(), vs.pin_memory()
        if not (host_mapped(ksd) and host_mapped(vsd)):
            pytest.skip("pinned host memory is not addressable at its host address here")
    ckv.append_kv(ksd[:, :n], vsd[:, :n], K, V, pos)
    K0[:, pos:pos + n] = ks[:, :n]
    V0[:, pos:pos + n] = vs[:, :n]
    torch.cuda.synchronize()
    assert torch.equal(K.cpu(), K0) and torch.equal(V.cpu(), V0)


def test_append_rejects_bad_arguments():
    torch.cuda.init()
    K = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros(2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ckv.CKVError):
        ckv.append_kv(kn, kn, K, K, 8)            # pos == max_len
    with pytest.raises(ckv.CKVError):
        ckv.append_kv(kn, kn, K, K, -1)
    kb = torch.zeros(2, 5, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ckv.CKVError):
        ckv.append_kv(kb, kb, K, K, 4)            # rows 4..8 run past max_len
