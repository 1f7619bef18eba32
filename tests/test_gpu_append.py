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


def test_append_rejects_bad_arguments():
    torch.cuda.init()
    K = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros(2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ckv.CKVError):
        ckv.append_kv(kn, kn, K, K, 8)            # pos == max_len
    with pytest.raises(ckv.CKVError):
        ckv.append_kv(kn, kn, K, K, -1)
