"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point include/ckv.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

from recallable_kv_cache_gb300 import build, ckv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ckv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ckv.lib()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(ckv_\w+)\s*\(", src, flags=re.M)))


def test_header_parses():
    fns = header_functions()
    assert "ckv_create" in fns and "ckv_sparse_decode_attn" in fns and len(fns) >= 16


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_binding_covers_header_exactly():
    assert sorted(ckv.SIGNATURES) == header_functions()


def test_config_struct_matches_header():
    src = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} ckv_config;", src, flags=re.S).group(1)
    fields = re.findall(r"int32_t\s+(\w+);", body)
    assert fields == [f for f, _ in ckv.Config._fields_]


def test_status_strings(lib):
    assert lib.ckv_status_str(0) == b"CKV_OK"
    for code in range(-1, -10, -1):
        assert lib.ckv_status_str(code).startswith(b"CKV_ERR_")
    assert lib.ckv_version() >= 100


def _cfg(**kw):
    base = dict(units=2, d=128, g=4, sinks=16, ratio=80, m=320, c_plus=4, iters=10, max_len=4096,
                max_clusters=64, max_budget=256, kv_dtype=ckv.BF16)
    base.update(kw)
    return ckv.Config(*[base[f] for f, _ in ckv.Config._fields_])


@pytest.mark.parametrize("bad,code", [
    (dict(d=64), -1), (dict(g=3), -1), (dict(units=0), -1), (dict(kv_dtype=7), -2),
    (dict(max_len=16), -1), (dict(iters=0), -1), (dict(c_plus=17), -1), (dict(max_budget=0), -1),
])
def test_create_rejects_bad_config_on_host(lib, bad, code):
    h = ctypes.c_void_p(123)
    cfg = _cfg(**bad)
    assert lib.ckv_create(ctypes.byref(cfg), ctypes.byref(h)) == code
    assert not h.value


def test_null_arguments_rejected(lib):
    h = ctypes.c_void_p()
    assert lib.ckv_create(None, ctypes.byref(h)) == -1
    assert lib.ckv_create(ctypes.byref(_cfg()), None) == -1
    assert lib.ckv_destroy(None) == -1
    assert lib.ckv_cluster_prefill(None, None, 100, 0, None) == -1
    assert lib.ckv_select(None, None, 1, 10, None, None, None) == -1
    assert lib.ckv_sparse_decode_attn(None, None, 1, None, None, None, None, 10, 100, None, None) == -1
    assert lib.ckv_get_device_error(None, None) == -1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(ckv, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(ckv, "_LIB", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        ckv.lib()


def test_set_wait_limit_rejects_on_host(lib):
    assert lib.ckv_set_wait_limit(None, 1000, 0) == -1


def test_set_l2_persistence_rejects_on_host(lib):
    assert lib.ckv_set_l2_persistence(None, -1) == -1
    assert lib.ckv_set_l2_persistence(None, 0) == -1
