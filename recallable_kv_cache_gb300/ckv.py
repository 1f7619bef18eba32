"""Thin ctypes binding of libckv.so (the C ABI declared in include/ckv.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, and a non-zero ckv_status becomes CKVError.
Every step of the path runs in the library's CUDA kernels; there is no CPU
fallback, and the library is loaded on first use (RuntimeError if it has not
been built).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libckv.so")

F32, BF16 = 0, 1
DEV_ERRORS = {0: "ok", 1: "timeout", 2: "bad index", 3: "bad count", 4: "bad label", 5: "bad csr"}

# Every entry point of include/ckv.h with its argument types.
_P, _I, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
SIGNATURES = {
    "ckv_status_str": ([_I], ctypes.c_char_p),
    "ckv_version": ([], _I),
    "ckv_create": ([_P, ctypes.POINTER(_P)], _I),
    "ckv_destroy": ([_P], _I),
    "ckv_cluster_prefill": ([_P, _P, _I, _I, _P], _I),
    "ckv_cluster_incremental": ([_P, _P, _I, _I, _I, _P], _I),
    "ckv_kmeans_assign": ([_P, _P, _I, _P, _P], _I),
    "ckv_kmeans_update": ([_P, _P, _I, _P, _P], _I),
    "ckv_score": ([_P, _P, _I, _P, _P], _I),
    "ckv_select_scored": ([_P, _P, _I, _P, _P, _P], _I),
    "ckv_select": ([_P, _P, _I, _I, _P, _P, _P], _I),
    "ckv_sparse_decode_attn": ([_P, _P, _I, _P, _P, _P, _P, _I, _I, _P, _P], _I),
    "ckv_decode_step": ([_P, _P, _I, _P, _P, _I, _I, _P, _P, _P, _P], _I),
    "ckv_quest_pages": ([_P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "ckv_quest_score": ([_P, _I, _P, _P, _I, _I, _I, _P, _P], _I),
    "ckv_selection_overlap": ([_I, _I, _I, _P, _P, _I, _P, _P, _I, _P, _P], _I),
    "ckv_centroid_channels": ([_P, _P, _P, _P], _I),
    "ckv_append_kv": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "ckv_channel_prescore": ([_P, _P, _I, _P, _P, _I, _P, _P, _P], _I),
    "ckv_cluster_incremental_begin": ([_P, _P, _I, _I, _I, _P], _I),
    "ckv_cluster_incremental_commit": ([_P, _P], _I),
    "ckv_get_info": ([_P, _P], _I),
    "ckv_export_clusters": ([_P, _P, _P, _P, _P, _P, _P], _I),
    "ckv_import_clusters": ([_P, _I, _I, _P, _P, _P, _P, _P], _I),
    "ckv_get_device_error": ([_P, ctypes.POINTER(_I)], _I),
    "ckv_set_wait_limit": ([_P, ctypes.c_int64, _I], _I),
    "ckv_set_l2_persistence": ([_P, ctypes.c_int64], _I),
    "ckv_sparse_decode_attn_noalloc": ([_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P], _I),
}


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "units", "d", "g", "sinks", "ratio", "m", "c_plus", "iters", "max_len",
        "max_clusters", "max_budget", "kv_dtype")]


class Info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_clusters", "prefill_clusters", "prefill_len", "clustered_end")]


class CKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib().ckv_status_str(status).decode()}")


_LIB = None


def lib():
    """The loaded libckv.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "recallable_kv_cache_gb300.build.build(); there is no CPU fallback")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = handle
    return _LIB


def _check(status: int, where: str):
    if status != 0:
        raise CKVError(status, where)


def ptr(t) -> int | None:
    """Device pointer of a tensor (or None)."""
    if t is None:
        return None
    return t.data_ptr()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _is_tensor(t) -> bool:
    return hasattr(t, "shape") and hasattr(t, "data_ptr")


class Context:
    """One library context: the cluster state of `units` (sequence, layer, KV
    head) triples, allocated on the current CUDA device.

    Tensor arguments are checked against the context's layout before the call
    (the C ABI takes plain pointers and cannot see extents): K and V must be
    contiguous [units, max_len, d], q contiguous [units, g, d], idx [units, >= B]
    and count [units] int32, out [units, g, d]; a mismatch raises ValueError
    and nothing is launched."""

    def __init__(self, units: int, g: int, max_len: int, max_clusters: int, max_budget: int,
                 kv_dtype: str = "bf16", d: int = 128, sinks: int = 16, ratio: int = 80,
                 m: int = 320, c_plus: int = 4, iters: int = 10):
        self.cfg = Config(units, d, g, sinks, ratio, m, c_plus, iters, max_len, max_clusters,
                          max_budget, BF16 if kv_dtype == "bf16" else F32)
        h = ctypes.c_void_p()
        _check(lib().ckv_create(ctypes.byref(self.cfg), ctypes.byref(h)), "ckv_create")
        self.handle = h

    def _kv(self, *ts):
        for t in ts:
            if _is_tensor(t) and (tuple(t.shape) != (self.cfg.units, self.cfg.max_len, self.cfg.d)
                                  or not t.is_contiguous()):
                raise ValueError(f"K/V must be contiguous [{self.cfg.units}, {self.cfg.max_len}, {self.cfg.d}], "
                                 f"got {tuple(t.shape)}")

    def _q(self, q):
        if _is_tensor(q) and (tuple(q.shape) != (self.cfg.units, self.cfg.g, self.cfg.d) or not q.is_contiguous()):
            raise ValueError(f"q must be contiguous [{self.cfg.units}, {self.cfg.g}, {self.cfg.d}], got {tuple(q.shape)}")

    def _sel(self, B, idx, count):
        if _is_tensor(idx) and (idx.dim() != 2 or idx.shape[0] != self.cfg.units or idx.shape[1] < max(B, 1)
                                or not idx.is_contiguous() or idx.stride(0) != B and B > 0):
            raise ValueError(f"idx must be contiguous [{self.cfg.units}, B={B}], got {tuple(idx.shape)}")
        if _is_tensor(count) and tuple(count.shape) != (self.cfg.units,):
            raise ValueError(f"count must be [{self.cfg.units}], got {tuple(count.shape)}")

    def _out(self, out):
        if _is_tensor(out) and (tuple(out.shape) != (self.cfg.units, self.cfg.g, self.cfg.d) or not out.is_contiguous()):
            raise ValueError(f"out must be contiguous [{self.cfg.units}, {self.cfg.g}, {self.cfg.d}], "
                             f"got {tuple(out.shape)}")

    def close(self):
        if getattr(self, "handle", None):
            _check(lib().ckv_destroy(self.handle), "ckv_destroy")
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- clustering ------------------------------------------------------------
    def cluster_prefill(self, K, L: int, n_clusters: int = 0, stream=None):
        self._kv(K)
        _check(lib().ckv_cluster_prefill(self.handle, ptr(K), L, n_clusters, _stream(stream)),
               "ckv_cluster_prefill")

    def cluster_incremental(self, K, start: int, m: int | None = None, c_plus: int | None = None,
                            stream=None):
        m = self.cfg.m if m is None else m
        c_plus = self.cfg.c_plus if c_plus is None else c_plus
        self._kv(K)
        _check(lib().ckv_cluster_incremental(self.handle, ptr(K), start, m, c_plus, _stream(stream)),
               "ckv_cluster_incremental")

    def cluster_incremental_begin(self, K, start: int, m: int | None = None, c_plus: int | None = None,
                                  stream=None):
        m = self.cfg.m if m is None else m
        c_plus = self.cfg.c_plus if c_plus is None else c_plus
        self._kv(K)
        _check(lib().ckv_cluster_incremental_begin(self.handle, ptr(K), start, m, c_plus, _stream(stream)),
               "ckv_cluster_incremental_begin")

    def cluster_incremental_commit(self, stream=None):
        _check(lib().ckv_cluster_incremental_commit(self.handle, _stream(stream)),
               "ckv_cluster_incremental_commit")

    def kmeans_assign(self, K, L: int, labels, stream=None):
        self._kv(K)
        _check(lib().ckv_kmeans_assign(self.handle, ptr(K), L, ptr(labels), _stream(stream)),
               "ckv_kmeans_assign")

    def kmeans_update(self, K, L: int, labels, stream=None):
        self._kv(K)
        _check(lib().ckv_kmeans_update(self.handle, ptr(K), L, ptr(labels), _stream(stream)),
               "ckv_kmeans_update")

    # -- decode ----------------------------------------------------------------
    def score(self, q, scores, stream=None):
        self._q(q)
        _check(lib().ckv_score(self.handle, ptr(q), _dtype_code(q), ptr(scores), _stream(stream)),
               "ckv_score")

    def centroid_channels(self, muT, chmax, stream=None):
        """Channel-major scoring centroids and per-channel maxima (see ckv_centroid_channels)."""
        _check(lib().ckv_centroid_channels(self.handle, ptr(muT), ptr(chmax), _stream(stream)),
               "ckv_centroid_channels")

    def channel_prescore(self, q, muT, chmax, r: int, scores, channels=None, stream=None):
        """Scores over the r critical channels (see ckv_channel_prescore)."""
        _check(lib().ckv_channel_prescore(self.handle, ptr(q), _dtype_code(q), ptr(muT), ptr(chmax), r,
                                          ptr(scores), ptr(channels), _stream(stream)), "ckv_channel_prescore")

    def select_scored(self, scores, B: int, idx, count, stream=None):
        _check(lib().ckv_select_scored(self.handle, ptr(scores), B, ptr(idx), ptr(count),
                                       _stream(stream)), "ckv_select_scored")

    def select(self, q, B: int, idx, count, stream=None):
        self._q(q)
        self._sel(B, idx, count)
        _check(lib().ckv_select(self.handle, ptr(q), _dtype_code(q), B, ptr(idx), ptr(count),
                                _stream(stream)), "ckv_select")

    def sparse_decode_attn(self, q, K, V, idx, count, B: int, cur_len: int, out, stream=None):
        self._q(q)
        self._kv(K, V)
        self._sel(B, idx, count)
        self._out(out)
        _check(lib().ckv_sparse_decode_attn(self.handle, ptr(q), _dtype_code(q), ptr(K), ptr(V),
                                            ptr(idx), ptr(count), B, cur_len, ptr(out),
                                            _stream(stream)), "ckv_sparse_decode_attn")

    def decode_step(self, q, K, V, B: int, cur_len: int, idx, count, out, stream=None):
        self._q(q)
        self._kv(K, V)
        self._sel(B, idx, count)
        self._out(out)
        _check(lib().ckv_decode_step(self.handle, ptr(q), _dtype_code(q), ptr(K), ptr(V), B, cur_len, ptr(idx),
                                     ptr(count), ptr(out), _stream(stream)), "ckv_decode_step")

    # -- state -----------------------------------------------------------------
    def info(self) -> Info:
        inf = Info()
        _check(lib().ckv_get_info(self.handle, ctypes.byref(inf)), "ckv_get_info")
        return inf

    def export_clusters(self, mu=None, mu_hat=None, sizes=None, offsets=None, perm=None, stream=None):
        _check(lib().ckv_export_clusters(self.handle, ptr(mu), ptr(mu_hat), ptr(sizes), ptr(offsets),
                                         ptr(perm), _stream(stream)), "ckv_export_clusters")

    def import_clusters(self, n_clusters: int, clustered_end: int, mu, sizes=None, offsets=None,
                        perm=None, stream=None):
        _check(lib().ckv_import_clusters(self.handle, n_clusters, clustered_end, ptr(mu), ptr(sizes),
                                         ptr(offsets), ptr(perm), _stream(stream)),
               "ckv_import_clusters")

    def set_wait_limit(self, cycles: int = 2_000_000_000, stall: bool = False):
        """Bounded-wait limit of this context's kernels, and the failure
        detection test switch (see ckv_set_wait_limit)."""
        _check(lib().ckv_set_wait_limit(self.handle, int(cycles), 1 if stall else 0), "ckv_set_wait_limit")

    def set_l2_persistence(self, nbytes: int = -1):
        """L2 set-aside for the centroid scoring copy and perm, which every
        decode step re-reads (see ckv_set_l2_persistence): -1 = what the
        context needs, 0 = off."""
        _check(lib().ckv_set_l2_persistence(self.handle, int(nbytes)), "ckv_set_l2_persistence")

    def device_error(self) -> int:
        v = ctypes.c_int32()
        _check(lib().ckv_get_device_error(self.handle, ctypes.byref(v)), "ckv_get_device_error")
        return v.value


def sparse_decode_attn_noalloc(q, K, V, idx, count, units: int, g: int, max_len: int, sinks: int,
                               clustered_end: int, cur_len: int, B: int, out, dev_err=None, stream=None):
    """Sparse decode attention without a context and without any allocation:
    for callers that may not allocate device memory (inside graph capture, or
    under an engine that owns all device memory).  Its scratch is a fixed
    8 MiB array inside the library; calls that overlap on the GPU race.  The
    first call on a device must come before any stream capture."""
    _check(lib().ckv_sparse_decode_attn_noalloc(ptr(q), _dtype_code(q), ptr(K), ptr(V), ptr(idx),
                                                ptr(count), units, g, max_len, sinks, clustered_end,
                                                cur_len, B, ptr(out), ptr(dev_err), _stream(stream)),
           "ckv_sparse_decode_attn_noalloc")


def quest_pages(K, L: int, page_max, page_min, sinks: int = 16, stream=None):
    """Page metadata of the page-granular comparator (see ckv_quest_pages)."""
    units, max_len = K.shape[0], K.shape[1]
    _check(lib().ckv_quest_pages(ptr(K), _dtype_code(K), units, max_len, sinks, L, ptr(page_max), ptr(page_min),
                                 _stream(stream)), "ckv_quest_pages")


def quest_score(q, page_max, page_min, scores, stream=None):
    """Page weights of the page-granular comparator (see ckv_quest_score)."""
    units, g = q.shape[0], q.shape[1]
    _check(lib().ckv_quest_score(ptr(q), _dtype_code(q), ptr(page_max), ptr(page_min), units, g,
                                 page_max.shape[1], ptr(scores), _stream(stream)), "ckv_quest_score")


def selection_overlap(prev, idx, count, hits, max_len: int, stream=None):
    """hits[u] = tokens of the selection (idx, count) that appear in any of the
    earlier selections ``prev`` = [(idx_r, count_r), ...] (see
    ckv_selection_overlap).  All idx_r share one shape [units, B_prev]."""
    units, B = idx.shape
    R = len(prev)
    B_prev = prev[0][0].shape[1] if R else 0
    ip = (ctypes.c_void_p * max(R, 1))(*[ptr(p[0]) for p in prev])
    cp = (ctypes.c_void_p * max(R, 1))(*[ptr(p[1]) for p in prev])
    _check(lib().ckv_selection_overlap(units, max_len, R, ip, cp, B_prev, ptr(idx), ptr(count), B, ptr(hits),
                                       _stream(stream)), "ckv_selection_overlap")


def append_kv(k_src, v_src, K, V, pos: int, n: int | None = None, stream=None):
    """Rows [pos, pos + n) of every unit of K and V := rows [0, n) of k_src /
    v_src (see ckv_append_kv).  k_src / v_src are [units, d] (one row, n = 1)
    or [units, src_len, d] (a view with a unit stride is taken as src_len =
    that stride / d); they may live in pinned host memory the device maps."""
    units, max_len, d = K.shape
    if k_src.dim() == 2:
        src_len, n = 1, 1
    else:
        src_len = k_src.stride(0) // d
        n = k_src.shape[1] if n is None else n
    _check(lib().ckv_append_kv(ptr(k_src), ptr(v_src), src_len, _dtype_code(K), units, max_len, pos, n, ptr(K),
                               ptr(V), _stream(stream)), "ckv_append_kv")
