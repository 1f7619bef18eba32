"""The C++ oracle (oracle/clusterkv_ref.cpp) behind the same Python functions
as the numpy oracle in oracle/clusterkv.py.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module; only
tests/, the smoke check in __graft_entry__ and the CPU-baseline leg of
bench.py do.  ``build()`` compiles the C++ file with g++ into
oracle/libckv_oracle.so; the functions below marshal numpy arrays and call it.
Each function does what the numpy function of the same name does (see that
module for the ClusterKV page sections they follow); the pins in
tests/test_oracle_pins.py run against both, and tests/test_oracle_cpp.py checks
the two against each other.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "clusterkv_ref.cpp")
LIB_PATH = os.path.join(HERE, "libckv_oracle.so")

SINKS, RATIO, M_INCR, C_PLUS = 16, 80, 320, 4

_D, _I, _L, _P = ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
_SIGS = {
    "ckvo_round_bf16": ([_D], _D),
    "ckvo_round_bf16_n": ([_P, _P, _L], None),
    "ckvo_normalize": ([_P, _I, _I, _I, _D, _P, _P], None),
    "ckvo_cosines": ([_P, _I, _I, _P, _I, _P], None),
    "ckvo_assign": ([_P, _I, _I, _P, _I, _P], None),
    "ckvo_update": ([_P, _I, _I, _P, _P, _I, _P], None),
    "ckvo_build_csr": ([_P, _I, _I, ctypes.c_int32, _P, _P, _P], None),
    "ckvo_objective": ([_P, _I, _I, _P, _P, _I], _D),
    "ckvo_seed_stride": ([_I, _I, _I], _I),
    "ckvo_kmeans": ([_P, _I, _I, _I, _I, _I, _I, ctypes.c_int32, _P, _P, _P, _P, _P], None),
    "ckvo_score": ([_P, _I, _I, _P, _I, _P], None),
    "ckvo_select": ([_P, _P, _P, _P, _I, _I, _P], _I),
    "ckvo_sparse_attention": ([_P, _I, _I, _P, _P, _P, _I, _P], None),
    "ckvo_unit_jobs": ([_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P], None),
}
_LIB = None


def build(verbose: bool = False) -> str:
    """Compile the C++ oracle (plain g++, no architecture flags) if it changed."""
    if not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", SRC, "-o", LIB_PATH]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"g++ failed on the C++ oracle:\n{r.stdout}\n{r.stderr}")
    return LIB_PATH


def lib():
    global _LIB
    if _LIB is None:
        build()
        h = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(h, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = h
    return _LIB


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- as in clusterkv.py
def cluster_count(L: int, sinks: int = SINKS, ratio: int = RATIO) -> int:
    return max(1, (L - sinks) // ratio)


def seed_stride(n: int, C: int, ratio: int = RATIO) -> int:
    return int(lib().ckvo_seed_stride(n, C, ratio))


def seed_centroids(keys, C: int, ratio: int = RATIO) -> np.ndarray:
    k = _f64(keys)
    return k[np.arange(C) * seed_stride(len(k), C, ratio)].copy()


def round_to_bf16(x) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    lib().ckvo_round_bf16_n(_p(x), _p(y), x.size)
    return y


def normalize_centroids(mu, operand: str = "bf16", rel_err: float = 2.0 ** -20):
    if operand not in ("bf16", "f64"):
        raise ValueError(operand)
    mu = _f64(mu)
    C, d = mu.shape
    mh, amb = np.empty_like(mu), np.empty_like(mu)
    lib().ckvo_normalize(_p(mu), C, d, 1 if operand == "bf16" else 0, rel_err, _p(mh), _p(amb))
    return mh, amb


def cosine_to_centroids(keys, mu_hat) -> np.ndarray:
    k, mh = _f64(keys), _f64(mu_hat)
    out = np.empty((len(k), len(mh)))
    lib().ckvo_cosines(_p(k), len(k), k.shape[1], _p(mh), len(mh), _p(out))
    return out


def assign(keys, mu_hat) -> np.ndarray:
    k, mh = _f64(keys), _f64(mu_hat)
    lab = np.empty(len(k), dtype=np.int32)
    lib().ckvo_assign(_p(k), len(k), k.shape[1], _p(mh), len(mh), _p(lab))
    return lab


def update(keys, labels, mu_old) -> np.ndarray:
    k, lab, old = _f64(keys), _i32(labels), _f64(mu_old)
    mu = np.empty_like(old)
    lib().ckvo_update(_p(k), len(k), k.shape[1], _p(lab), _p(old), len(old), _p(mu))
    return mu


def build_csr(labels, C: int, token_base: int = 0):
    lab = _i32(labels)
    sizes, offsets, perm = np.empty(C, np.int32), np.empty(C + 1, np.int32), np.empty(len(lab), np.int32)
    lib().ckvo_build_csr(_p(lab), len(lab), C, token_base, _p(sizes), _p(offsets), _p(perm))
    return sizes, offsets, perm


def objective(keys, labels, mu) -> float:
    k, lab, m = _f64(keys), _i32(labels), _f64(mu)
    return float(lib().ckvo_objective(_p(k), len(k), k.shape[1], _p(lab), _p(m), len(m)))


def kmeans(keys, C: int, iters: int, operand: str = "bf16", ratio: int = RATIO, token_base: int = 0,
           trace: bool = False):
    """The C++ K-means; with ``trace`` the same iterations are composed here
    from the C++ steps so that every intermediate state can be returned."""
    k = _f64(keys)
    n, d = k.shape
    if not trace:
        mu = np.empty((C, d))
        lab, sizes = np.empty(n, np.int32), np.empty(C, np.int32)
        offsets, perm = np.empty(C + 1, np.int32), np.empty(n, np.int32)
        lib().ckvo_kmeans(_p(k), n, d, C, iters, 1 if operand == "bf16" else 0, ratio, token_base, _p(mu),
                          _p(lab), _p(sizes), _p(offsets), _p(perm))
        return dict(mu=mu, labels=lab, sizes=sizes, offsets=offsets, perm=perm)
    mu = seed_centroids(k, C, ratio)
    labels = np.zeros(n, dtype=np.int32)
    steps = []
    for _ in range(iters):
        labels = assign(k, normalize_centroids(mu, operand)[0])
        mu_new = update(k, labels, mu)
        steps.append(dict(mu_in=mu, labels=labels, mu_out=mu_new, J_assign=objective(k, labels, mu),
                          J_update=objective(k, labels, mu_new)))
        mu = mu_new
    sizes, offsets, perm = build_csr(labels, C, token_base)
    return dict(mu=mu, labels=labels, sizes=sizes, offsets=offsets, perm=perm, trace=steps)


def cluster_prefill(K, L: int, C: int | None = None, iters: int = 10, operand: str = "bf16",
                    sinks: int = SINKS, ratio: int = RATIO, trace: bool = False):
    if C is None or C == 0:
        C = cluster_count(L, sinks, ratio)
    return kmeans(np.asarray(K, dtype=np.float64)[sinks:L], C, iters, operand, ratio, token_base=sinks, trace=trace)


def cluster_incremental(K, start: int, m: int = M_INCR, c_plus: int = C_PLUS, iters: int = 10,
                        operand: str = "bf16", ratio: int = RATIO, trace: bool = False):
    return kmeans(np.asarray(K, dtype=np.float64)[start:start + m], c_plus, iters, operand, ratio,
                  token_base=start, trace=trace)


def append_clusters(state: dict, new: dict) -> dict:
    n_old = int(state["offsets"][-1])
    return dict(mu=np.concatenate([state["mu"], new["mu"]]),
                sizes=np.concatenate([state["sizes"], new["sizes"]]).astype(np.int32),
                offsets=np.concatenate([state["offsets"][:-1], new["offsets"] + n_old]).astype(np.int32),
                perm=np.concatenate([state["perm"], new["perm"]]).astype(np.int32))


def score(q, mu) -> np.ndarray:
    q, m = _f64(np.atleast_2d(q)), _f64(mu)
    out = np.empty(len(m))
    lib().ckvo_score(_p(q), q.shape[0], q.shape[1], _p(m), len(m), _p(out))
    return out


def select(scores, sizes, offsets, perm, B: int):
    sc, sz, of, pm = _f64(scores), _i32(sizes), _i32(offsets), _i32(perm)
    idx = np.empty(max(B, 1), dtype=np.int32)
    cnt = int(lib().ckvo_select(_p(sc), _p(sz), _p(of), _p(pm), len(sc), max(B, 0), _p(idx)))
    return idx[:cnt].copy(), cnt


def attention_tokens(sinks: int, clustered_end: int, cur_len: int, idx) -> np.ndarray:
    return np.concatenate([np.arange(sinks), np.arange(clustered_end, cur_len),
                           np.asarray(idx, dtype=np.int64)]).astype(np.int64)


def sparse_attention(q, K, V, tokens) -> np.ndarray:
    q, Kf, Vf = _f64(np.atleast_2d(q)), _f64(K), _f64(V)
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    out = np.empty((q.shape[0], Kf.shape[1]))
    lib().ckvo_sparse_attention(_p(q), q.shape[0], q.shape[1], _p(Kf), _p(Vf), _p(tok), len(tok), _p(out))
    return out


def full_attention(q, K, V, cur_len: int) -> np.ndarray:
    return sparse_attention(q, K, V, np.arange(cur_len))


def unit_jobs(Ks, Vs, Qs, L: int, C: int, B: int, iters: int = 10, m: int = M_INCR, c_plus: int = C_PLUS,
              sinks: int = SINKS, ratio: int = RATIO, operand: str = "bf16", threads: int | None = None):
    """Whole per-unit jobs (prefill clustering, then every decode step with
    incremental clustering every m steps) on a pool of threads.  Ks, Vs:
    lists of [max_len, d] arrays; Qs: list of [T, g, d].  Returns (outputs
    [units, T, g, d], per-unit (prefill s, decode s))."""
    U = len(Ks)
    Ks = [_f64(k) for k in Ks]
    Vs = [_f64(v) for v in Vs]
    Qs = [_f64(q) for q in Qs]
    T, g, d = Qs[0].shape
    outs = [np.empty((T, g, d)) for _ in range(U)]
    arr = lambda xs: (ctypes.c_void_p * U)(*[x.ctypes.data for x in xs])
    times = np.empty(2 * U)
    lib().ckvo_unit_jobs(U, arr(Ks), arr(Vs), arr(Qs), arr(outs), L, T, C, B, iters, m, c_plus, sinks, ratio, g, d,
                         1 if operand == "bf16" else 0, threads or os.cpu_count() or 1, _p(times))
    return np.stack(outs), times.reshape(U, 2)
