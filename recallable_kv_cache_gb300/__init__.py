"""GB300-native ClusterKV decode path: cluster-granular recallable KV selection.

The compute lives in ``libckv.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/ckv.h``).  ``recallable_kv_cache_gb300.ckv`` is the thin
ctypes binding; it loads the library on first use and raises if it is missing
(there is no CPU fallback).  ``synth`` holds the seeded synthetic workloads.
"""
